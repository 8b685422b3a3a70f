"""sage_attn_fwd_fused_q: the attention kernel quantises Q itself, as the
pages' kernel does (issue #15014, contract bullet "quantized per 32-row block
... inside the kernel").  sage_debug_fused_q writes out the codes and block
scales the kernel computed; they must equal the oracle's bit for bit, and the
output must equal sage_attn_fwd's.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits
from tests.gpu_common import ensure_library, gen
from tests.test_gpu_parity import SHAPES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def _check(qkv, q_bits):
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in qkv]
    out, q_i8, q_scale = qad.debug_fused_q(q, k, v)
    out_fused = qad.attn_fwd(q, k, v, fused_q=True)
    out_plain = qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    ref_codes, ref_scale = oracle.quantize_qk(q_bits)
    g_codes, g_scale = q_i8.cpu().numpy(), q_scale.cpu().numpy()
    assert g_codes.shape == ref_codes.shape and g_scale.shape == ref_scale.shape
    bad = g_codes != ref_codes
    assert not bad.any(), f"{int(bad.sum())} Q codes differ, first at {np.argwhere(bad)[0].tolist()}"
    assert np.array_equal(g_scale.view(np.uint32), ref_scale.view(np.uint32))
    assert torch.equal(out.view(torch.int16), out_plain.view(torch.int16))
    assert torch.equal(out_fused.view(torch.int16), out_plain.view(torch.int16))


@pytest.mark.parametrize("B,S,H,recipe,seed", SHAPES)
def test_fused_q_codes_bit_exact(B, S, H, recipe, seed):
    qkv, bits = gen(B, S, H, recipe, seed)
    _check(qkv, bits[0])


def test_fused_q_special_values_bit_exact():
    """Zero blocks, negative zeros, scales near the subnormal range and huge
    values (the division path), quotients exactly on .5 (ties to even)."""
    B, S, H = 1, 200, 2
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, size=(B, S, H, 128)).astype(np.float32)
    x[0, 0:32] = 0.0
    x[0, 32:64, 0] = -0.0
    x[0, 64:96, 1] *= 1e-37
    x[0, 96:128, 0] *= 3e30
    x[0, 130, 0, :4] = [127.0, 63.5, -0.5, 1.5]
    x[0, 160:192, 1] = np.clip(np.round(rng.normal(0, 40, size=(32, 128))), -120, 120) + 0.5  # exact halves
    x[0, 160, 1, 0] = 127.0                                                 # scale exactly 1
    t = torch.from_numpy(x).to(torch.bfloat16)
    _check((t, t, t), bf16_bits(t))


def test_fused_q_full_size_4096x24_bit_exact():
    qkv, bits = gen(1, 4096, 24, "k_channel_offset", 1)
    _check(qkv, bits[0])


def test_fused_q_output_equals_plain_at_bench_size():
    """B=2 S=16384 H=24 with outlier channels (the benchmark's workload and
    launch configuration): the in-kernel Q quantisation gives the separate
    pass's codes, so the two outputs are the same bits."""
    import quantized_attention_diffusion_gb300 as qad
    from quantized_attention_diffusion_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["b2_s16384_h24_outlier"]
    q, k, v = [t.cuda() for t in make_workload(w)]
    out_fused = qad.attn_fwd(q, k, v, w.softmax_scale, fused_q=True)
    out_plain = qad.attn_fwd(q, k, v, w.softmax_scale)
    torch.cuda.synchronize()
    diff = out_fused.view(torch.int16) != out_plain.view(torch.int16)
    assert not diff.any(), f"{int(diff.sum())} outputs differ"
