"""GPU parity of the optional log-sum-exp output (sage_attn_fwd_lse) against
the oracle's reading R13, lse = ln 2 * (m + log2 L - log2 448).

Source: diffusers PR #15060, "What does this PR do?" (the pages' kernel
returns no LSE; it is the quantity that merging partial attentions needs).
The attention output of sage_attn_fwd_lse must be bit-identical to
sage_attn_fwd's.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import WORKLOADS, bf16_bits, make_workload, sample_rows
from tests.gpu_common import default_scale, ensure_library, gen, lse_tolerance
from tests.test_gpu_parity import SHAPES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def _check_lse(lse_gpu, quant, S, scale, rows, what):
    _, _, lse_ref, lse_tie = oracle.attend_rows(quant, S, scale, rows, return_ties=True,
                                                return_lse=True)
    got = lse_gpu[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    tol = lse_tolerance(S, lse_ref, lse_tie)
    err = np.abs(got - lse_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} rows beyond tolerance; worst "
                           f"{err.max():.3g} (tol {tol[np.argmax(err)]:.3g})")
    return float(err.max())


@pytest.mark.parametrize("B,S,H,recipe,seed", SHAPES)
def test_lse_matches_oracle(B, S, H, recipe, seed):
    import quantized_attention_diffusion_gb300 as qad
    (q, k, v), bits = gen(B, S, H, recipe, seed)
    scale = default_scale()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out_ref = qad.attn_fwd(qd, kd, vd, scale)
    out, lse = qad.attn_fwd_lse(qd, kd, vd, scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    assert lse.shape == (B, H, S) and lse.dtype == torch.float32
    quant = oracle.quantize(*bits)
    _check_lse(lse.cpu().numpy(), quant, S, scale, oracle.all_rows(B, S, H), f"B{B} S{S} H{H}")


def test_lse_full_size_sampled_rows():
    """B=2 S=16384 H=24 with outlier channels (the image-DiT workload), 4
    heads x 512 sampled rows, in the benchmark's launch configuration."""
    import quantized_attention_diffusion_gb300 as qad
    w = WORKLOADS["b2_s16384_h24_outlier"]
    q, k, v = make_workload(w)
    out, lse = qad.attn_fwd_lse(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale)
    out_ref = qad.attn_fwd(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=512, seed=w.seed)
    quant = oracle.quantize(*[bf16_bits(t) for t in (q, k, v)])
    err = _check_lse(lse.cpu().numpy(), quant, w.S, w.softmax_scale, rows, w.name)
    print(f"{w.name}: max |lse gpu - oracle| {err:.3g}")


def test_lse_rejects_bad_buffer():
    import quantized_attention_diffusion_gb300 as qad
    (q, k, v), _ = gen(1, 40, 1)
    with pytest.raises(ValueError):
        qad.attn_fwd_lse(q.cuda(), k.cuda(), v.cuda(), lse=torch.empty(1, 1, 39, device="cuda"))
