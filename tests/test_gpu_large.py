"""GPU parity at the full sizes of the pages' image and video workloads, on
sampled query rows (attention rows are independent, so each sampled row is
checked exactly as in a full comparison): 4 heads x 512 rows including the
first and last 128-row tiles and the last (short) 32-row block.

Workloads (synthetic stand-ins for the pages' diffusion/video models,
InvokeAI PR #9657 "Summary" and diffusers PR #15060 "Results"):
  B=2 S=16384 H=24 with 1% of Q/K channels x8 (image DiT, 2048^2 latents);
  B=1 S=32760 H=40 (length not a multiple of the tile: tail blocks);
  B=1 S=65536 H=24 with per-channel K offsets (long video latent).
The same launch configuration as the benchmark runs (sage_attn_fwd).

Each sampled row is checked three ways: element-wise against the oracle's
96-key online form, against its two-pass form within the derived bound of
reading R16, and by cosine against unquantized float64 attention.  The
cosine bar is 0.999 outright except on the outlier-channel workload, where
the quantized algorithm itself (the oracle, tiled or two-pass) reaches only
0.99891 on these rows: there the kernel must not fall more than 1e-4 below
the oracle's own cosine.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import WORKLOADS, bf16_bits, make_workload, sample_rows
from tests.gpu_common import (COS_BAR, assert_close_to_oracle, assert_within_two_pass_bound, cosine,
                              ensure_library, f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


# Workloads on which the quantized algorithm itself stays below the cosine
# bar against float64 (measured with the oracle on the sampled rows).
BELOW_BAR = {"b2_s16384_h24_outlier": 0.99891}


@pytest.mark.parametrize("name", ["b2_s16384_h24_outlier", "b1_s32760_h40", "b1_s65536_h24_koffset"])
def test_full_size_sampled_rows(name):
    import quantized_attention_diffusion_gb300 as qad
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out = qad.attn_fwd(q.cuda(), k.cuda(), v.cuda(), softmax_scale=w.softmax_scale)
    quant = qad.quantize_qkv(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    bits = [bf16_bits(t) for t in (q, k, v)]
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=512, seed=w.seed)
    rt = torch.from_numpy(rows).long().cuda()
    got = out[rt[:, 0], rt[:, 2], rt[:, 1]].float().cpu().numpy()
    # quantisation of the whole tensors is bit-exact
    ref_quant = oracle.quantize(*bits)
    for g, r in zip(quant, ref_quant):
        assert np.array_equal(g.cpu().numpy().view(np.uint8), r.view(np.uint8))
    ref_bits, ties = oracle.attend_rows(ref_quant, w.S, w.softmax_scale, rows, return_ties=True)
    ref = f32(ref_bits)
    exact = oracle.attention_fp64(*bits, w.softmax_scale, rows=rows)
    err, n_ties = assert_close_to_oracle(got, ref, ties, name)
    err2, used = assert_within_two_pass_bound(got, ref_quant, w.S, w.softmax_scale, rows, ties, name)
    cos_gpu, cos_oracle = cosine(got, exact), cosine(ref, exact)
    print(f"{name}: max-abs vs oracle {err:.4g} ({n_ties} rows with P ties); vs two-pass {err2:.4g} "
          f"({used:.3f} of the bound); cosine vs fp64 gpu {cos_gpu:.6f} oracle {cos_oracle:.6f}")
    if name in BELOW_BAR:
        assert cos_oracle < COS_BAR
        assert cos_gpu >= cos_oracle - 1e-4
    else:
        assert cos_oracle >= COS_BAR and cos_gpu >= COS_BAR
