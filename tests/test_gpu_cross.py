"""GPU parity of cross-attention (sage_attn_fwd_cross: Q with Sq rows, K and
V with Skv rows) against the oracle's reading R14.

Source: the pages' second workload, shorter K/V (issue #15014, "Describe the
solution you'd like": the gfx1201 kernel falls back for it; SageAttention
2.2's "partial-tile cross-attention shape" in InvokeAI PR #9657, "Summary").
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import WORKLOADS, bf16_bits, make_qkv, make_workload
from tests.gpu_common import (COS_BAR, assert_close_to_oracle, assert_within_two_pass_bound, cosine,
                              default_scale, ensure_library, f32,
                              lse_tolerance)

pytestmark = pytest.mark.gpu

CROSS_SHAPES = [  # (B, Sq, Skv, H, recipe, seed): single key, single query, ragged tiles both ways
    (1, 70, 1, 2, "normal", 200),
    (1, 1, 70, 1, "normal", 201),
    (2, 300, 50, 3, "k_channel_offset", 202),
    (1, 100, 257, 2, "normal", 203),
    (1, 129, 385, 1, "qk_outlier_channels", 204),
    (1, 1000, 97, 1, "normal", 205),
    (1, 64, 4096, 2, "k_channel_offset", 206),
]


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def _gen(B, Sq, Skv, H, recipe, seed):
    q, k, v = make_qkv(B, Sq, H, recipe=recipe, seed=seed, Skv=Skv)
    return (q, k, v), [bf16_bits(t) for t in (q, k, v)]


def _check(out, lse, bits, Sq, Skv, scale, rows, what):
    quant = oracle.quantize(*bits)
    ref_bits, ties, lse_ref, lse_tie = oracle.attend_rows(quant, Sq, scale, rows, return_ties=True,
                                                          return_lse=True, Skv=Skv)
    got = out[rows[:, 0], rows[:, 2], rows[:, 1]]
    err, _ = assert_close_to_oracle(got, f32(ref_bits), ties, what)
    assert_within_two_pass_bound(got, quant, Sq, scale, rows, ties, what + " vs two-pass", Skv=Skv)
    lse_got = lse[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
    lerr = np.abs(lse_got - lse_ref)
    tol = lse_tolerance(Skv, lse_ref, lse_tie)
    assert (lerr <= tol).all(), f"{what}: lse off by {lerr.max():.3g}"
    return err, f32(ref_bits)


@pytest.mark.parametrize("B,Sq,Skv,H,recipe,seed", CROSS_SHAPES)
def test_cross_matches_oracle(B, Sq, Skv, H, recipe, seed):
    import quantized_attention_diffusion_gb300 as qad
    (q, k, v), bits = _gen(B, Sq, Skv, H, recipe, seed)
    scale = default_scale()
    out, lse = qad.attn_fwd_cross(q.cuda(), k.cuda(), v.cuda(), scale, return_lse=True)
    torch.cuda.synchronize()
    assert out.shape == (B, Sq, H, 128) and lse.shape == (B, H, Sq)
    _check(out.float().cpu().numpy(), lse.cpu().numpy(), bits, Sq, Skv, scale,
           oracle.all_rows(B, Sq, H), f"Sq{Sq} Skv{Skv}")


def test_cross_with_equal_lengths_is_self_attention():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(2, 333, 3, recipe="qk_outlier_channels", seed=207)]
    a = qad.attn_fwd(q, k, v)
    b = qad.attn_fwd_cross(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_cross_rejects_mismatched_kv():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(1, 40, 2, seed=208, Skv=30)]
    with pytest.raises(ValueError):
        qad.attn_fwd_cross(q, k, v[:, :29].contiguous())
    with pytest.raises(ValueError):
        qad.attn_fwd_cross(q, k[:, :, :1].contiguous(), v[:, :, :1].contiguous())


@pytest.mark.parametrize("name", ["b2_sq16384_skv333_h24_cross", "b1_sq4096_skv16384_h24_cross"])
def test_cross_full_size_sampled_rows(name):
    """The two cross-attention workloads at full size, 4 heads x 512 sampled
    query rows (first and last tiles and the last short block included)."""
    import quantized_attention_diffusion_gb300 as qad
    from quantized_attention_diffusion_gb300.workloads import sample_rows
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    out, lse = qad.attn_fwd_cross(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale, return_lse=True)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=512, seed=w.seed)
    bits = [bf16_bits(t) for t in (q, k, v)]
    err, ref = _check(out.float().cpu().numpy(), lse.cpu().numpy(), bits, w.S, w.skv, w.softmax_scale,
                      rows, name)
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    exact = oracle.attention_fp64(*bits, w.softmax_scale, rows=rows)
    cos_gpu, cos_oracle = cosine(got, exact), cosine(ref, exact)
    print(f"{name}: max-abs vs oracle {err:.4g}; cosine vs fp64 gpu {cos_gpu:.6f} oracle {cos_oracle:.6f}")
    assert cos_gpu >= min(COS_BAR, cos_oracle - 1e-4)
