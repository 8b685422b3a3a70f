"""GPU parity of K smoothing (sage_quantize_qkv_smooth_k,
sage_attn_fwd_smooth_k) against the oracle's reading R15.

Source: InvokeAI PR #9657, "Summary" / "How it works" (SageAttention's
smooth_k: per-channel K mean subtraction before quantisation).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import WORKLOADS, bf16_bits, make_workload, sample_rows
from tests.gpu_common import (assert_close_to_oracle, assert_within_two_pass_bound, default_scale, ensure_library,
                              f32, gen)
from tests.test_gpu_parity import SHAPES

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def _eq(name, g, r):
    g = g.cpu().numpy() if isinstance(g, torch.Tensor) else g
    assert g.shape == r.shape, name
    eq = g.view(np.uint32) == r.view(np.uint32) if g.dtype == np.float32 else g == r
    assert eq.all(), f"{name}: {int((~eq).sum())} mismatches, first at {np.argwhere(~eq)[0].tolist()}"


def _check_quant(qkv, bits):
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in qkv]
    got = qad.quantize_qkv_smooth_k(q, k, v)
    torch.cuda.synchronize()
    qc, qs = oracle.quantize_qk(bits[0])
    kc, ks, km = oracle.quantize_k_smooth(bits[1])
    vt, vs = oracle.quantize_v(bits[2])
    for name, g, r in zip(["q_i8", "q_scale", "k_i8", "k_scale", "vt", "v_scale", "k_mean"], got,
                          [qc, qs, kc, ks, vt, vs, km]):
        _eq(name, g, r)


@pytest.mark.parametrize("B,S,H,recipe,seed", SHAPES)
def test_smooth_k_quantisation_bit_exact(B, S, H, recipe, seed):
    qkv, bits = gen(B, S, H, recipe, seed)
    _check_quant(qkv, bits)


def test_smooth_k_quantisation_full_size_4096x24_bit_exact():
    qkv, bits = gen(1, 4096, 24, "k_channel_offset", 1)
    _check_quant(qkv, bits)


@pytest.mark.parametrize("B,S,H,recipe,seed", SHAPES)
def test_smooth_k_attention_matches_oracle(B, S, H, recipe, seed):
    import quantized_attention_diffusion_gb300 as qad
    qkv, bits = gen(B, S, H, recipe, seed)
    scale = default_scale()
    out = qad.attn_fwd(*[t.cuda() for t in qkv], scale, smooth_k=True)
    torch.cuda.synchronize()
    quant = oracle.quantize(*bits, smooth_k=True)
    rows = oracle.all_rows(B, S, H)
    ref, ties = oracle.attend_rows(quant, S, scale, rows, return_ties=True)
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_close_to_oracle(got, f32(ref), ties, f"smooth B{B} S{S} H{H}")
    assert_within_two_pass_bound(got, quant, S, scale, rows, ties, f"smooth B{B} S{S} H{H} vs two-pass")


def test_smooth_k_means_exact_over_wide_magnitudes():
    """Channels 0-63 of K ordinary N(0,1) values (each thread's fp32 partial
    sums are exact and kept), channels 64-127 spread log-uniformly over
    [2^-33, 2^3) with random signs (fp32 additions round, so those threads
    redo their slices in 2^-40 fixed point); 1000 tokens, four slices, the
    last one partial.  Every channel's sum stays below 2^13, where the mean
    is the exactly rounded one: the means and the K codes equal the
    oracle's bit for bit."""
    g = torch.Generator().manual_seed(340)
    B, S, H = 1, 1000, 2
    q = torch.randn((B, S, H, 128), generator=g).to(torch.bfloat16)
    v = torch.randn((B, S, H, 128), generator=g).to(torch.bfloat16)
    mag = torch.exp2(torch.rand((B, S, H, 64), generator=g, dtype=torch.float64) * 36.0 - 33.0)
    sign = torch.where(torch.rand((B, S, H, 64), generator=g) < 0.5, -1.0, 1.0).to(torch.float64)
    k = torch.cat([torch.randn((B, S, H, 64), generator=g, dtype=torch.float64), mag * sign], dim=-1)
    k = k.to(torch.bfloat16)
    ak = k.float().abs()
    assert bool(((ak == 0) | ((ak >= 2.0 ** -33) & (ak < 2.0 ** 22))).all())
    assert float(k.double().sum(dim=1).abs().max()) < 2.0 ** 13
    _check_quant((q, k, v), [bf16_bits(t) for t in (q, k, v)])


def test_exact_channel_offset_is_removed_on_gpu():
    """Zero-mean integer keys plus an exact per-channel offset: smoothed
    attention equals plain attention on the offset-free keys bit for bit."""
    import quantized_attention_diffusion_gb300 as qad
    B, S, H = 1, 256, 2
    rng = np.random.default_rng(60)
    half = rng.integers(-8, 9, size=(B, S // 2, H, 128)).astype(np.float32)
    kz = np.concatenate([half, -half], axis=1)
    c = rng.integers(-40, 41, size=(1, 1, H, 128)).astype(np.float32)
    k0 = torch.from_numpy(kz).to(torch.bfloat16).cuda()
    k1 = torch.from_numpy(kz + c).to(torch.bfloat16).cuda()
    (q, _, v), _ = gen(B, S, H, "normal", 61)
    q, v = q.cuda(), v.cuda()
    plain = qad.attn_fwd(q, k0, v)
    smooth = qad.attn_fwd(q, k1, v, smooth_k=True)
    torch.cuda.synchronize()
    assert torch.equal(plain.view(torch.int16), smooth.view(torch.int16))


def test_smooth_k_full_size_sampled_rows():
    """B=1 S=4096 H=24 with per-channel K offsets (where smoothing acts),
    4 heads x 512 sampled rows against the oracle."""
    import quantized_attention_diffusion_gb300 as qad
    w = WORKLOADS["b1_s4096_h24_koffset"]
    q, k, v = make_workload(w)
    out = qad.attn_fwd(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale, smooth_k=True)
    torch.cuda.synchronize()
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=512, seed=w.seed)
    bits = [bf16_bits(t) for t in (q, k, v)]
    quant = oracle.quantize(*bits, smooth_k=True)
    ref, ties = oracle.attend_rows(quant, w.S, w.softmax_scale, rows, return_ties=True)
    got = out.float().cpu().numpy()[rows[:, 0], rows[:, 2], rows[:, 1]]
    err, _ = assert_close_to_oracle(got, f32(ref), ties, w.name)
    err2, used = assert_within_two_pass_bound(got, quant, w.S, w.softmax_scale, rows, ties, w.name + " vs two-pass")
    print(f"{w.name} smooth_k: max-abs vs oracle {err:.4g}; vs two-pass {err2:.4g} ({used:.3f} of the bound)")


@pytest.mark.parametrize("name", ["b1_s4096_h24_koffset", "b2_s16384_h24_outlier", "b1_s65536_h24_koffset"])
def test_smooth_k_accuracy_compared_with_plain(name):
    """The comparison the pages make for smooth_k (InvokeAI PR #9657,
    "Summary": it helps on some heads and hurts on outlier heads): the same
    call with and without K smoothing against unquantized float64 attention
    on 4 heads x 256 sampled rows of the K-offset (4096 and 65536 tokens) and
    outlier-channel (2 x 16384) workloads.  Both must keep the accuracy bar
    (cosine 0.999); the printed cosine and relative L2 are the comparison."""
    import quantized_attention_diffusion_gb300 as qad
    from tests.gpu_common import COS_BAR, cosine
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=256, seed=w.seed + 7)
    rt = torch.from_numpy(rows).long().cuda()
    exact = oracle.attention_fp64(*[bf16_bits(t) for t in (q, k, v)], w.softmax_scale, rows=rows).ravel()
    report = []
    for smooth in (False, True):
        out = qad.attn_fwd(qd, kd, vd, w.softmax_scale, smooth_k=smooth)
        got = out[rt[:, 0], rt[:, 2], rt[:, 1]].double().cpu().numpy().ravel()
        cos = cosine(got, exact)
        rel = float(np.linalg.norm(got - exact) / np.linalg.norm(exact))
        report.append(f"smooth_k={smooth}: cosine {cos:.6f} rel-L2 {rel:.4e}")
        assert cos >= COS_BAR, (name, smooth, cos)
    print(f"{name}: " + "; ".join(report))
