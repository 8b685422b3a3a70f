"""Pins for the oracle's cross-attention reading (R14): Q with Sq rows against
K and V with Skv != Sq rows, each tensor quantised over its own blocks/tokens.

Source: diffusers issue #15014 (the kernel contract assumes equal shapes and
falls back otherwise, "Describe the solution you'd like") and the
SageAttention 2.2 cross-attention results quoted in the InvokeAI PR #9657
thread ("Summary"): shorter K/V is the pages' second workload.
"""
import math

import numpy as np
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv


def bits(B, S, H, seed, recipe="normal"):
    return [bf16_bits(t) for t in make_qkv(B, S, H, recipe=recipe, seed=seed)]


def f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_single_kv_token_returns_v():
    """One key: P~ = 448, L = 448, and V's single token quantises to itself."""
    q, _, _ = bits(2, 70, 3, seed=31)
    _, k, v = bits(2, 1, 3, seed=32)
    out = oracle.attention(q, k, v, 1 / math.sqrt(128))
    assert out.shape == (2, 70, 3, 128)
    assert np.array_equal(out, np.broadcast_to(v, out.shape))


def test_query_prefix_equals_self_attention_rows():
    """Cross-attention of the first 64 query rows (two whole Q blocks) with the
    full K, V equals those rows of self-attention bit for bit, LSE included."""
    B, S, H = 1, 300, 2
    q, k, v = bits(B, S, H, seed=33, recipe="k_channel_offset")
    scale = 1 / math.sqrt(128)
    quant_self = oracle.quantize(q, k, v)
    rows = oracle.all_rows(B, 64, H)
    ref, _, lse_ref, _ = oracle.attend_rows(quant_self, S, scale, rows, return_ties=True,
                                            return_lse=True)
    qp = np.ascontiguousarray(q[:, :64])
    quant_x = oracle.quantize(qp, k, v)
    got, _, lse_got, _ = oracle.attend_rows(quant_x, 64, scale, rows, return_ties=True,
                                            return_lse=True, Skv=S)
    assert np.array_equal(got, ref)
    assert np.array_equal(lse_got, lse_ref)


def test_equal_keys_give_mean_of_dequantised_v():
    Sq, Skv = 45, 150
    q, _, _ = bits(1, Sq, 1, seed=34)
    _, k, v = bits(1, Skv, 1, seed=35)
    k = np.broadcast_to(k[:, :1], k.shape).copy()
    out = oracle.attention(q, k, v, 1 / math.sqrt(128))
    vt, vs = oracle.quantize_v(v)
    mean = oracle.e4m3_decode(vt[0, 0, :, :Skv]).sum(axis=1) * vs[0, 0].astype(np.float64) / Skv
    expect = bf16_bits(torch.tensor(mean.astype(np.float32)).to(torch.bfloat16))
    assert np.array_equal(out[0, :, 0, :], np.broadcast_to(expect, (Sq, 128)))


def test_shorter_and_longer_kv_track_float64():
    """Both directions (Skv < Sq, Skv > Sq, ragged tiles) stay at the pages'
    accuracy bar (cosine 0.9993 against SDPA, rounded down to 0.999) against
    unquantised float64 attention on normally distributed activations, the
    recipe that bar was quoted for in the tiny self-attention pin too."""
    scale = 1 / math.sqrt(128)
    for (Sq, Skv, seed) in [(300, 50, 36), (100, 257, 37), (64, 33, 40)]:
        q, _, _ = bits(1, Sq, 2, seed=seed)
        _, k, v = bits(1, Skv, 2, seed=seed + 100)
        out = oracle.attention(q, k, v, scale)
        ref = oracle.attention_fp64(q, k, v, scale)
        a, b = f64(out).ravel(), ref.ravel()
        cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))
        assert cos >= 0.999, (Sq, Skv, cos)


def test_fp64_reference_cross_matches_torch_sdpa():
    q, _, _ = bits(1, 40, 2, seed=38)
    _, k, v = bits(1, 23, 2, seed=39)
    ref = oracle.attention_fp64(q, k, v, 0.1)
    t = [torch.from_numpy(f64(x)).permute(0, 2, 1, 3) for x in (q, k, v)]
    sdpa = torch.nn.functional.scaled_dot_product_attention(*t, scale=0.1).permute(0, 2, 1, 3)
    assert np.allclose(ref, sdpa.numpy(), rtol=0, atol=1e-12)
