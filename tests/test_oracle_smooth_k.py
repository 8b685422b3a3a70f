"""Pins for the oracle's optional K smoothing (reading R15): subtract each
(batch, head, channel) mean of K over the tokens before quantising K.

Source: InvokeAI PR #9657, "Summary" and "How it works" (SageAttention's
smooth_k, a per-channel K mean subtraction; it is softmax-invariant because
every score of a query row moves by the same q . mean, and on an outlier head
the pages measure it making things worse, relative L2 1.62 against 0.10).
"""
import math

import numpy as np
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv


def bits(B, S, H, seed, recipe="normal"):
    return [bf16_bits(t) for t in make_qkv(B, S, H, recipe=recipe, seed=seed)]


def to_bits(x):
    return bf16_bits(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def zero_mean_int_keys(B, S, H, seed):
    """Integer keys in [-8, 8] whose every channel sums to zero (second half
    of the tokens negates the first), so the channel means are exactly 0."""
    assert S % 2 == 0
    rng = np.random.default_rng(seed)
    half = rng.integers(-8, 9, size=(B, S // 2, H, 128)).astype(np.float32)
    return np.concatenate([half, -half], axis=1)


def test_channel_mean_is_the_exactly_rounded_mean():
    _, k, _ = bits(2, 77, 3, seed=41, recipe="k_channel_offset")
    _, _, mean = oracle.quantize_k_smooth(k)
    kf = f64(k)
    for b in range(2):
        for h in range(3):
            for d in range(128):
                exact = math.fsum(kf[b, :, h, d]) / 77
                assert mean[b, h, d] == np.float32(exact), (b, h, d)


def test_zero_mean_keys_are_left_alone():
    k = to_bits(zero_mean_int_keys(1, 64, 2, seed=42))
    codes_s, scale_s, mean = oracle.quantize_k_smooth(k)
    codes, scale = oracle.quantize_qk(k)
    assert np.all(mean == 0)
    assert np.array_equal(codes_s, codes) and np.array_equal(scale_s, scale)


def test_a_per_channel_offset_is_removed_exactly():
    """K + c (c an integer per head and channel, exact in bf16) smooths to the
    same codes as K itself, and attention with smoothing equals plain
    attention on the zero-mean K bit for bit."""
    B, S, H = 1, 64, 2
    kz = zero_mean_int_keys(B, S, H, seed=43)
    rng = np.random.default_rng(44)
    c = rng.integers(-40, 41, size=(1, 1, H, 128)).astype(np.float32)
    k0, k1 = to_bits(kz), to_bits(kz + c)
    assert np.array_equal(f64(k1), f64(k0) + c)              # the offset is exact in bf16
    codes0, scale0 = oracle.quantize_qk(k0)
    codes1, scale1, mean1 = oracle.quantize_k_smooth(k1)
    assert np.array_equal(mean1, np.broadcast_to(c[0, 0], mean1.shape))
    assert np.array_equal(codes1, codes0) and np.array_equal(scale1, scale0)
    q, _, v = bits(B, S, H, seed=45)
    plain = oracle.attention(q, k0, v, 1 / math.sqrt(128))
    smooth = oracle.attention(q, k1, v, 1 / math.sqrt(128), smooth_k=True)
    assert np.array_equal(plain, smooth)


def test_constant_keys_smooth_to_zero_and_give_the_mean_of_v():
    B, S, H = 1, 50, 1
    q, k, v = bits(B, S, H, seed=46)
    k = np.broadcast_to(k[:, :1], k.shape).copy()
    codes, scale, _ = oracle.quantize_k_smooth(k)
    assert np.all(codes == 0) and np.all(scale == 0)
    out = oracle.attention(q, k, v, 1 / math.sqrt(128), smooth_k=True)
    vt, vs = oracle.quantize_v(v)
    mean_v = oracle.e4m3_decode(vt[0, 0, :, :S]).sum(axis=1) * vs[0, 0].astype(np.float64) / S
    expect = to_bits(mean_v.astype(np.float32))
    assert np.array_equal(out[0, :, 0, :], np.broadcast_to(expect, (S, 128)))


def test_smoothed_attention_tracks_float64():
    """Softmax invariance: with or without smoothing the output stays at the
    pages' accuracy bar (cosine 0.999) against float64 on normal and on
    channel-offset keys."""
    scale = 1 / math.sqrt(128)
    for recipe, seed in [("normal", 47), ("k_channel_offset", 48)]:
        q, k, v = bits(1, 256, 2, seed=seed, recipe=recipe)
        ref = oracle.attention_fp64(q, k, v, scale).ravel()
        for smooth in (False, True):
            out = f64(oracle.attention(q, k, v, scale, smooth_k=smooth)).ravel()
            cos = float(out @ ref / (np.linalg.norm(out) * np.linalg.norm(ref)))
            assert cos >= 0.999, (recipe, smooth, cos)
