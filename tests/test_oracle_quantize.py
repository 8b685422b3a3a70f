"""Pins for the oracle's Q/K INT8 and V FP8 quantisation and its integer QK^T.

Source: diffusers issue #15014, "Is your feature request related to a
problem?", kernel contract bullets -- Q/K quantized per 32-row block, V per
channel; INT8 QK^T with FP32 accumulation.  Readings (one FP32 scale per 32
tokens of a head, symmetric +-127, V per (batch, head, channel) over all
tokens, E4M3FN) are listed in the oracle's header.  Each test checks a
property that a plausible slip (wrong block axis, crossing heads, transposed
layout, dropped clamp, wrong divisor) would break.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv


def bf16(x):
    return bf16_bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rand_bits(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return bf16_bits((torch.randn(shape, generator=g) * scale).to(torch.bfloat16))


# ---------------------------------------------------------------- Q / K --

def test_single_nonzero_element_maps_to_127():
    x = np.zeros((1, 64, 1, 128), dtype=np.float32)
    x[0, 37, 0, 5] = -3.25
    codes, scale = oracle.quantize_qk(bf16(x))
    assert codes.shape == (1, 1, 128, 128) and scale.shape == (1, 1, 2)
    assert scale[0, 0, 0] == 0.0                       # block 0 is all zero
    assert scale[0, 0, 1] == np.float32(3.25) / np.float32(127)
    expect = np.zeros_like(codes)
    expect[0, 0, 37, 5] = -127
    assert np.array_equal(codes, expect)


def test_sign_symmetry_and_power_of_two_scaling():
    x = rand_bits((2, 100, 3, 128), seed=1)
    c0, s0 = oracle.quantize_qk(x)
    c1, s1 = oracle.quantize_qk(x ^ np.uint16(0x8000))            # negate
    assert np.array_equal(c1, -c0) and np.array_equal(s1, s0)
    for k in (-3, -1, 2, 5):
        xk = bf16(f32(x) * np.float32(2.0 ** k))                   # exact in bf16
        ck, sk = oracle.quantize_qk(xk)
        assert np.array_equal(ck, c0)
        assert np.array_equal(sk, s0 * np.float32(2.0 ** k))


def test_code_range_max_element_and_dequant_error():
    x = rand_bits((1, 320, 2, 128), seed=2, scale=3.0)
    codes, scale = oracle.quantize_qk(x)
    assert codes.min() >= -127 and codes.max() <= 127
    xf = f32(x).astype(np.float64)
    for h in range(2):
        for blk in range(10):
            rows = xf[0, 32 * blk:32 * blk + 32, h, :]
            c = codes[0, h, 32 * blk:32 * blk + 32, :].astype(np.float64)
            sc = float(scale[0, h, blk])
            i = np.unravel_index(np.argmax(np.abs(rows)), rows.shape)
            assert abs(c[i]) == 127 and np.sign(c[i]) == np.sign(rows[i])
            # rint error 1/2 plus the fp32 rounding of x / scale (|x/scale| <= 127)
            assert np.all(np.abs(c * sc - rows) <= sc * (0.5 + 127 * 2.0 ** -24))


def test_blocks_are_32_tokens_of_one_head():
    B, S, H = 2, 200, 3
    x = rand_bits((B, S, H, 128), seed=3)
    c0, s0 = oracle.quantize_qk(x)
    xf = f32(x).copy()
    xf[1, 77, 2, 9] = 1000.0                                         # token 77 -> block 2
    c1, s1 = oracle.quantize_qk(bf16(xf))
    changed = np.argwhere(s1 != s0)
    assert changed.tolist() == [[1, 2, 2]]
    diff = np.argwhere(np.any(c1 != c0, axis=-1))
    assert set(map(tuple, diff[:, :3].tolist())) <= {(1, 2, t) for t in range(64, 96)}


def test_tail_block_and_padding_rows():
    S = 70                                    # blocks of 32, 32, 6 rows; padded to 128
    x = rand_bits((1, S, 1, 128), seed=4)
    codes, scale = oracle.quantize_qk(x)
    assert codes.shape == (1, 1, 128, 128) and scale.shape == (1, 1, 3)
    assert np.all(codes[0, 0, S:, :] == 0)
    tail = f32(x)[0, 64:70, 0, :]
    assert scale[0, 0, 2] == np.float32(np.abs(tail).max()) / np.float32(127)


def test_layout_is_b_h_s_d():
    B, S, H = 2, 40, 3
    x = np.zeros((B, S, H, 128), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            x[b, 5 + b, h, 7 + h] = 1.0 + b + 2 * h                   # the block max
    codes, scale = oracle.quantize_qk(bf16(x))
    for b in range(B):
        for h in range(H):
            assert codes[b, h, 5 + b, 7 + h] == 127
            assert np.count_nonzero(codes[b, h]) == 1
            assert scale[b, h, 0] == np.float32(1.0 + b + 2 * h) / np.float32(127)


def test_zero_block_has_zero_scale_and_codes():
    x = np.zeros((1, 33, 1, 128), dtype=np.float32)
    x[0, 32, 0, 0] = 0.5
    codes, scale = oracle.quantize_qk(bf16(x))
    assert scale[0, 0, 0] == 0.0 and np.all(codes[0, 0, :32] == 0)
    assert codes[0, 0, 32, 0] == 127


# -------------------------------------------------------------------- V --

def test_v_channel_max_maps_to_448_and_error_bound():
    v = rand_bits((1, 300, 2, 128), seed=5, scale=2.0)
    vt, vs = oracle.quantize_v(v)
    assert vt.shape == (1, 2, 128, 384) and vs.shape == (1, 2, 128)
    assert np.all(vt[..., 300:] == 0)
    vf = f32(v).astype(np.float64)
    dec = oracle.e4m3_decode(vt[..., :300])                        # [1, 2, 128, 300]
    for h in range(2):
        col = vf[0, :, h, :].T                                     # [128, 300]
        amax = np.abs(col).max(axis=1)
        assert np.array_equal(vs[0, h], (amax.astype(np.float32) / np.float32(448)))
        arg = np.abs(col).argmax(axis=1)
        peak = vt[0, h, np.arange(128), arg]
        assert np.all((peak & 0x7F) == 0x7E)
        y = col / vs[0, h][:, None].astype(np.float64)
        a = np.abs(y)
        quantum = np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3)
        assert np.all(np.abs(dec[0, h] - y) <= quantum / 2 * (1 + 1e-6))


def test_v_scale_is_per_batch_head_channel():
    v = rand_bits((2, 64, 3, 128), seed=6)
    vt0, vs0 = oracle.quantize_v(v)
    vf = f32(v).copy()
    vf[1, 10, 0, 99] = 500.0
    vt1, vs1 = oracle.quantize_v(bf16(vf))
    assert np.argwhere(vs1 != vs0).tolist() == [[1, 0, 99]]
    rows = np.argwhere(np.any(vt1 != vt0, axis=-1)).tolist()
    assert rows == [[1, 0, 99]]


def test_v_constant_and_zero_channels():
    v = np.zeros((1, 50, 1, 128), dtype=np.float32)
    v[0, :, 0, 3] = -2.5
    v[0, :, 0, 4] = 7.0
    vt, vs = oracle.quantize_v(bf16(v))
    assert np.all(vt[0, 0, 3, :50] == 0xFE) and np.all(vt[0, 0, 4, :50] == 0x7E)
    assert vs[0, 0, 0] == 0.0 and np.all(vt[0, 0, 0] == 0)


# ---------------------------------------------------------------- QK^T --

def test_qk_int32_equals_bruteforce_integer_matmul():
    q, k, _ = make_qkv(2, 150, 3, recipe="k_channel_offset", seed=8)
    qc, _ = oracle.quantize_qk(bf16_bits(q))
    kc, _ = oracle.quantize_qk(bf16_bits(k))
    s = oracle.qk_int32(qc, kc, 150)
    ref = np.einsum("bhic,bhjc->bhij", qc[:, :, :150].astype(np.int64),
                    kc[:, :, :150].astype(np.int64))
    assert np.array_equal(s, ref)


def test_qk_int32_chunk_additivity_and_extremes():
    q, k, _ = make_qkv(1, 64, 1, seed=9)
    qc, _ = oracle.quantize_qk(bf16_bits(q))
    kc, _ = oracle.quantize_qk(bf16_bits(k))
    full = oracle.qk_int32(qc, kc, 64).astype(np.int64)
    parts = np.zeros_like(full)
    for c0 in range(0, 128, 32):
        qm = np.zeros_like(qc)
        qm[..., c0:c0 + 32] = qc[..., c0:c0 + 32]
        parts += oracle.qk_int32(qm, kc, 64)
    assert np.array_equal(parts, full)
    one = np.full((1, 1, 128, 128), 127, dtype=np.int8)
    neg = -one
    assert oracle.qk_int32(one, one, 2)[0, 0, 0, 0] == 128 * 127 * 127
    assert oracle.qk_int32(one, neg, 2)[0, 0, 1, 1] == -128 * 127 * 127


@pytest.mark.parametrize("S", [1, 31, 33])
def test_odd_lengths_pad_to_128(S):
    x = rand_bits((1, S, 1, 128), seed=S)
    codes, scale = oracle.quantize_qk(x)
    assert codes.shape[2] == 128 and scale.shape[2] == (S + 31) // 32
    assert np.all(codes[0, 0, S:] == 0)
    vt, vs = oracle.quantize_v(x)
    assert vt.shape[3] == 128 and np.all(vt[..., S:] == 0)
