"""Pins for the oracle's KV tiling (reading R7), its two-pass form and the
bound that links them (reading R16), and for the value of the tie bound
(R12).

Source: diffusers issue #15014, "Is your feature request related to a
problem?" (kernel contract: softmax in FP32, P requantised to FP8 for PV).
The pages fix no KV tile.  The oracle's default tile, 96 keys, follows the
CUDA kernel; tile 0 is one tile holding every key, the exact two-pass softmax
(the row's true max, no rescale).  These tests pin what the tile changes and
bound it independently of any tile.
"""
import math

import numpy as np
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import (WORKLOADS, bf16_bits, make_workload,
                                                          sample_rows)

L2E = np.float32(1.4426950408889634)
LOG2_448 = np.float32(math.log2(448.0))


def bf16(x):
    return bf16_bits(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_ulp(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    return np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7)


def _two_key_row(first_is_max: bool, softmax_scale: float):
    """One query (channel 0 = 127, so its block scale is 1) and two keys with
    channel-0 codes 126 and 127 (K scale 1).  V channel d is +2^(d%4) at key 0
    and -2^(d%4) at key 1, so every V code is +-448 and sv = 2^(d%4)/448."""
    D = 128
    q = np.zeros((1, 2, 1, D), np.float32)
    k = np.zeros((1, 2, 1, D), np.float32)
    v = np.zeros((1, 2, 1, D), np.float32)
    q[0, :, 0, 0] = 127.0
    k[0, :, 0, 0] = [127.0, 126.0] if first_is_max else [126.0, 127.0]
    pw = 2.0 ** (np.arange(D) % 4)
    v[0, 0, 0, :] = pw
    v[0, 1, 0, :] = -pw
    quant = oracle.quantize(bf16(q), bf16(k), bf16(v))
    assert quant[1][0, 0, 0] == 1.0 and quant[3][0, 0, 0] == 1.0
    return quant, pw


def test_tile_of_one_key_rescales_instead_of_requantising():
    """Lower-scoring key first, tiles of one key: key 0 is coded against its
    own max (448) and later multiplied by alpha = fp32(2^(x0 - x1)), while the
    two-pass form codes it once as e4m3(448 * 2^(x0 - x1)).

    softmax_scale 2^-11: x1 - x0 = 127 * 2^-11 * log2 e = 0.0895, alpha =
    0.9399, 448 alpha = 421.1, whose E4M3 code is 416 (grid step 32).  So
    tile 1: L = 448 alpha + 448, out = 2^(d%4) (alpha - 1) / (alpha + 1);
    two-pass: L = 864, out = 2^(d%4) (416 - 448) / 864 = -2^(d%4) / 27."""
    scale = 2.0 ** -11
    quant, pw = _two_key_row(first_is_max=False, softmax_scale=scale)
    c = np.float32(np.float32(scale) * L2E)                 # c_row = sq * c, sq = 1; cb = c_row * 1
    x0, x1 = np.float32(126 * 127) * c, np.float32(127 * 127) * c
    alpha = float(np.float32(2.0 ** float(np.float32(x0 - x1))))
    assert 0.93 < alpha < 0.95

    out_t, codes_t, L_t = oracle.attend_row_debug(quant, 2, scale, 0, 0, 0, kv_tile=1)
    assert list(oracle.e4m3_decode(codes_t)) == [448.0, 448.0]
    assert abs(L_t - 448.0 * (alpha + 1.0)) <= 1e-12 * L_t
    expect_t = (pw * (alpha - 1.0) / (alpha + 1.0)).astype(np.float32)
    assert np.allclose(f32(out_t), expect_t, rtol=2.0 ** -8, atol=0)

    out_0, codes_0, L_0 = oracle.attend_row_debug(quant, 2, scale, 0, 0, 0, kv_tile=oracle.TWO_PASS)
    assert list(oracle.e4m3_decode(codes_0)) == [416.0, 448.0] and L_0 == 864.0
    assert np.array_equal(f32(out_0), f32(bf16(-pw / 27.0)))
    assert not np.array_equal(out_t, out_0)

    # the bound of R16 covers the difference, and is not zero here
    rows = np.array([[0, 0, 0]], np.int32)
    G = oracle.requant_bound(quant, 2, scale, rows, kv_tile=1)[0]
    spread = oracle.v_spread(quant, 2)[0, 0]
    assert G > 0
    diff = np.abs(f32(out_t).astype(np.float64) - f32(out_0))
    assert np.all(diff <= spread * G + bf16_ulp(np.maximum(np.abs(f32(out_t)), np.abs(f32(out_0)))))


def test_max_first_leaves_nothing_to_rescale():
    """Max-scoring key first: the running max never moves, so tiles of one
    key give the two-pass codes, normaliser and output bit for bit, and the
    bound of R16 is exactly 0."""
    scale = 2.0 ** -11
    quant, _ = _two_key_row(first_is_max=True, softmax_scale=scale)
    a = oracle.attend_row_debug(quant, 2, scale, 0, 0, 0, kv_tile=1)
    b = oracle.attend_row_debug(quant, 2, scale, 0, 0, 0, kv_tile=oracle.TWO_PASS)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2]
    assert oracle.requant_bound(quant, 2, scale, np.array([[0, 0, 0]], np.int32), kv_tile=1)[0] == 0.0


def test_a_tile_holding_every_key_is_the_two_pass_form():
    w = WORKLOADS["b1_s256_h2"]
    bits = [bf16_bits(t) for t in make_workload(w)]
    quant = oracle.quantize(*bits)
    rows = oracle.all_rows(w.B, w.S, w.H)
    two_pass = oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=oracle.TWO_PASS)
    for tile in (w.S, w.S + 1, 10 ** 6):
        assert np.array_equal(oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=tile),
                              two_pass)


def test_rows_whose_max_is_in_the_first_tile_match_two_pass_exactly():
    """Reading R16's premise: only keys of tiles before the one holding the
    row max can weigh differently.  Rows whose max sits in tile 0 (G = 0)
    are bit-identical to the two-pass output; the others are not all."""
    w = WORKLOADS["b1_s256_h2"]
    bits = [bf16_bits(t) for t in make_workload(w)]
    quant = oracle.quantize(*bits)
    rows = oracle.all_rows(w.B, w.S, w.H)
    G = oracle.requant_bound(quant, w.S, w.softmax_scale, rows, kv_tile=96)
    tiled = oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=96)
    two_pass = oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=oracle.TWO_PASS)
    same = np.all(tiled == two_pass, axis=1)
    assert (G == 0).sum() > 50 and (G > 0).sum() > 50
    assert np.all(same[G == 0])
    assert not np.all(same[G > 0])
    # the row max's tile, found from the integer scores, agrees with G = 0
    s = oracle.qk_int32(quant[0], quant[2], w.S).astype(np.float64)
    for n in np.flatnonzero(G == 0)[:20]:
        b, h, i = rows[n]
        x = s[b, h, i] * quant[3][b, h, np.arange(w.S) // 32]
        assert np.argmax(x) < 96


def _bound_check(name, rows, tiles):
    w = WORKLOADS[name]
    bits = [bf16_bits(t) for t in make_workload(w)]
    quant = oracle.quantize(*bits)
    spread = oracle.v_spread(quant, w.S)[rows[:, 0], rows[:, 1]]
    two_pass = f32(oracle.attend_rows(quant, w.S, w.softmax_scale, rows,
                                      kv_tile=oracle.TWO_PASS)).astype(np.float64)
    worst = 0.0
    for tile in tiles:
        tiled = f32(oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=tile)).astype(np.float64)
        G = oracle.requant_bound(quant, w.S, w.softmax_scale, rows, kv_tile=tile)
        bound = spread * G[:, None] + bf16_ulp(np.maximum(np.abs(tiled), np.abs(two_pass)))
        diff = np.abs(tiled - two_pass)
        assert np.all(diff <= bound), (name, tile, float((diff - bound).max()))
        worst = max(worst, float((diff / bound).max()))
    return worst


def test_requant_bound_holds_on_the_small_workload_every_row():
    rows = oracle.all_rows(1, 256, 2)
    assert _bound_check("b1_s256_h2", rows, (1, 7, 32, 96, 128)) < 1.0


def test_requant_bound_holds_on_the_4096_token_workload_sampled_rows():
    w = WORKLOADS["b1_s4096_h24_koffset"]
    rows = sample_rows(w.B, w.S, w.H, heads=4, rows_per_head=192, seed=w.seed)
    assert _bound_check(w.name, rows, (96, 1)) < 1.0


def test_requant_bound_is_tight_enough_to_catch_a_planted_scale_error():
    """A 1% error in softmax_scale on the two-pass side breaks the bound on
    many outputs: the check is not vacuous."""
    w = WORKLOADS["b1_s256_h2"]
    bits = [bf16_bits(t) for t in make_workload(w)]
    quant = oracle.quantize(*bits)
    rows = oracle.all_rows(w.B, w.S, w.H)
    tiled = f32(oracle.attend_rows(quant, w.S, w.softmax_scale, rows, kv_tile=96)).astype(np.float64)
    wrong = f32(oracle.attend_rows(quant, w.S, w.softmax_scale * 1.01, rows,
                                   kv_tile=oracle.TWO_PASS)).astype(np.float64)
    G = oracle.requant_bound(quant, w.S, w.softmax_scale, rows, kv_tile=96)
    spread = oracle.v_spread(quant, w.S)[rows[:, 0], rows[:, 1]]
    bound = spread * G[:, None] + bf16_ulp(np.maximum(np.abs(tiled), np.abs(wrong)))
    assert (np.abs(tiled - wrong) > bound).sum() > 1000


def _midpoint_row(p_target: float):
    """One query row against two keys whose P codes are 448 and e4m3(p1),
    p1 = 448 * 2^(x1 - x0) aimed at p_target.  The query's channel 0 has
    code 1 (channel 5 = 127 fixes its block scale at 1), the keys' channel 0
    codes are 1 and 0 (channel 6 = 127 fixes the K scale at 1), so the
    scores are x0 = cb and x1 = 0 with cb = fl(softmax_scale * log2 e): with
    p1 = 2^(LOG2_448 - cb) small rounding errors only.  V channel d is
    2^(d%4) at key 0 and 0 at key 1, so vmax = 448 * max sv = 8."""
    D = 128
    cb_target = float(LOG2_448) - math.log2(p_target)
    scale = float(np.float32(cb_target / float(L2E)))
    q = np.zeros((1, 2, 1, D), np.float32)          # row 1 stays zero
    k = np.zeros((1, 2, 1, D), np.float32)
    v = np.zeros((1, 2, 1, D), np.float32)
    q[0, 0, 0, 0], q[0, 0, 0, 5] = 1.0, 127.0
    k[0, 0, 0, 0] = 1.0
    k[0, :, 0, 6] = 127.0
    v[0, 0, 0, :] = 2.0 ** (np.arange(D) % 4)
    quant = oracle.quantize(bf16(q), bf16(k), bf16(v))
    return quant, scale


def test_tie_bound_value_at_an_e4m3_midpoint():
    """p1 within 2^-19 of 8.5, the midpoint of the E4M3 neighbours 8 and 9
    (grid step 1 in [8, 16)): the row's tie bound is exactly
    step * 2 * vmax / (L - step) = 2 vmax / (L - 1), vmax = 448 max sv ~ 8,
    with L = 448 + dec(code1) (8 or 9, whichever side p1 fell on); just off
    the midpoint it is 0."""
    quant, scale = _midpoint_row(8.5)
    kc = quant[2]
    assert kc[0, 0, 0, 0] == 1 and kc[0, 0, 1, 0] == 0 and quant[1][0, 0, 0] == 1.0
    rows = np.array([[0, 0, 0]], np.int32)
    _, codes, L = oracle.attend_row_debug(quant, 2, scale, 0, 0, 0, kv_tile=oracle.TWO_PASS)
    p1 = oracle.e4m3_decode(codes)[1]
    assert p1 in (8.0, 9.0) and oracle.e4m3_decode(codes)[0] == 448.0
    assert L == 448.0 + p1
    _, ties = oracle.attend_rows(quant, 2, scale, rows, return_ties=True)
    vmax = 448.0 * float(quant[5].max())              # fp32 sv = fl(8 / 448): vmax ~ 8
    assert abs(vmax - 8.0) < 1e-6
    assert ties[0] == 1.0 * 2.0 * vmax / (L - 1.0)
    quant_off, scale_off = _midpoint_row(8.4)
    _, ties_off = oracle.attend_rows(quant_off, 2, scale_off, rows, return_ties=True)
    assert ties_off[0] == 0.0


def test_requant_bound_holds_for_cross_attention():
    """Reading R14 with R16: a short query block against longer and shorter
    key/value sequences (ragged lengths), every row, tiles 96 and 1."""
    from quantized_attention_diffusion_gb300.workloads import make_qkv
    for (Sq, Skv, seed) in [(40, 333, 60), (200, 97, 61)]:
        q, k, v = [bf16_bits(t) for t in make_qkv(1, Sq, 2, recipe="k_channel_offset", seed=seed, Skv=Skv)]
        quant = oracle.quantize(q, k, v)
        rows = oracle.all_rows(1, Sq, 2)
        scale = 1 / math.sqrt(128)
        spread = oracle.v_spread(quant, Skv)[rows[:, 0], rows[:, 1]]
        two_pass = f32(oracle.attend_rows(quant, Sq, scale, rows, kv_tile=oracle.TWO_PASS,
                                          Skv=Skv)).astype(np.float64)
        for tile in (96, 1):
            tiled = f32(oracle.attend_rows(quant, Sq, scale, rows, kv_tile=tile, Skv=Skv)).astype(np.float64)
            G = oracle.requant_bound(quant, Sq, scale, rows, kv_tile=tile, Skv=Skv)
            bound = spread * G[:, None] + bf16_ulp(np.maximum(np.abs(tiled), np.abs(two_pass)))
            assert np.all(np.abs(tiled - two_pass) <= bound), (Sq, Skv, tile)
            if tile == 96 and Skv <= 96:
                assert np.all(G == 0) and np.array_equal(tiled, two_pass)
