"""Pins for the oracle's optional log-sum-exp output (reading R13 in the
oracle's header): lse_i = ln 2 * (m_i + log2 L_i - log2 448), the natural
log of sum_j exp(scores_ij) as the quantised computation estimates it.

Sources: diffusers PR #15060, "What does this PR do?" (the kernel returns no
LSE; an LSE output is what merging partial attentions needs), and the kernel
contract of diffusers issue #15014 for everything upstream of the row sum.
Each pin derives the expected value from the quantised logits in float64,
not from the oracle's formula.
"""
import math

import numpy as np

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv


def qkv_bits(B, S, H, seed, recipe="normal"):
    return [bf16_bits(t) for t in make_qkv(B, S, H, recipe=recipe, seed=seed)]


def dequant_logits(quant, scale, b, h, i, S):
    """float64 scores scale * (q_hat . k_hat_j) of query row i from the codes."""
    qc, qs, kc, ks, _, _ = quant
    q = qc[b, h, i].astype(np.float64) * float(qs[b, h, i // 32])
    k = kc[b, h, :S].astype(np.float64) * np.repeat(ks[b, h].astype(np.float64), 32)[:S, None]
    return scale * (k @ q)


def lse_of(quant, S, scale, rows):
    _, _, lse, lse_tie = oracle.attend_rows(quant, S, scale, rows, return_ties=True,
                                            return_lse=True)
    return lse, lse_tie


def test_single_key_lse_is_the_logit():
    """One key: P~ = 448 exactly, L = 448, so lse is the (quantised) logit."""
    B, S, H = 2, 1, 3
    scale = 1 / math.sqrt(128)
    quant = oracle.quantize(*qkv_bits(B, S, H, seed=21))
    rows = oracle.all_rows(B, S, H)
    lse, tie = lse_of(quant, S, scale, rows)
    for n, (b, h, i) in enumerate(rows):
        s = dequant_logits(quant, scale, b, h, i, S)[0]
        assert abs(lse[n] - s) <= 1e-6 * (1 + abs(s)), (n, lse[n], s)
    assert np.all(tie == 0)


def test_equal_keys_lse_is_logit_plus_log_count():
    """S identical keys over three KV tiles (96 + 96 + 8): every P~ is 448,
    L = 448 S, lse = s + ln S."""
    B, S, H = 1, 200, 1
    scale = 1 / math.sqrt(128)
    q, k, v = qkv_bits(B, S, H, seed=22)
    k = np.broadcast_to(k[:, :1], k.shape).copy()
    quant = oracle.quantize(q, k, v)
    rows = oracle.all_rows(B, S, H)
    lse, _ = lse_of(quant, S, scale, rows)
    for n, (b, h, i) in enumerate(rows):
        s = dequant_logits(quant, scale, b, h, i, S)
        assert np.ptp(s) == 0.0
        expect = s[0] + math.log(S)
        assert abs(lse[n] - expect) <= 1e-6 * (1 + abs(expect)), (n, lse[n], expect)


def test_two_tile_rescale_closed_form():
    """Tile 0: 96 copies of key a; tile 1: 40 copies of key b = 2a (same codes,
    exactly twice the block scale), so s_b = 2 s_a.  For rows with s_a > 0 the
    running max moves at tile 1 and L is rescaled once; every P~ is 448 and
    lse = log(96 e^{s_a} + 40 e^{s_b})."""
    B, S, H = 1, 136, 1
    scale = 1 / math.sqrt(128)
    q, k, v = [np.asarray(t) for t in qkv_bits(B, S, H, seed=23)]
    ka = k[0, 0, 0].copy()
    kf = (ka.astype(np.uint32) << 16).view(np.float32)
    kb = bf16_bits_from_f32(kf * 2.0)
    k[0, :96, 0] = ka
    k[0, 96:, 0] = kb
    # queries along key a plus noise, so that s_a > 0 for most rows
    qf = (q[0, :, 0].astype(np.uint32) << 16).view(np.float32)
    q[0, :, 0] = bf16_bits_from_f32(0.2 * qf + kf[None, :])
    quant = oracle.quantize(q, k, v)
    assert np.array_equal(quant[2][0, 0, 0], quant[2][0, 0, 100])          # same codes
    assert quant[3][0, 0, 3] == 2 * quant[3][0, 0, 0]                       # twice the scale
    rows = oracle.all_rows(B, S, H)
    lse, _ = lse_of(quant, S, scale, rows)
    checked = 0
    for n, (b, h, i) in enumerate(rows):
        s = dequant_logits(quant, scale, b, h, i, S)
        sa, sb = s[0], s[100]
        if not sa > 0:
            continue
        expect = sb + math.log(96 * math.exp(sa - sb) + 40)
        assert abs(lse[n] - expect) <= 2e-6 * (1 + abs(sb)), (n, lse[n], expect)
        checked += 1
    assert checked > S // 2


def bf16_bits_from_f32(x):
    import torch
    return bf16_bits(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def test_lse_within_quantisation_bound_of_fp64():
    """Against the unquantised float64 log-sum-exp: lse is 1-Lipschitz in the
    max-norm of the logits, and E4M3 rounds each P~ within 1/16 relative (or
    2^-10 absolute below the normal range), so per row
    |lse - lse64| <= max_j |s_hat_j - s_j| + ln(1 + 1/16) + S 2^-10 / 448."""
    B, S, H = 1, 257, 2
    scale = 1 / math.sqrt(128)
    q, k, v = qkv_bits(B, S, H, seed=24, recipe="qk_outlier_channels")
    quant = oracle.quantize(q, k, v)
    rows = oracle.all_rows(B, S, H)
    lse, _ = lse_of(quant, S, scale, rows)
    ref = oracle.lse_fp64(q, k, scale, rows)
    qf = [(np.asarray(t).astype(np.uint32) << 16).view(np.float32).astype(np.float64) for t in (q, k)]
    for n, (b, h, i) in enumerate(rows):
        s_hat = dequant_logits(quant, scale, b, h, i, S)
        s = scale * (qf[1][b, :, h, :] @ qf[0][b, i, h, :])
        bound = np.abs(s_hat - s).max() + math.log1p(1 / 16) + S * 2.0 ** -10 / 448 + 1e-6
        err = abs(lse[n] - ref[n])
        # a dropped ln 2 (|lse| (1/ln 2 - 1)) or log2 448 term (6.1) exceeds it
        assert err <= bound, (n, err, bound)


def test_fp64_lse_matches_logsumexp():
    q, k, _ = qkv_bits(1, 33, 1, seed=25)
    rows = oracle.all_rows(1, 33, 1)
    ref = oracle.lse_fp64(q, k, 0.125, rows)
    qf = (np.asarray(q).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kf = (np.asarray(k).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    s = 0.125 * qf[0, :, 0, :] @ kf[0, :, 0, :].T
    import scipy.special
    assert np.allclose(ref, scipy.special.logsumexp(s, axis=1), rtol=0, atol=1e-12)
