"""Unquantized attention in float64 (test infrastructure).

TEST INFRASTRUCTURE ONLY: used by the tests and the smoke check as the
accuracy yardstick.  It computes plain ``softmax(Q K^T * softmax_scale) V``
per (batch, head) from the same bf16 inputs, non-causal and without a mask,
the attention the quantized kernel approximates (diffusers issue #15014,
"Is your feature request related to a problem?": BF16 [B, S, H, 128], no
mask, non-causal).  It shares no code with the quantized oracle.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def attention_fp64(q: np.ndarray, k: np.ndarray, v: np.ndarray, softmax_scale: float,
                   rows: np.ndarray | None = None) -> np.ndarray:
    """float64 attention.

    q, k, v: bf16 bits [B, S, H, D].  rows None: returns float64 [B, S, H, D];
    otherwise rows is int [n, 3] of (b, h, i) and the result is float64 [n, D].
    """
    B, S, H, D = q.shape
    if rows is None:
        out = np.empty((B, S, H, D), dtype=np.float64)
        for b in range(B):
            for h in range(H):
                qh = bf16_bits_to_f64(q[b, :, h, :])
                kh = bf16_bits_to_f64(k[b, :, h, :])
                vh = bf16_bits_to_f64(v[b, :, h, :])
                out[b, :, h, :] = _attend(qh, kh, vh, softmax_scale)
        return out
    rows = np.asarray(rows).reshape(-1, 3)
    out = np.empty((rows.shape[0], D), dtype=np.float64)
    heads = {}
    for n, (b, h, i) in enumerate(rows):
        heads.setdefault((int(b), int(h)), []).append((n, int(i)))
    for (b, h), items in heads.items():
        idx = np.array([n for n, _ in items])
        qi = np.array([i for _, i in items])
        qh = bf16_bits_to_f64(q[b, qi, h, :])
        kh = bf16_bits_to_f64(k[b, :, h, :])
        vh = bf16_bits_to_f64(v[b, :, h, :])
        out[idx] = _attend(qh, kh, vh, softmax_scale)
    return out


def _attend(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, scale: float) -> np.ndarray:
    s = (qh @ kh.T) * scale
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ vh


def lse_fp64(q: np.ndarray, k: np.ndarray, softmax_scale: float,
             rows: np.ndarray) -> np.ndarray:
    """float64 log-sum-exp of the scaled scores, ``log sum_j exp(scale q_i.k_j)``.

    q, k: bf16 bits [B, S, H, D]; rows int [n, 3] of (b, h, i).  Returns
    float64 [n].  The max is subtracted before exponentiating.
    """
    rows = np.asarray(rows).reshape(-1, 3)
    out = np.empty(rows.shape[0], dtype=np.float64)
    for n, (b, h, i) in enumerate(rows):
        qi = bf16_bits_to_f64(q[int(b), int(i), int(h), :])
        kh = bf16_bits_to_f64(k[int(b), :, int(h), :])
        s = (kh @ qi) * softmax_scale
        m = s.max()
        out[n] = m + np.log(np.exp(s - m).sum())
    return out
