"""CPU oracle for SageAttention-style quantized attention (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports it, and it imports nothing from the product.

Two independent statements of the method live here:

* ``sage_oracle.c`` -- the quantize-then-attend algorithm step by step (INT8
  Q/K per 32-row block, FP8 E4M3 V per channel, exact integer QK^T, FP32
  softmax, FP8 P, exactly summed PV, BF16 output).  Its header lists every
  reading of a point the pages leave open.
* ``fp64_reference.py`` -- unquantized ``softmax(Q K^T * scale) V`` in float64.

BF16 tensors are passed as ``numpy.uint16`` arrays holding the bf16 bit
patterns, shape ``[B, S, H, D]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .fp64_reference import attention_fp64, lse_fp64  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsage_oracle.so")
_CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
           "-shared", "-fPIC", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` (gcc, OpenMP) and return its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_e4m3_decode_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_quantize_qk.argtypes = [P, I, I, I, I, I, P, P]
        lib.oracle_quantize_v.argtypes = [P, I, I, I, I, I, P, P]
        lib.oracle_quantize_k_smooth.argtypes = [P, I, I, I, I, I, P, P, P]
        lib.oracle_qk_int32.restype = I
        lib.oracle_qk_int32.argtypes = [P, P, I, I, I, I, I, P]
        lib.oracle_attend_rows.restype = I
        lib.oracle_attend_rows.argtypes = [P, P, P, P, P, P, I, I, I, I, I,
                                           ctypes.c_float, I, I, P, ctypes.c_int64, P, P, P, P]
        lib.oracle_attend_rows_cross.restype = I
        lib.oracle_attend_rows_cross.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                 ctypes.c_float, I, I, P, ctypes.c_int64, P, P,
                                                 P, P]
        lib.oracle_attend_row_debug.restype = I
        lib.oracle_attend_row_debug.argtypes = [P, P, P, P, P, P, I, I, I, I, I,
                                                ctypes.c_float, I, I, I, I, I, P, P, P, P]
        lib.oracle_requant_bound.restype = I
        lib.oracle_requant_bound.argtypes = [P, P, P, P, I, I, I, I, I, I, I, ctypes.c_float, I,
                                             P, ctypes.c_int64, P]
        lib.oracle_num_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def padded_len(S: int) -> int:
    """Token count of the quantised layouts: S rounded up to a multiple of 128."""
    return (S + 127) // 128 * 128


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ------------------------------------------------------------------ E4M3FN --

def e4m3_encode(y) -> np.ndarray:
    """fp32 values -> E4M3FN codes (RNE, saturating to +-448)."""
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.empty(y.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(y), y.size, _ptr(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    """E4M3FN codes -> exact float64 values."""
    c = np.ascontiguousarray(np.asarray(c, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(_ptr(c), c.size, _ptr(out))
    return out


# ------------------------------------------------------------ quantisation --

def quantize_qk(x: np.ndarray):
    """bf16 bits [B,S,H,D] -> (int8 codes [B,H,S_pad,D], fp32 scales [B,H,ceil(S/32)])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    B, S, H, D = x.shape
    Sp = padded_len(S)
    codes = np.empty((B, H, Sp, D), dtype=np.int8)
    scale = np.empty((B, H, (S + 31) // 32), dtype=np.float32)
    _load().oracle_quantize_qk(_ptr(x), B, S, H, D, Sp, _ptr(codes), _ptr(scale))
    return codes, scale


def quantize_v(v: np.ndarray):
    """bf16 bits [B,S,H,D] -> (E4M3 codes of V^T [B,H,D,S_pad], fp32 scales [B,H,D])."""
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, S, H, D = v.shape
    Sp = padded_len(S)
    vt = np.empty((B, H, D, Sp), dtype=np.uint8)
    vs = np.empty((B, H, D), dtype=np.float32)
    _load().oracle_quantize_v(_ptr(v), B, S, H, D, Sp, _ptr(vt), _ptr(vs))
    return vt, vs


def qk_int32(q_codes: np.ndarray, k_codes: np.ndarray, S: int) -> np.ndarray:
    """Exact integer Q K^T per head: int32 [B,H,S,S]."""
    q_codes = np.ascontiguousarray(q_codes, dtype=np.int8)
    k_codes = np.ascontiguousarray(k_codes, dtype=np.int8)
    B, H, Sp, D = q_codes.shape
    out = np.empty((B, H, S, S), dtype=np.int32)
    rc = _load().oracle_qk_int32(_ptr(q_codes), _ptr(k_codes), B, S, H, D, Sp, _ptr(out))
    if rc != 0:
        raise OverflowError("QK^T sum outside int32")
    return out


# --------------------------------------------------------------- attention --

#: KV tile of the online softmax (reading R7).  The pages fix none; 96 keys
#: (three K blocks) follows the CUDA kernel's tile.  0 selects one tile of
#: all keys: the exact two-pass softmax.
KV_TILE = 96
TWO_PASS = 0


def all_rows(B: int, S: int, H: int) -> np.ndarray:
    """Every (b, h, i) query row, in [B, S, H] output order."""
    b, s, h = np.meshgrid(np.arange(B), np.arange(S), np.arange(H), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), s.ravel()], axis=1).astype(np.int32)


def attend_rows(quant, S: int, softmax_scale: float, rows: np.ndarray, l_mode: int = 0,
                return_ties: bool = False, return_lse: bool = False, Skv: int | None = None,
                kv_tile: int = KV_TILE):
    """Attention output for selected query rows from quantised operands.

    quant = (q_codes, q_scale, k_codes, k_scale, vt_codes, v_scale) in the
    layouts returned by ``quantize_qk`` / ``quantize_v``.  rows: int32 [n, 3]
    of (b, h, i).  Returns bf16 bits [n, D]; with return_ties also each row's
    tie bound (float64 [n]): the most an equally correct rounding of P codes
    that sit on an E4M3 rounding midpoint could move that row's outputs; with
    return_lse also each row's log-sum-exp (reading R13) and its tie bound
    (two float64 [n]), appended in that order.  S is the number of query
    rows; Skv (default S) the number of keys and values (cross-attention,
    reading R14).  kv_tile: the online softmax's KV tile (reading R7; 0 or
    ``TWO_PASS`` for one tile of all keys).
    """
    qc, qs, kc, ks, vt, vs = [np.ascontiguousarray(a) for a in quant]
    B, H, Sp, D = qc.shape
    Skv = S if Skv is None else int(Skv)
    Skv_pad = kc.shape[2]
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    out = np.empty((rows.shape[0], D), dtype=np.uint16)
    ties = np.zeros(rows.shape[0], dtype=np.float64)
    lse = np.zeros(rows.shape[0], dtype=np.float64)
    lse_ties = np.zeros(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_attend_rows_cross(_ptr(qc), _ptr(qs), _ptr(kc), _ptr(ks), _ptr(vt),
                                          _ptr(vs), B, S, Skv, H, D, Sp, Skv_pad,
                                          float(softmax_scale), int(l_mode), int(kv_tile), _ptr(rows),
                                          rows.shape[0], _ptr(out), _ptr(ties), _ptr(lse),
                                          _ptr(lse_ties))
    if rc != 0:
        raise MemoryError("oracle_attend_rows failed to allocate")
    res = (out,)
    if return_ties:
        res += (ties,)
    if return_lse:
        res += (lse, lse_ties)
    return res if len(res) > 1 else out


def attend_row_debug(quant, S: int, softmax_scale: float, b: int, h: int, i: int,
                     l_mode: int = 0, kv_tile: int = KV_TILE):
    """One row with its FP8 P codes and normaliser L: (out bf16 [D], codes [S], L)."""
    qc, qs, kc, ks, vt, vs = [np.ascontiguousarray(a) for a in quant]
    B, H, Sp, D = qc.shape
    out = np.empty(D, dtype=np.uint16)
    pc = np.empty(S, dtype=np.uint8)
    L = ctypes.c_double(0.0)
    tie = ctypes.c_double(0.0)
    rc = _load().oracle_attend_row_debug(_ptr(qc), _ptr(qs), _ptr(kc), _ptr(ks), _ptr(vt),
                                         _ptr(vs), B, S, H, D, Sp, float(softmax_scale),
                                         int(l_mode), int(kv_tile), b, h, i, _ptr(out), _ptr(pc),
                                         ctypes.byref(L), ctypes.byref(tie))
    if rc != 0:
        raise MemoryError("oracle_attend_row_debug failed to allocate")
    return out, pc, L.value


def quantize_k_smooth(k: np.ndarray):
    """K smoothing then quantisation (reading R15): returns (codes int8
    [B, H, S_pad, D], scales fp32 [B, H, nb], channel means fp32 [B, H, D])."""
    k = np.ascontiguousarray(k, dtype=np.uint16)
    B, S, H, D = k.shape
    Sp = padded_len(S)
    codes = np.empty((B, H, Sp, D), dtype=np.int8)
    scale = np.empty((B, H, (S + 31) // 32), dtype=np.float32)
    mean = np.empty((B, H, D), dtype=np.float32)
    _load().oracle_quantize_k_smooth(_ptr(k), B, S, H, D, Sp, _ptr(codes), _ptr(scale), _ptr(mean))
    return codes, scale, mean


def quantize(q: np.ndarray, k: np.ndarray, v: np.ndarray, smooth_k: bool = False):
    """The three quantisation steps: returns (qc, qs, kc, ks, vt, vs); with
    smooth_k, K is smoothed first (R15)."""
    qc, qs = quantize_qk(q)
    kc, ks = quantize_k_smooth(k)[:2] if smooth_k else quantize_qk(k)
    vt, vs = quantize_v(v)
    return qc, qs, kc, ks, vt, vs


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, softmax_scale: float,
              rows: np.ndarray | None = None, l_mode: int = 0, return_ties: bool = False,
              smooth_k: bool = False, kv_tile: int = KV_TILE):
    """Whole quantize-then-attend path from bf16 bits.

    rows None: full output bf16 bits [B,S,H,D] (ties [B,S,H]); otherwise
    bf16 bits [n, D] (ties [n]) for the given (b, h, i) rows.
    """
    B, S, H, D = q.shape
    Skv = k.shape[1]
    quant = quantize(q, k, v, smooth_k=smooth_k)
    if rows is None:
        out, ties = attend_rows(quant, S, softmax_scale, all_rows(B, S, H), l_mode, True, Skv=Skv,
                                kv_tile=kv_tile)
        out, ties = out.reshape(B, S, H, D), ties.reshape(B, S, H)
    else:
        out, ties = attend_rows(quant, S, softmax_scale, rows, l_mode, True, Skv=Skv,
                                kv_tile=kv_tile)
    return (out, ties) if return_ties else out


# ------------------------------------------------- tiling bound (R16) --

def requant_bound(quant, S: int, softmax_scale: float, rows: np.ndarray,
                  kv_tile: int = KV_TILE, Skv: int | None = None) -> np.ndarray:
    """Per row, the factor G of reading R16: the output with KV tiles of
    ``kv_tile`` keys and the two-pass output differ by at most
    ``v_spread(quant)[b, h, d] * G`` in channel d (plus one BF16 ulp).
    G is computed from the exact scores alone.  Returns float64 [n]."""
    qc, qs, kc, ks, _, _ = [np.ascontiguousarray(a) for a in quant]
    B, H, Sp, D = qc.shape
    Skv = S if Skv is None else int(Skv)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    G = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_requant_bound(_ptr(qc), _ptr(qs), _ptr(kc), _ptr(ks), B, S, Skv, H, D, Sp,
                                      kc.shape[2], float(softmax_scale), int(kv_tile), _ptr(rows),
                                      rows.shape[0], _ptr(G))
    if rc != 0:
        raise MemoryError("oracle_requant_bound failed to allocate")
    return G


def v_spread(quant, Skv: int) -> np.ndarray:
    """max - min over the Skv tokens of the dequantised V, per (b, h, d):
    float64 [B, H, D] (the spread_d of reading R16)."""
    _, _, _, _, vt, vs = quant
    dec = e4m3_decode(vt[..., :int(Skv)]) * vs.astype(np.float64)[..., None]
    return dec.max(axis=-1) - dec.min(axis=-1)
