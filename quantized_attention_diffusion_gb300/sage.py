"""Thin ctypes binding over ``libsage.so`` (declared in ``include/sage.h``).

The binding marshals torch tensors into pointers, sizes and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or a call fails, a
``SageError`` is raised.

Accepted inputs mirror the kernel contract of diffusers issue #15014
("gfx1201 (RDNA4) SageAttention attention backend", kernel contract bullets):
BF16 Q/K/V of equal shape [B, S, H, 128], no mask, non-causal.  Anything else
(another dtype, head dim, layout or device) is rejected with a clear error, as
that issue's "Describe the solution you'd like" asks.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsage.so")
HEAD_DIM = 128

_STATUS = {
    0: "SAGE_OK", 1: "SAGE_ERR_INVALID_ARG", 2: "SAGE_ERR_UNSUPPORTED", 3: "SAGE_ERR_MISALIGNED",
    4: "SAGE_ERR_CUDA", 5: "SAGE_ERR_NO_MEMORY", 6: "SAGE_ERR_TIMEOUT", 7: "SAGE_ERR_WORKSPACE",
}
EXPORTED = (
    "sage_padded_len", "sage_workspace_bytes", "sage_quantize_qkv", "sage_attn_fwd",
    "sage_attn_fwd_ws", "sage_attn_fwd_quantized", "sage_debug_qk_int32",
    "sage_debug_wait_timeout", "sage_sync_status", "sage_set_wait_timeout_ns",
    "sage_last_error", "sage_status_string", "sage_set_attention_events",
    "sage_quantize_qkv_noalloc", "sage_attn_fwd_lse", "sage_attn_fwd_cross",
    "sage_debug_fused_q", "sage_attn_fwd_fused_q", "sage_quantize_qkv_smooth_k",
    "sage_attn_fwd_smooth_k", "sage_attn_fwd_launches", "sage_debug_staging_codes",
    "sage_debug_inject_fault", "sage_debug_pool_state", "sage_plan_create", "sage_plan_launch",
    "sage_plan_destroy", "sage_plan_create_ex",
)

# Options of sage_plan_create_ex (include/sage.h).
PLAN_SMOOTH_K, PLAN_FUSED_Q = 1, 2

# Fault sites of sage_debug_inject_fault (include/sage.h).
FAULT_NONE, FAULT_POOL_ALLOC, FAULT_QUANT_LAUNCH, FAULT_ATTN_LAUNCH = 0, 1, 2, 3


class SageError(RuntimeError):
    """A non-zero sage_status, with the library's message."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.name = _STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}: {message}")


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libsage.so and declare its signatures (no CUDA call is made)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m quantized_attention_diffusion_gb300.build`")
        lib = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        S = ctypes.c_int
        sigs = {
            "sage_padded_len": (ctypes.c_int64, [I]),
            "sage_attn_fwd_launches": (I, [I, I, I, I, I]),
            "sage_workspace_bytes": (Z, [I, I, I, I]),
            "sage_quantize_qkv": (S, [P, P, P, I, I, I, I, P, P, P, P, P, P, P]),
            "sage_quantize_qkv_noalloc": (S, [P, P, P, I, I, I, I, P, P, P, P, P, P, P]),
            "sage_attn_fwd": (S, [P, P, P, P, I, I, I, I, F, P]),
            "sage_attn_fwd_ws": (S, [P, P, P, P, I, I, I, I, F, P, Z, P]),
            "sage_attn_fwd_lse": (S, [P, P, P, P, P, I, I, I, I, F, P]),
            "sage_attn_fwd_cross": (S, [P, P, P, P, P, I, I, I, I, I, F, P]),
            "sage_plan_create": (S, [P, P, P, P, P, I, I, I, I, I, F, P]),
            "sage_plan_create_ex": (S, [P, P, P, P, P, I, I, I, I, I, F, ctypes.c_uint, P]),
            "sage_plan_launch": (S, [P, P]),
            "sage_plan_destroy": (S, [P]),
            "sage_debug_fused_q": (S, [P, P, P, P, I, I, I, I, F, P, P, P]),
            "sage_attn_fwd_fused_q": (S, [P, P, P, P, I, I, I, I, F, P]),
            "sage_quantize_qkv_smooth_k": (S, [P, P, P, I, I, I, I, P, P, P, P, P, P, P, P]),
            "sage_attn_fwd_smooth_k": (S, [P, P, P, P, I, I, I, I, F, P]),
            "sage_attn_fwd_quantized": (S, [P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]),
            "sage_debug_qk_int32": (S, [P, P, P, P, P, P, P, P, I, I, I, I, F, P, Z, P]),
            "sage_debug_wait_timeout": (S, [ctypes.c_uint64, P]),
            "sage_debug_staging_codes": (S, [P, P, I, I, I, I, P, P, P, P, P]),
            "sage_debug_inject_fault": (S, [I, I]),
            "sage_debug_pool_state": (S, [P, P]),
            "sage_sync_status": (S, [P]),
            "sage_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
            "sage_set_attention_events": (None, [P, P]),
            "sage_last_error": (ctypes.c_char_p, []),
            "sage_status_string": (ctypes.c_char_p, [S]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        msg = _lib.sage_last_error().decode(errors="replace")
        raise SageError(status, msg)


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16 (got {t.dtype})")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, S, H, D] (got {tuple(t.shape)})")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous in [B, S, H, D] order")
    if not (q.shape == k.shape == v.shape):
        raise ValueError(f"Q, K and V must have equal shapes (got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)})")
    if not (q.device == k.device == v.device):
        raise ValueError("Q, K and V must be on one device")
    B, S, H, D = q.shape
    return B, S, H, D


def padded_len(S: int) -> int:
    return int(load_library().sage_padded_len(S))


def attn_fwd_launches(B: int, Sq: int, H: int, Skv: int | None = None, smooth_k: bool = False) -> int:
    """Kernels one sage_attn_fwd (or _lse, _cross, _fused_q; _smooth_k with
    smooth_k) call launches for this shape."""
    n = int(load_library().sage_attn_fwd_launches(B, Sq, Sq if Skv is None else Skv, H, int(smooth_k)))
    if n < 0:
        raise ValueError(f"invalid shape B={B} Sq={Sq} Skv={Skv} H={H}")
    return n


def workspace_bytes(B: int, S: int, H: int, D: int = HEAD_DIM) -> int:
    return int(load_library().sage_workspace_bytes(B, S, H, D))


def attn_fwd(q, k, v, softmax_scale: float | None = None, out=None, workspace=None, fused_q=False,
             smooth_k=False):
    """Quantized attention forward: bf16 [B, S, H, 128] -> bf16 [B, S, H, 128].

    ``workspace`` (optional uint8 CUDA tensor of >= workspace_bytes) selects
    sage_attn_fwd_ws; otherwise the library's stream-ordered pool is used.
    ``fused_q`` selects sage_attn_fwd_fused_q (Q quantised in the attention
    kernel; same result); ``smooth_k`` selects sage_attn_fwd_smooth_k (K loses
    its per-channel mean before quantisation).
    """
    lib = load_library()
    B, S, H, D = _check_qkv(q, k, v)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    with torch.cuda.device(q.device):
        st = _stream(q.device)
        if smooth_k:
            _check(lib.sage_attn_fwd_smooth_k(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D,
                                              float(softmax_scale), st))
        elif fused_q:
            _check(lib.sage_attn_fwd_fused_q(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D,
                                             float(softmax_scale), st))
        elif workspace is None:
            _check(lib.sage_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D,
                                     float(softmax_scale), st))
        else:
            _check(lib.sage_attn_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D,
                                        float(softmax_scale), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), st))
    return out


def attn_fwd_lse(q, k, v, softmax_scale: float | None = None, out=None, lse=None):
    """attn_fwd that also returns each query row's log-sum-exp.

    Returns (out bf16 [B, S, H, 128], lse fp32 [B, H, S]); ``out`` and
    ``lse`` may be given to be filled (sage_attn_fwd_lse).
    """
    lib = load_library()
    B, S, H, D = _check_qkv(q, k, v)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, S) or not lse.is_contiguous() \
            or lse.device != q.device:
        raise ValueError("lse must be a contiguous float32 [B, H, S] tensor on q's device")
    with torch.cuda.device(q.device):
        _check(lib.sage_attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, D,
                                     float(softmax_scale), _stream(q.device)))
    return out, lse


def attn_fwd_cross(q, k, v, softmax_scale: float | None = None, out=None, lse=None,
                   return_lse: bool = False):
    """Cross-attention: q bf16 [B, Sq, H, 128], k and v bf16 [B, Skv, H, 128]
    -> out bf16 [B, Sq, H, 128] (and lse fp32 [B, H, Sq] with return_lse or
    when ``lse`` is given), through sage_attn_fwd_cross."""
    lib = load_library()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda \
                or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, S, H, D]")
    B, Sq, H, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != H or k.shape[3] != D:
        raise ValueError(f"k and v must be [B, Skv, H, D] with B, H, D of q; got {tuple(k.shape)}, "
                         f"{tuple(v.shape)} for q {tuple(q.shape)}")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k and v must be on one device")
    Skv = k.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq)
                            or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, H, Sq] tensor on q's device")
    with torch.cuda.device(q.device):
        _check(lib.sage_attn_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                       _ptr(lse) if lse is not None else None, B, Sq, Skv, H, D,
                                       float(softmax_scale), _stream(q.device)))
    return (out, lse) if lse is not None else out


class Plan:
    """One fixed attention call recorded as a CUDA graph (sage_plan_create_ex):
    q bf16 [B, Sq, H, 128], k and v bf16 [B, Skv, H, 128] (Skv = Sq for
    self-attention), out bf16 [B, Sq, H, 128] and optionally lse fp32
    [B, H, Sq], all fixed at creation.  ``smooth_k`` records attn_fwd_smooth_k
    instead and ``fused_q`` attn_fwd_fused_q (self-attention without lse, one
    at a time).  ``launch()`` replays the call on the current stream, reading
    q, k and v as they are then; launches of one plan must not overlap (one
    stream, or ordered).  ``close()`` (or leaving a ``with`` block) releases
    the graph and its workspace."""

    def __init__(self, q, k, v, softmax_scale: float | None = None, out=None, lse=None, smooth_k: bool = False,
                 fused_q: bool = False):
        lib = load_library()
        for name, t in (("q", q), ("k", k), ("v", v)):
            if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16 or not t.is_cuda \
                    or not t.is_contiguous() or t.dim() != 4:
                raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, S, H, D]")
        B, Sq, H, D = q.shape
        if k.shape != v.shape or k.shape[0] != B or k.shape[2] != H or k.shape[3] != D:
            raise ValueError(f"k and v must be [B, Skv, H, D] with B, H, D of q; got {tuple(k.shape)}, "
                             f"{tuple(v.shape)} for q {tuple(q.shape)}")
        if k.device != q.device or v.device != q.device:
            raise ValueError("q, k and v must be on one device")
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(D)
        if out is None:
            out = torch.empty_like(q)
        if out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous() or out.device != q.device:
            raise ValueError("out must be a contiguous bf16 tensor of q's shape on q's device")
        if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Sq)
                                or not lse.is_contiguous() or lse.device != q.device):
            raise ValueError("lse must be a contiguous float32 [B, H, Sq] tensor on q's device")
        self.q, self.k, self.v, self.out, self.lse = q, k, v, out, lse   # kept alive with the graph
        self.device = q.device
        self._lib = lib
        self._h = ctypes.c_void_p(0)
        with torch.cuda.device(q.device):
            flags = (PLAN_SMOOTH_K if smooth_k else 0) | (PLAN_FUSED_Q if fused_q else 0)
            _check(lib.sage_plan_create_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                           _ptr(lse) if lse is not None else None, B, Sq, k.shape[1], H, D,
                                           float(softmax_scale), flags, ctypes.byref(self._h)))

    def launch(self):
        if not self._h:
            raise RuntimeError("plan is closed")
        with torch.cuda.device(self.device):
            _check(self._lib.sage_plan_launch(self._h, _stream(self.device)))
        return self.out

    def close(self):
        if self._h:
            with torch.cuda.device(self.device):
                st = self._lib.sage_plan_destroy(self._h)
            self._h = ctypes.c_void_p(0)
            _check(st)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            if self._h and self._lib is not None:
                self._lib.sage_plan_destroy(self._h)
                self._h = ctypes.c_void_p(0)
        except Exception:
            pass


def debug_fused_q(q, k, v, softmax_scale: float | None = None):
    """Run sage_attn_fwd's path and return (out, q_i8 [B,H,S_pad,D],
    q_scale [B,H,nb]): the Q codes and scales the attention kernel computed."""
    lib = load_library()
    B, S, H, D = _check_qkv(q, k, v)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    Sp = padded_len(S)
    nb = (S + 31) // 32
    out = torch.empty_like(q)
    q_i8 = torch.zeros((B, H, Sp, D), dtype=torch.int8, device=q.device)
    q_scale = torch.zeros((B, H, nb), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        _check(lib.sage_debug_fused_q(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S, H, D, float(softmax_scale),
                                      _ptr(q_i8), _ptr(q_scale), _stream(q.device)))
    return out, q_i8, q_scale


def quantize_qkv(q, k, v, out=None, noalloc=False):
    """Returns (q_i8 [B,H,S_pad,D], q_scale [B,H,nb], k_i8, k_scale,
    vt_fp8 uint8 [B,H,D,S_pad], v_scale [B,H,D]).

    ``out`` (optional) is a tuple of those six tensors to fill.  With
    ``noalloc`` the call goes to sage_quantize_qkv_noalloc, which uses the
    library's built-in scratch instead of allocating (B*H <= 8192)."""
    lib = load_library()
    if out is not None:
        B, S, H, D = _check_qkv(q, k, v)
        q_i8, q_sc, k_i8, k_sc, vt, v_sc = out
        fn = lib.sage_quantize_qkv_noalloc if noalloc else lib.sage_quantize_qkv
        with torch.cuda.device(q.device):
            _check(fn(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(q_i8), _ptr(q_sc), _ptr(k_i8),
                      _ptr(k_sc), _ptr(vt), _ptr(v_sc), _stream(q.device)))
        return out
    B, S, H, D = _check_qkv(q, k, v)
    Sp = padded_len(S)
    nb = (S + 31) // 32
    dev = q.device
    q_i8 = torch.empty((B, H, Sp, D), dtype=torch.int8, device=dev)
    k_i8 = torch.empty_like(q_i8)
    q_sc = torch.empty((B, H, nb), dtype=torch.float32, device=dev)
    k_sc = torch.empty_like(q_sc)
    vt = torch.empty((B, H, D, Sp), dtype=torch.uint8, device=dev)
    v_sc = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    fn = lib.sage_quantize_qkv_noalloc if noalloc else lib.sage_quantize_qkv
    with torch.cuda.device(dev):
        _check(fn(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(q_i8), _ptr(q_sc),
                  _ptr(k_i8), _ptr(k_sc), _ptr(vt), _ptr(v_sc), _stream(dev)))
    return q_i8, q_sc, k_i8, k_sc, vt, v_sc


def quantize_qkv_smooth_k(q, k, v):
    """sage_quantize_qkv_smooth_k: returns (q_i8, q_scale, k_i8, k_scale,
    vt_fp8, v_scale, k_mean [B,H,D]) with K smoothed before quantisation."""
    lib = load_library()
    B, S, H, D = _check_qkv(q, k, v)
    Sp = padded_len(S)
    nb = (S + 31) // 32
    dev = q.device
    q_i8 = torch.empty((B, H, Sp, D), dtype=torch.int8, device=dev)
    k_i8 = torch.empty_like(q_i8)
    q_sc = torch.empty((B, H, nb), dtype=torch.float32, device=dev)
    k_sc = torch.empty_like(q_sc)
    vt = torch.empty((B, H, D, Sp), dtype=torch.uint8, device=dev)
    v_sc = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    k_mean = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        _check(lib.sage_quantize_qkv_smooth_k(_ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(q_i8), _ptr(q_sc),
                                              _ptr(k_i8), _ptr(k_sc), _ptr(vt), _ptr(v_sc), _ptr(k_mean),
                                              _stream(dev)))
    return q_i8, q_sc, k_i8, k_sc, vt, v_sc, k_mean


def _quant_shape(q_i8, S):
    B, H, Sp, D = q_i8.shape
    if q_i8.dtype != torch.int8 or not q_i8.is_cuda or not q_i8.is_contiguous():
        raise ValueError("q_i8 must be a contiguous int8 CUDA tensor [B, H, S_pad, D]")
    if Sp != padded_len(S):
        raise ValueError(f"S_pad {Sp} does not match S {S}")
    return B, H, D


def attn_fwd_quantized(quant, S: int, softmax_scale: float, out=None, workspace=None,
                       s_out=None):
    """Attention from sage_quantize_qkv outputs.  quant = (q_i8, q_scale,
    k_i8, k_scale, vt_fp8, v_scale).  With ``s_out`` (int32 [B,H,S,S]) the
    debug entry also dumps the integer QK^T accumulators."""
    lib = load_library()
    q_i8, q_sc, k_i8, k_sc, vt, v_sc = quant
    B, H, D = _quant_shape(q_i8, S)
    dev = q_i8.device
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(B, S, H, D), dtype=torch.uint8, device=dev)
    nbytes = workspace.numel() * workspace.element_size()
    with torch.cuda.device(dev):
        st = _stream(dev)
        if s_out is None:
            _check(lib.sage_attn_fwd_quantized(_ptr(q_i8), _ptr(q_sc), _ptr(k_i8), _ptr(k_sc),
                                               _ptr(vt), _ptr(v_sc), _ptr(out), B, S, H, D,
                                               float(softmax_scale), _ptr(workspace), nbytes, st))
        else:
            _check(lib.sage_debug_qk_int32(_ptr(q_i8), _ptr(q_sc), _ptr(k_i8), _ptr(k_sc),
                                           _ptr(vt), _ptr(v_sc), _ptr(out), _ptr(s_out), B, S, H,
                                           D, float(softmax_scale), _ptr(workspace), nbytes, st))
    return out


def debug_qk_int32(quant, S: int, softmax_scale: float):
    """(out bf16 [B,S,H,D], s int32 [B,H,S,S]) from the debug entry point."""
    q_i8 = quant[0]
    B, H, _, D = q_i8.shape
    s_out = torch.empty((B, H, S, S), dtype=torch.int32, device=q_i8.device)
    out = attn_fwd_quantized(quant, S, softmax_scale, s_out=s_out)
    return out, s_out


def debug_wait_timeout(timeout_ns: int, device=None):
    """Launch the bounded-wait probe; returns the status sync_status() reports."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = _stream(dev)
        _check(lib.sage_debug_wait_timeout(int(timeout_ns), st))
        return int(lib.sage_sync_status(st))


def sync_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib.sage_sync_status(_stream(dev)))


def set_wait_timeout_ns(ns: int):
    load_library().sage_set_wait_timeout_ns(int(ns))


def set_attention_events(before=None, after=None):
    """Install (or with no arguments clear) the attention-kernel timing hook.

    ``before``/``after`` are ``torch.cuda.Event`` objects that have been
    recorded at least once (so that their CUDA handles exist)."""
    lib = load_library()
    if before is None or after is None:
        lib.sage_set_attention_events(None, None)
    else:
        lib.sage_set_attention_events(ctypes.c_void_p(before.cuda_event), ctypes.c_void_p(after.cuda_event))


def debug_staging_codes(q, k):
    """The Q/K quantisation exactly as sage_attn_fwd feeds the attention
    kernel: (q16 fp16 [B,H,S_pad,D], q_scale [B,H,nb], k16, k_scale)."""
    lib = load_library()
    B, S, H, D = _check_qkv(q, k, k)
    Sp = padded_len(S)
    nb = (S + 31) // 32
    dev = q.device
    q16 = torch.empty((B, H, Sp, D), dtype=torch.float16, device=dev)
    k16 = torch.empty_like(q16)
    q_sc = torch.empty((B, H, nb), dtype=torch.float32, device=dev)
    k_sc = torch.empty_like(q_sc)
    with torch.cuda.device(dev):
        _check(lib.sage_debug_staging_codes(_ptr(q), _ptr(k), B, S, H, D, _ptr(q16), _ptr(q_sc), _ptr(k16),
                                            _ptr(k_sc), _stream(dev)))
    return q16, q_sc, k16, k_sc


def debug_inject_fault(site: int, skip: int = 0):
    """Arm the library's host-side fault injection (FAULT_* sites)."""
    _check(load_library().sage_debug_inject_fault(int(site), int(skip)))


def debug_pool_state(device=None):
    """(created, used_bytes) of the library's private memory pool on a device."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    created, used = ctypes.c_int(0), ctypes.c_uint64(0)
    with torch.cuda.device(dev):
        _check(lib.sage_debug_pool_state(ctypes.byref(created), ctypes.byref(used)))
    return bool(created.value), int(used.value)
