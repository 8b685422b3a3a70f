"""The C ABI without a GPU: the library loads, exports every entry point that
include/sage.h declares, and rejects bad arguments on the host before any
CUDA call (diffusers issue #15014, "Describe the solution you'd like":
unsupported inputs are rejected with a clear error; diffusers PR #15060,
"Tests": head dim 64, fp32, cross-attention, causal and masked calls are
not taken by the kernel)."""
import ctypes
import os
import re

import pytest

import quantized_attention_diffusion_gb300 as qad
from quantized_attention_diffusion_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sage.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, NOMEM, TIMEOUT, WORKSPACE = range(8)
FAKE = 0x10000          # a 256-byte aligned, never dereferenced address
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qad.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sage_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(qad.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_no_cuda_runtime_dependency_on_host_checks(lib):
    assert lib.sage_padded_len(1) == 128
    assert lib.sage_padded_len(128) == 128
    assert lib.sage_padded_len(32760) == 32768
    assert lib.sage_padded_len(0) == 0
    assert lib.sage_status_string(TIMEOUT) == b"SAGE_ERR_TIMEOUT"


def test_launch_count(lib):
    assert lib.sage_attn_fwd_launches(2, 16384, 16384, 24, 0) == 4
    assert lib.sage_attn_fwd_launches(2, 16384, 16384, 24, 1) == 6
    assert lib.sage_attn_fwd_launches(2, 16384, 333, 24, 0) == 4
    assert lib.sage_attn_fwd_launches(0, 16, 16, 1, 0) == -1
    assert lib.sage_attn_fwd_launches(1, 16, 0, 1, 0) == -1
    assert qad.attn_fwd_launches(2, 16384, 24) == 4
    assert qad.attn_fwd_launches(2, 16384, 24, smooth_k=True) == 6


def test_workspace_bytes(lib):
    B, S, H = 1, 4096, 24
    n = lib.sage_workspace_bytes(B, S, H, 128)
    # fp16 Q/K codes (2 B each), E4M3 V^T (1 B), scales and channel maxima
    assert n >= B * H * 4096 * 128 * 5
    assert n < B * H * 4096 * 128 * 5 + (1 << 20)
    assert lib.sage_workspace_bytes(B, S, H, 64) == 0
    assert lib.sage_workspace_bytes(0, S, H, 128) == 0


def _fwd(lib, D=128, B=1, S=64, H=2, scale=0.125, q=FAKE, k=FAKE, v=FAKE, out=FAKE):
    return lib.sage_attn_fwd(P(q), P(k), P(v), P(out), B, S, H, D, scale, None)


def test_head_dim_other_than_128_is_unsupported(lib):
    assert _fwd(lib, D=64) == UNSUPPORTED
    assert b"128" in lib.sage_last_error()


@pytest.mark.parametrize("B,S,H", [(0, 64, 2), (1, 0, 2), (1, 64, 0), (-1, 64, 2)])
def test_empty_or_negative_sizes_are_invalid(lib, B, S, H):
    assert _fwd(lib, B=B, S=S, H=H) == INVALID


@pytest.mark.parametrize("scale", [float("nan"), float("inf"), 0.0, -0.1])
def test_bad_softmax_scale_is_invalid(lib, scale):
    assert _fwd(lib, scale=scale) == INVALID


def test_null_and_misaligned_pointers(lib):
    assert _fwd(lib, q=0) == INVALID
    assert b"q is NULL" in lib.sage_last_error()
    assert _fwd(lib, v=FAKE + 8) == MISALIGNED
    assert b"v is not 16-byte aligned" in lib.sage_last_error()
    # the attention kernel writes output rows as 32-byte vectors
    assert _fwd(lib, out=FAKE + 16) == MISALIGNED
    assert b"out is not 32-byte aligned" in lib.sage_last_error()
    h = ctypes.c_void_p(0)
    assert lib.sage_plan_create(P(FAKE), P(FAKE), P(FAKE), P(FAKE + 16), None, 1, 256, 256, 2, 128, 0.1,
                                ctypes.byref(h)) == MISALIGNED


def test_workspace_checks(lib):
    need = lib.sage_workspace_bytes(1, 64, 2, 128)
    st = lib.sage_attn_fwd_ws(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 64, 2, 128, 0.1, P(FAKE),
                              need - 1, None)
    assert st == WORKSPACE
    st = lib.sage_attn_fwd_ws(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 64, 2, 128, 0.1,
                              P(FAKE + 16), need, None)
    assert st == MISALIGNED
    st = lib.sage_attn_fwd_quantized(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE),
                                     P(FAKE), 1, 64, 2, 128, 0.1, P(0), need, None)
    assert st == INVALID


def test_quantize_and_debug_entry_checks(lib):
    st = lib.sage_quantize_qkv(P(FAKE), P(FAKE), P(FAKE), 1, 64, 2, 96, *[P(FAKE)] * 6, None)
    assert st == UNSUPPORTED
    st = lib.sage_quantize_qkv(P(FAKE), P(FAKE), P(FAKE), 1, 64, 2, 128, P(FAKE), P(FAKE + 4),
                               P(FAKE), P(FAKE), P(FAKE), P(FAKE), None)
    assert st == MISALIGNED
    st = lib.sage_debug_qk_int32(*[P(FAKE)] * 7, P(0), 1, 64, 2, 128, 0.1, P(FAKE), 1 << 30, None)
    assert st == INVALID
    assert lib.sage_debug_wait_timeout(0, None) == INVALID


def test_binding_rejects_what_the_kernel_cannot_take():
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 8, 1, 128), dtype=torch.float32)
    with pytest.raises(ValueError, match="bfloat16"):
        qad.attn_fwd(q, q, q)
    qb = torch.zeros((1, 8, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        qad.attn_fwd(qb, qb, qb)
    kb = torch.zeros((1, 4, 1, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        qad.attn_fwd(qb, kb, kb)      # cross-attention shape (shorter K/V)


def test_test_hooks_check_their_arguments_on_the_host(lib):
    assert lib.sage_debug_inject_fault(4, 0) == INVALID
    assert lib.sage_debug_inject_fault(-1, 0) == INVALID
    assert lib.sage_debug_inject_fault(1, -1) == INVALID
    assert b"out of range" in lib.sage_last_error()
    assert lib.sage_debug_inject_fault(0, 0) == OK          # disarm: no CUDA call
    assert lib.sage_debug_pool_state(None, None) == INVALID
    st = lib.sage_debug_staging_codes(P(FAKE), P(FAKE), 1, 64, 2, 64, *[P(FAKE)] * 4, None)
    assert st == UNSUPPORTED
    st = lib.sage_debug_staging_codes(P(FAKE), P(FAKE), 1, 64, 2, 128, P(FAKE), P(FAKE), P(FAKE + 8),
                                      P(FAKE), None)
    assert st == MISALIGNED
    assert b"k16" in lib.sage_last_error()


def test_plan_checks_its_arguments_on_the_host(lib):
    """sage_plan_create rejects what sage_attn_fwd_cross rejects, before any
    CUDA call, and leaves *plan NULL; launch and destroy check for NULL."""
    h = ctypes.c_void_p(FAKE)
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), None)
    assert lib.sage_plan_create(*args, 1, 256, 256, 2, 128, 0.1, None) == INVALID
    assert lib.sage_plan_create(*args, 1, 256, 256, 2, 64, 0.1, ctypes.byref(h)) == UNSUPPORTED
    assert h.value is None
    h = ctypes.c_void_p(FAKE)
    assert lib.sage_plan_create(*args, 1, 256, 0, 2, 128, 0.1, ctypes.byref(h)) == INVALID
    assert h.value is None
    assert lib.sage_plan_create(*args, 1, 256, 256, 2, 128, float("nan"), ctypes.byref(h)) == INVALID
    assert lib.sage_plan_create(P(FAKE), P(FAKE), P(FAKE + 8), P(FAKE), None, 1, 256, 256, 2, 128, 0.1,
                                ctypes.byref(h)) == MISALIGNED
    assert b"v" in lib.sage_last_error()
    assert lib.sage_plan_create(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE + 4), 1, 256, 256, 2, 128, 0.1,
                                ctypes.byref(h)) == MISALIGNED
    assert b"lse" in lib.sage_last_error()
    assert lib.sage_plan_launch(None, None) == INVALID
    assert lib.sage_plan_destroy(None) == OK


def test_plan_options_are_checked_on_the_host(lib):
    """sage_plan_create_ex records the K-smoothing or fused-Q call: unknown
    bits and both options at once are UNSUPPORTED, either option with
    Sq != Skv or an lse buffer is INVALID_ARG, all before any CUDA call and
    with *plan left NULL."""
    args = (P(FAKE), P(FAKE), P(FAKE), P(FAKE), None)
    for flags, want in ((4, UNSUPPORTED), (qad.PLAN_SMOOTH_K | qad.PLAN_FUSED_Q, UNSUPPORTED)):
        h = ctypes.c_void_p(FAKE)
        assert lib.sage_plan_create_ex(*args, 1, 256, 256, 2, 128, 0.1, flags, ctypes.byref(h)) == want
        assert h.value is None
    for flags in (qad.PLAN_SMOOTH_K, qad.PLAN_FUSED_Q):
        h = ctypes.c_void_p(FAKE)
        assert lib.sage_plan_create_ex(*args, 1, 256, 300, 2, 128, 0.1, flags, ctypes.byref(h)) == INVALID
        assert b"self-attention" in lib.sage_last_error()
        assert h.value is None
        assert lib.sage_plan_create_ex(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 256, 256, 2, 128, 0.1, flags,
                                       ctypes.byref(h)) == INVALID
        assert lib.sage_plan_create_ex(*args, 1, 256, 256, 2, 64, 0.1, flags, ctypes.byref(h)) == UNSUPPORTED
    assert lib.sage_plan_create_ex(*args, 1, 256, 256, 2, 128, 0.1, 0, None) == INVALID
