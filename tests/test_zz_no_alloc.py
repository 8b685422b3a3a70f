"""sage_quantize_qkv_noalloc: quantisation for callers that cannot allocate.

Some callers cannot call cudaMalloc or another allocating routine where they
quantise (a framework that owns all device memory, a real-time loop that
must not take allocation locks, memory reserved up front).  The entry point
uses a fixed scratch array built into the library instead of the pool that
sage_quantize_qkv allocates from.  These tests call it through the C ABI and
check that it returns exactly what sage_quantize_qkv returns and exactly what
the CPU oracle computes (quantisation is bit-exact), on two calls in a row
whose inputs differ in scale, so that the second call cannot see the first
call's leftover channel maxima; and, in a fresh process, that it never
creates the library's memory pool and leaves the device's free memory
unchanged from one call to the next.

This file is collected last on purpose.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from tests.gpu_common import ensure_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _inputs(B, S, H, seed, scale):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn((B, S, H, 128), generator=g) * scale).to(torch.bfloat16).cuda()
            for _ in range(3)]


def _empty_like_quant(B, S, H):
    Sp = (S + 127) // 128 * 128
    nb = (S + 31) // 32
    dev = "cuda"
    return (torch.empty((B, H, Sp, 128), dtype=torch.int8, device=dev),
            torch.empty((B, H, nb), dtype=torch.float32, device=dev),
            torch.empty((B, H, Sp, 128), dtype=torch.int8, device=dev),
            torch.empty((B, H, nb), dtype=torch.float32, device=dev),
            torch.empty((B, H, 128, Sp), dtype=torch.uint8, device=dev),
            torch.empty((B, H, 128), dtype=torch.float32, device=dev))


def _call_noalloc(lib, q, k, v, out):
    B, S, H, D = q.shape
    P = ctypes.c_void_p
    st = P(torch.cuda.current_stream().cuda_stream)
    status = lib.sage_quantize_qkv_noalloc(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), B, S, H, D,
                                           *[P(t.data_ptr()) for t in out], st)
    assert status == 0, lib.sage_last_error()


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def test_noalloc_matches_pooled_quantisation_on_consecutive_calls(lib):
    import quantized_attention_diffusion_gb300 as qad
    for seed, scale, (B, S, H) in [(31, 6.0, (2, 300, 3)), (32, 0.25, (2, 300, 3))]:
        q, k, v = _inputs(B, S, H, seed, scale)
        ref = qad.quantize_qkv(q, k, v)
        got = _empty_like_quant(B, S, H)
        for t in got:                                     # poison: every element must be written
            t.fill_(1e30 if t.dtype == torch.float32 else 0x7F)
        _call_noalloc(lib, q, k, v, got)
        torch.cuda.synchronize()
        for name, g_t, r_t in zip(("q_i8", "q_scale", "k_i8", "k_scale", "vt_fp8", "v_scale"), got, ref):
            g_np, r_np = g_t.cpu().numpy(), r_t.cpu().numpy()
            assert np.array_equal(g_np.view(np.uint8), r_np.view(np.uint8)), name


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)
    status = lib.sage_quantize_qkv_noalloc(fake, fake, fake, 2, 64, 4097, 128, *[fake] * 6, None)
    assert status == 1                                    # SAGE_ERR_INVALID_ARG
    assert b"8192" in lib.sage_last_error()


def test_noalloc_matches_the_oracle_on_consecutive_calls(lib):
    import oracle
    from quantized_attention_diffusion_gb300.workloads import bf16_bits
    for seed, scale, (B, S, H) in [(33, 4.0, (1, 333, 2)), (34, 0.5, (1, 333, 2))]:
        q, k, v = _inputs(B, S, H, seed, scale)
        got = _empty_like_quant(B, S, H)
        for t in got:
            t.fill_(1e30 if t.dtype == torch.float32 else 0x7F)
        _call_noalloc(lib, q, k, v, got)
        torch.cuda.synchronize()
        ref = oracle.quantize(*[bf16_bits(t.cpu()) for t in (q, k, v)])
        for name, g_t, r in zip(("q_i8", "q_scale", "k_i8", "k_scale", "vt_fp8", "v_scale"), got, ref):
            assert np.array_equal(g_t.cpu().numpy().view(np.uint8), r.view(np.uint8)), name


_FRESH_PROCESS = r"""
import ctypes, json, sys
import torch
sys.path.insert(0, sys.argv[1])
import quantized_attention_diffusion_gb300 as qad
lib = qad.load_library()
B, S, H = 2, 300, 3
g = torch.Generator().manual_seed(5)
q, k, v = [torch.randn((B, S, H, 128), generator=g).to(torch.bfloat16).cuda() for _ in range(3)]
Sp, nb = (S + 127) // 128 * 128, (S + 31) // 32
outs = [torch.empty((B, H, Sp, 128), dtype=torch.int8, device="cuda"),
        torch.empty((B, H, nb), dtype=torch.float32, device="cuda"),
        torch.empty((B, H, Sp, 128), dtype=torch.int8, device="cuda"),
        torch.empty((B, H, nb), dtype=torch.float32, device="cuda"),
        torch.empty((B, H, 128, Sp), dtype=torch.uint8, device="cuda"),
        torch.empty((B, H, 128), dtype=torch.float32, device="cuda")]
P = ctypes.c_void_p
st = P(torch.cuda.current_stream().cuda_stream)
def call():
    rc = lib.sage_quantize_qkv_noalloc(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), B, S, H, 128,
                                       *[P(t.data_ptr()) for t in outs], st)
    assert rc == 0, lib.sage_last_error()
call()                          # first call: loads the kernels, looks up the array's address
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
call(); call()
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
created, used = qad.debug_pool_state()
print(json.dumps({"free0": free0, "free1": free1, "pool_created": created, "pool_used": used}))
"""


def test_noalloc_allocates_nothing_in_a_fresh_process(lib):
    """Only sage_quantize_qkv_noalloc runs in the child: the library's pool is
    never created and the device's free memory does not move between calls
    (the first call may load the library's kernels, which the driver does
    once per process)."""
    res = subprocess.run([sys.executable, "-c", _FRESH_PROCESS, ROOT], capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    rec = json.loads(res.stdout.strip().splitlines()[-1])
    assert rec["pool_created"] is False and rec["pool_used"] == 0, rec
    assert rec["free1"] == rec["free0"], rec
