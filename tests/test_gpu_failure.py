"""Failure handling and buffer bounds on the GPU, without a GPU fault.

* Host-side fault injection (sage_debug_inject_fault): a failed workspace
  allocation or a failed launch step reports SAGE_ERR_NO_MEMORY /
  SAGE_ERR_CUDA with a message, releases the workspace, and leaves the CUDA
  context usable -- InvokeAI PR #9657, review "Advisory": a sticky CUDA error
  poisons the context, and out-of-memory must be handled.
* Canary-guarded buffers: every output the entry points write (out, lse, the
  INT8/E4M3 codes and scales, V^T, the caller workspace) sits between margins
  of a known byte pattern, and no margin byte changes, at the tail lengths
  S = 1, 31, 33, 127, 129 and 32760 (the pages' non-multiple-of-tile video
  length).  The inputs are checked unchanged too.
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import default_scale, ensure_library, gen

pytestmark = pytest.mark.gpu

MARGIN = 4096            # bytes on each side of a guarded buffer
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


@pytest.fixture(autouse=True)
def disarm():
    import quantized_attention_diffusion_gb300 as qad
    yield
    qad.debug_inject_fault(qad.FAULT_NONE)


# ------------------------------------------------------- fault injection --

def _qkv(S=300, H=2, seed=40):
    qkv, _ = gen(1, S, H, "normal", seed)
    return [t.cuda() for t in qkv]


def test_injected_pool_failure_reports_no_memory_and_the_next_call_works():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = _qkv()
    ref = qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    qad.debug_inject_fault(qad.FAULT_POOL_ALLOC)
    with pytest.raises(qad.SageError, match="SAGE_ERR_NO_MEMORY.*injected fault"):
        qad.attn_fwd(q, k, v)
    again = qad.attn_fwd(q, k, v)                     # disarmed after one event
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), ref.view(torch.int16))
    assert qad.sync_status() == 0


@pytest.mark.parametrize("site_name", ["FAULT_QUANT_LAUNCH", "FAULT_ATTN_LAUNCH"])
def test_injected_launch_failure_releases_the_workspace(site_name):
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = _qkv()
    ref = qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    created, used_before = qad.debug_pool_state()
    assert created
    qad.debug_inject_fault(getattr(qad, site_name))
    with pytest.raises(qad.SageError, match="SAGE_ERR_CUDA.*injected fault"):
        qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert qad.debug_pool_state() == (True, used_before)   # the workspace went back to the pool
    out = qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert qad.sync_status() == 0


def test_injection_skips_the_requested_number_of_events():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = _qkv()
    qad.debug_inject_fault(qad.FAULT_ATTN_LAUNCH, skip=1)
    qad.attn_fwd(q, k, v)                                   # passes
    with pytest.raises(qad.SageError, match="attention launch: injected fault"):
        qad.attn_fwd(q, k, v)                               # fails
    qad.attn_fwd(q, k, v)                                   # disarmed
    torch.cuda.synchronize()


def test_injected_scratch_failure_in_quantize_qkv():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = _qkv()
    ref = [t.clone() for t in qad.quantize_qkv(q, k, v)]
    qad.debug_inject_fault(qad.FAULT_POOL_ALLOC)
    with pytest.raises(qad.SageError, match="SAGE_ERR_NO_MEMORY.*V maxima scratch"):
        qad.quantize_qkv(q, k, v)
    got = qad.quantize_qkv(q, k, v)
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        assert torch.equal(g.view(torch.uint8), r.view(torch.uint8))


# ------------------------------------------------------------- canaries --

class Guarded:
    """A tensor of `shape`/`dtype` inside a byte buffer with MARGIN bytes of
    PATTERN on each side (16-byte aligned: MARGIN is a multiple of 256)."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((MARGIN + n + MARGIN,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[MARGIN:MARGIN + n].view(dtype).view(shape)
        self.n = n

    def margins_intact(self):
        r = self.raw.cpu().numpy()
        return bool((r[:MARGIN] == PATTERN).all() and (r[MARGIN + self.n:] == PATTERN).all())


TAIL_SHAPES = [(1, 1, 2), (1, 31, 2), (2, 33, 1), (1, 127, 1), (1, 129, 3), (1, 32760, 1)]


@pytest.mark.parametrize("B,S,H", TAIL_SHAPES)
def test_attention_outputs_stay_inside_their_buffers(B, S, H):
    import quantized_attention_diffusion_gb300 as qad
    qkv, _ = gen(B, S, H, "normal", 41 + S)
    q, k, v = [t.cuda() for t in qkv]
    inputs = [t.clone() for t in (q, k, v)]
    out = Guarded((B, S, H, 128), torch.bfloat16)
    qad.attn_fwd(q, k, v, out=out.t)
    out2 = Guarded((B, S, H, 128), torch.bfloat16)
    lse = Guarded((B, H, S), torch.float32)
    qad.attn_fwd_lse(q, k, v, out=out2.t, lse=lse.t)
    ws_bytes = qad.workspace_bytes(B, S, H)
    ws = Guarded((ws_bytes,), torch.uint8)
    out3 = Guarded((B, S, H, 128), torch.bfloat16)
    qad.attn_fwd(q, k, v, out=out3.t, workspace=ws.t)
    torch.cuda.synchronize()
    for name, g in (("out", out), ("out (lse call)", out2), ("lse", lse), ("workspace", ws),
                    ("out (workspace call)", out3)):
        assert g.margins_intact(), name
    assert torch.equal(out.t.view(torch.int16), out2.t.view(torch.int16))
    assert torch.equal(out.t.view(torch.int16), out3.t.view(torch.int16))
    for a, b in zip(inputs, (q, k, v)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert qad.sync_status() == 0


@pytest.mark.parametrize("B,S,H", TAIL_SHAPES)
@pytest.mark.parametrize("noalloc", [False, True])
def test_quantised_codes_stay_inside_their_buffers(B, S, H, noalloc):
    import quantized_attention_diffusion_gb300 as qad
    qkv, _ = gen(B, S, H, "k_channel_offset", 42 + S)
    q, k, v = [t.cuda() for t in qkv]
    Sp, nb = qad.padded_len(S), (S + 31) // 32
    bufs = [Guarded((B, H, Sp, 128), torch.int8), Guarded((B, H, nb), torch.float32),
            Guarded((B, H, Sp, 128), torch.int8), Guarded((B, H, nb), torch.float32),
            Guarded((B, H, 128, Sp), torch.uint8), Guarded((B, H, 128), torch.float32)]
    qad.quantize_qkv(q, k, v, out=tuple(g.t for g in bufs), noalloc=noalloc)
    staged = [Guarded((B, H, Sp, 128), torch.float16), Guarded((B, H, nb), torch.float32),
              Guarded((B, H, Sp, 128), torch.float16), Guarded((B, H, nb), torch.float32)]
    lib = qad.load_library()
    import ctypes
    P = ctypes.c_void_p
    st = P(torch.cuda.current_stream().cuda_stream)
    assert lib.sage_debug_staging_codes(P(q.data_ptr()), P(k.data_ptr()), B, S, H, 128,
                                        *[P(g.t.data_ptr()) for g in staged], st) == 0
    torch.cuda.synchronize()
    names = ["q_i8", "q_scale", "k_i8", "k_scale", "vt_fp8", "v_scale", "q16", "q16 scale", "k16", "k16 scale"]
    for name, g in zip(names, bufs + staged):
        assert g.margins_intact(), name
    # pad rows / columns past S are zero
    assert not bufs[0].t[:, :, S:].any() and not bufs[4].t[..., S:].any()
    assert not staged[0].t[:, :, S:].any()


def test_attention_margins_at_the_default_scale_of_the_video_length():
    """The longest tail shape with the benchmark's H: 32760 tokens x 40 heads
    (the pages' non-multiple-of-tile video length, full size)."""
    import quantized_attention_diffusion_gb300 as qad
    qkv, _ = gen(1, 32760, 40, "normal", 3)
    q, k, v = [t.cuda() for t in qkv]
    out = Guarded((1, 32760, 40, 128), torch.bfloat16)
    qad.attn_fwd(q, k, v, default_scale(), out=out.t)
    torch.cuda.synchronize()
    assert out.margins_intact()
