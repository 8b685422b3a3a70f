"""sage_plan on the GPU: one attention call recorded as a CUDA graph and
replayed.

The plan runs the same kernels as sage_attn_fwd / sage_attn_fwd_cross (the
method of issue #15014's kernel contract: Q/K per-32-row-block INT8, V
per-channel FP8, attend), so its output is checked against the oracle
directly and, bit for bit, against the direct call.  A replay reads the
inputs as they are at that point of the stream, allocates nothing from the
library's pool, and failures injected on the host during creation leave the
library usable.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv
from tests.gpu_common import (assert_close_to_oracle, assert_within_two_pass_bound, default_scale, ensure_library,
                              f32, lse_tolerance)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return ensure_library()


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _check_oracle(out, lse, host_qkv, Sq, Skv, scale, what):
    B, _, H, _ = host_qkv[0].shape
    bits = [bf16_bits(t) for t in host_qkv]
    quant = oracle.quantize(*bits)
    rows = oracle.all_rows(B, Sq, H)
    ref_bits, ties, lse_ref, lse_tie = oracle.attend_rows(quant, Sq, scale, rows, return_ties=True,
                                                          return_lse=True, Skv=Skv)
    o = out.float().cpu().numpy()
    got = o[rows[:, 0], rows[:, 2], rows[:, 1]]
    assert_close_to_oracle(got, f32(ref_bits), ties, what)
    assert_within_two_pass_bound(got, quant, Sq, scale, rows, ties, what + " vs two-pass", Skv=Skv)
    if lse is not None:
        l = lse.cpu().numpy()
        lse_got = l[rows[:, 0], rows[:, 1], rows[:, 2]].astype(np.float64)
        tol = lse_tolerance(Skv, lse_ref, lse_tie)
        assert (np.abs(lse_got - lse_ref) <= tol).all(), f"{what}: lse"


@pytest.mark.parametrize("B,Sq,Skv,H,recipe,seed,with_lse", [
    (1, 200, 200, 2, "normal", 300, False),
    (2, 333, 333, 3, "qk_outlier_channels", 301, True),
    (1, 129, 70, 2, "k_channel_offset", 302, True),
    (2, 64, 385, 1, "normal", 303, False),
])
def test_plan_matches_oracle_and_direct_call(B, Sq, Skv, H, recipe, seed, with_lse):
    import quantized_attention_diffusion_gb300 as qad
    host = make_qkv(B, Sq, H, recipe=recipe, seed=seed, Skv=Skv)
    q, k, v = [t.cuda() for t in host]
    scale = default_scale()
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda") if with_lse else None
    with qad.Plan(q, k, v, scale, lse=lse) as plan:
        for _ in range(3):                      # replays give the same bytes
            out = plan.launch()
        torch.cuda.synchronize()
        assert qad.sync_status() == 0
        _check_oracle(out, lse, host, Sq, Skv, scale, f"plan B{B} Sq{Sq} Skv{Skv}")
        d_out, d_lse = qad.attn_fwd_cross(q, k, v, scale, return_lse=True)
        torch.cuda.synchronize()
        assert _same_bits(out, d_out)
        if with_lse:
            assert torch.equal(lse, d_lse)


def test_plan_reads_the_inputs_at_launch_time():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(1, 300, 2, seed=310)]
    q2, k2, v2 = [t.cuda() for t in make_qkv(1, 300, 2, recipe="k_channel_offset", seed=311)]
    plan = qad.Plan(q, k, v)
    first = plan.launch().clone()
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)                                 # same stream: ordered before the next replay
    second = plan.launch().clone()
    plan.close()
    torch.cuda.synchronize()
    assert _same_bits(second, qad.attn_fwd(q2, k2, v2))
    assert not _same_bits(first, second)


def test_plan_replays_allocate_nothing_from_the_pool():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(2, 700, 2, seed=312)]
    qad.attn_fwd(q, k, v)                       # the pool exists from here on
    torch.cuda.synchronize()
    with qad.Plan(q, k, v) as plan:
        _, used0 = qad.debug_pool_state()
        for _ in range(5):
            plan.launch()
        _, used1 = qad.debug_pool_state()
        torch.cuda.synchronize()
        _, used2 = qad.debug_pool_state()
    assert used0 == used1 == used2


def test_plan_creation_failures_leave_the_library_usable():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(1, 256, 2, seed=313)]
    ref = qad.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    qad.debug_inject_fault(qad.FAULT_POOL_ALLOC)             # the plan's workspace allocation
    with pytest.raises(qad.SageError) as ei:
        qad.Plan(q, k, v)
    assert ei.value.status == 5                              # SAGE_ERR_NO_MEMORY
    qad.debug_inject_fault(qad.FAULT_QUANT_LAUNCH)           # a launch inside the capture
    with pytest.raises(qad.SageError) as ei:
        qad.Plan(q, k, v)
    assert ei.value.status == 4                              # SAGE_ERR_CUDA
    with qad.Plan(q, k, v) as plan:                          # the capture was ended cleanly
        out = plan.launch()
        torch.cuda.synchronize()
        assert _same_bits(out, ref)
    assert _same_bits(qad.attn_fwd(q, k, v), ref)
    torch.cuda.synchronize()
    assert qad.sync_status() == 0


def test_plan_on_a_side_stream_and_after_close():
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(1, 500, 3, seed=314)]
    ref = qad.attn_fwd(q, k, v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    plan = qad.Plan(q, k, v)
    with torch.cuda.stream(s):
        out = plan.launch()
    s.synchronize()
    assert _same_bits(out, ref)
    plan.close()
    with pytest.raises(RuntimeError):
        plan.launch()


@pytest.mark.parametrize("option", ["smooth_k", "fused_q"])
@pytest.mark.parametrize("B,S,H,recipe,seed", [(1, 300, 2, "k_channel_offset", 320),
                                               (2, 129, 3, "qk_outlier_channels", 321)])
def test_plan_variants_replay_their_direct_calls(option, B, S, H, recipe, seed):
    """A plan made with smooth_k (fused_q) replays sage_attn_fwd_smooth_k
    (sage_attn_fwd_fused_q) bit for bit; the smooth-K and fused-Q tests pin
    those calls to the oracle.  On a K-offset input smoothing changes the
    output, so the option is seen to take effect."""
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(B, S, H, recipe=recipe, seed=seed)]
    ref = qad.attn_fwd(q, k, v, **{option: True})
    plain = qad.attn_fwd(q, k, v)
    with qad.Plan(q, k, v, **{option: True}) as plan:
        for _ in range(2):
            out = plan.launch()
        torch.cuda.synchronize()
        assert qad.sync_status() == 0
        assert _same_bits(out, ref)
    if option == "smooth_k" and recipe == "k_channel_offset":
        assert not _same_bits(ref, plain)


def test_out_must_be_32_byte_aligned():
    """The attention kernel writes output rows as 32-byte vectors: an `out`
    that is only 16-byte aligned is rejected on the host, before any launch,
    by the direct call and by plan creation alike."""
    import quantized_attention_diffusion_gb300 as qad
    q, k, v = [t.cuda() for t in make_qkv(1, 64, 2, seed=315)]
    n = q.numel()
    buf = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")      # 8 bf16 = 16 bytes
    out16 = buf[8:].view(q.shape)
    assert out16.data_ptr() % 32 == 16
    with pytest.raises(qad.SageError) as ei:
        qad.attn_fwd(q, k, v, out=out16)
    assert ei.value.status == 3 and "32-byte" in str(ei.value)
    with pytest.raises(qad.SageError) as ei:
        qad.Plan(q, k, v, out=out16)
    assert ei.value.status == 3
    torch.cuda.synchronize()
    assert bool((buf == 0).all())                                         # nothing was written


_FIRST_CALLS_ARE_PLANS = r"""
import json, sys
import torch
sys.path.insert(0, sys.argv[1])
import quantized_attention_diffusion_gb300 as qad
from quantized_attention_diffusion_gb300.workloads import make_qkv
q, k, v = [t.cuda() for t in make_qkv(1, 300, 2, recipe="k_channel_offset", seed=330)]
outs = {}
for name, opts in (("smooth_k", {"smooth_k": True}), ("fused_q", {"fused_q": True}), ("plain", {})):
    with qad.Plan(q, k, v, **opts) as plan:               # before any direct call of the library
        outs[name] = plan.launch().clone()
torch.cuda.synchronize()
status = qad.sync_status()
same = {name: torch.equal(outs[name].view(torch.int16), qad.attn_fwd(q, k, v, **opts).view(torch.int16))
        for name, opts in (("smooth_k", {"smooth_k": True}), ("fused_q", {"fused_q": True}), ("plain", {}))}
torch.cuda.synchronize()
print(json.dumps({"status": status, "same": same}))
"""


def test_plans_recorded_before_any_direct_call():
    """In a fresh process with lazy module loading, plans are the library's
    first calls: creation loads every kernel it records before the capture,
    and each plan's replay equals the direct call made afterwards."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    res = subprocess.run([sys.executable, "-c", _FIRST_CALLS_ARE_PLANS, root], capture_output=True, text=True,
                         timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    rec = json.loads(res.stdout.strip().splitlines()[-1])
    assert rec["status"] == 0 and all(rec["same"].values()), rec
