"""Helpers shared by the GPU parity tests (no test functions here)."""
import math

import numpy as np
import torch

import oracle
from quantized_attention_diffusion_gb300 import build as qbuild
from quantized_attention_diffusion_gb300.workloads import bf16_bits, make_qkv

# Output tolerance against the oracle: 2e-2 absolute, but never less than one
# BF16 ulp of the expected value (the kernel and the oracle agree to ~1e-5
# relative before the final BF16 rounding, so they may round to neighbouring
# BF16 values), plus the row's tie bound from the oracle (P codes on an E4M3
# rounding midpoint may round either way).  Accuracy bar against float64
# unquantized attention: cosine >= 0.999 (the 0.9993 the pages report
# against SDPA, rounded down to three digits).
OUT_ATOL = 2e-2
COS_BAR = 0.999


def ensure_library():
    qbuild.build()
    import quantized_attention_diffusion_gb300 as qad
    return qad.load_library()


def to_dev(bits: np.ndarray, dtype=torch.bfloat16):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(dtype)
    return t.cuda()


def f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_out_to_f32(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def gen(B, S, H, recipe="normal", seed=0):
    """(cpu bf16 tensors, bf16 bit arrays) for one synthetic workload."""
    q, k, v = make_qkv(B, S, H, recipe=recipe, seed=seed)
    return (q, k, v), [bf16_bits(t) for t in (q, k, v)]


def quant_to_dev(quant):
    qc, qs, kc, ks, vt, vs = quant
    return (torch.from_numpy(qc).cuda(), torch.from_numpy(qs).cuda(), torch.from_numpy(kc).cuda(),
            torch.from_numpy(ks).cuda(), torch.from_numpy(vt).cuda(), torch.from_numpy(vs).cuda())


def default_scale(D=128):
    return 1.0 / math.sqrt(D)


def bf16_ulp(x):
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def oracle_tolerance(ref, ties):
    """Per-element bound |gpu - oracle| may reach (see OUT_ATOL)."""
    return np.maximum(OUT_ATOL, bf16_ulp(ref)) + np.asarray(ties)[..., None]


def assert_close_to_oracle(got, ref, ties, what=""):
    tol = oracle_tolerance(ref, ties)
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} outputs beyond tolerance; worst at {i}: "
                             f"gpu {got[i]} oracle {ref[i]} tol {tol[i]:.4g}")
    return float(err.max()), int((np.asarray(ties) > 0).sum())


def lse_tolerance(S, lse_ref, lse_ties):
    """Per-row bound on |lse_gpu - lse_oracle| (same codes and running max on
    both sides; see the derivation in the design notes): the kernel's fp32
    row sum L is accumulated by the tensor cores over S/32 E4M3 MMA steps and
    rescaled at most S/96 times, each a relative rounding of at most 2^-24;
    the final fp32 expression (m + log2f(L) - log2 448) * ln 2 adds a few
    roundings of a value below |m| + 32 (|m| <= |lse|/ln 2 + log2 S); plus
    the oracle's LSE tie bound."""
    eps = 2.0 ** -24
    steps = S / 32 + S / 96 + 4
    mag = np.abs(np.asarray(lse_ref)) / math.log(2) + math.log2(max(S, 1)) + 32
    return steps * eps + 8 * eps * mag + np.asarray(lse_ties)


def assert_within_two_pass_bound(got, quant, S, scale, rows, ties, what="", Skv=None):
    """The kernel's output against the oracle's two-pass form (one tile of
    all keys: no dependence on the kernel's 96-key tiling), within the
    derived bound of reading R16 plus what separates the kernel from the
    tiled oracle:

      |gpu - two_pass| <= spread_d * G       (tiled vs two-pass, R16)
                          + ties             (P codes on an E4M3 midpoint, R12)
                          + 2 BF16 ulps      (the two outputs' final roundings)
                          + (Skv/32 + Skv/96 + 8) 2^-24 max_j |v_jd|
                                             (the kernel's fp32 accumulation:
                                              Skv/32 MMA steps, Skv/96 rescales)

    S: query rows; Skv: keys and values (default S).  got: float [n, D] for
    the rows (b, h, i).  Returns (max |gpu - two_pass|, the largest fraction
    of the tolerance used)."""
    Skv = S if Skv is None else int(Skv)
    rows = np.asarray(rows, dtype=np.int32).reshape(-1, 3)
    two_pass = f32(oracle.attend_rows(quant, S, scale, rows, kv_tile=oracle.TWO_PASS,
                                      Skv=Skv)).astype(np.float64)
    G = oracle.requant_bound(quant, S, scale, rows, kv_tile=oracle.KV_TILE, Skv=Skv)
    spread = oracle.v_spread(quant, Skv)[rows[:, 0], rows[:, 1]]
    vt, vs = quant[4], quant[5]
    vmaxabs = (np.abs(oracle.e4m3_decode(vt[..., :Skv])).max(axis=-1) * vs.astype(np.float64))
    noise = (Skv / 32 + Skv / 96 + 8) * 2.0 ** -24 * vmaxabs[rows[:, 0], rows[:, 1]]
    got = np.asarray(got, dtype=np.float64)
    tol = (spread * G[:, None] + np.asarray(ties)[:, None] + noise
           + 2 * bf16_ulp(np.maximum(np.abs(got), np.abs(two_pass))))
    err = np.abs(got - two_pass)
    bad = err > tol
    if bad.any():
        i = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} outputs beyond the two-pass bound; worst at {i}: "
                             f"gpu {got[i]} two-pass {two_pass[i]} tol {tol[i]:.4g} (G {G[i[0]]:.3g})")
    return float(err.max()), float((err / tol).max())
