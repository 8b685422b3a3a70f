"""Seeded synthetic Q/K/V generators.

This module draws the BF16 inputs that both the CUDA path and the CPU oracle
consume.  It holds none of the attention method's arithmetic: it only samples
normal variates and shapes them like the pages' diffusion and video
workloads (Q/K/V ``[B, S, H, 128]``, BF16; K and V may have their own
length Skv for cross-attention).

Recipes (each input is drawn fp32 from one ``torch.Generator`` seeded per
workload, in the order Q, K, V, then the recipe's extra draws, and rounded to
BF16 with round-to-nearest-even by ``Tensor.to(torch.bfloat16)``):

* ``normal``            -- Q, K, V ~ N(0, 1).
* ``k_channel_offset``  -- as ``normal``, then K += offset[h, d] with offset ~
  N(0, std 2), one value per (head, channel) shared by every token and batch:
  the channel outliers in K that InvokeAI PR #9657 ("Summary", K smoothing
  notes) reports for real diffusion heads.
* ``qk_outlier_channels`` -- as ``normal``, then ceil(1% of D) = 2 channel
  indices (a seeded choice, shared by all heads and by Q and K) are scaled by 8.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    recipe: str
    seed: int
    D: int = HEAD_DIM
    Skv: int | None = None      # keys/values; None: self-attention (Skv = S)

    @property
    def skv(self) -> int:
        return self.S if self.Skv is None else self.Skv

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def ops(self) -> int:
        """Tensor operations of one attention call: 4 * B * H * S * Skv * D."""
        return 4 * self.B * self.H * self.S * self.skv * self.D

    def describe(self) -> str:
        kv = "" if self.Skv is None else f" Skv={self.Skv}"
        return f"B={self.B} S={self.S}{kv} H={self.H} D={self.D} {self.recipe} seed={self.seed}"


# The pages' workloads, by what they are.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("b1_s256_h2", 1, 256, 2, "normal", 0),
        Workload("b1_s4096_h24_koffset", 1, 4096, 24, "k_channel_offset", 1),
        Workload("b2_s16384_h24_outlier", 2, 16384, 24, "qk_outlier_channels", 2),
        Workload("b1_s32760_h40", 1, 32760, 40, "normal", 3),
        Workload("b1_s65536_h24_koffset", 1, 65536, 24, "k_channel_offset", 4),
        # cross-attention: image tokens attending to a short, ragged text context,
        # and a short query block against a long key/value sequence
        Workload("b2_sq16384_skv333_h24_cross", 2, 16384, 24, "normal", 5, Skv=333),
        Workload("b1_sq4096_skv16384_h24_cross", 1, 4096, 24, "k_channel_offset", 6, Skv=16384),
    ]
}


def make_qkv(B: int, S: int, H: int, D: int = HEAD_DIM, recipe: str = "normal",
             seed: int = 0, device: str | torch.device = "cpu", Skv: int | None = None):
    """Return (q, k, v) BF16 tensors on ``device``: q [B, S, H, D], k and v
    [B, Skv, H, D] (Skv defaults to S).

    Values are drawn on the CPU so that a workload has the same bytes on
    every device; the tensors are then copied.
    """
    g = torch.Generator(device="cpu").manual_seed(int(seed))
    Skv = S if Skv is None else int(Skv)

    def draw(n):
        return torch.randn((B, n, H, D), generator=g, dtype=torch.float32)

    q = draw(S)
    k = draw(Skv)
    v = draw(Skv)
    if recipe == "k_channel_offset":
        offset = torch.randn((H, D), generator=g, dtype=torch.float32) * 2.0
        k += offset.view(1, 1, H, D)
    elif recipe == "qk_outlier_channels":
        n = math.ceil(0.01 * D)
        ch = torch.randperm(D, generator=g)[:n]
        q[..., ch] *= 8.0
        k[..., ch] *= 8.0
    elif recipe != "normal":
        raise ValueError(f"unknown recipe {recipe!r}")
    out = []
    for t in (q, k, v):
        out.append(t.to(torch.bfloat16).to(device))
    return tuple(out)


def make_workload(w: Workload, device="cpu"):
    return make_qkv(w.B, w.S, w.H, w.D, w.recipe, w.seed, device, Skv=w.Skv)


def bf16_bits(t: torch.Tensor):
    """A CPU BF16 tensor as a numpy uint16 array of its bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def sample_rows(B: int, S: int, H: int, heads: int = 4, rows_per_head: int = 512,
                seed: int = 0):
    """(b, h, i) query rows for sampled parity at large S.

    Picks ``heads`` (b, h) pairs (first, last and seeded others) and, in each,
    ``rows_per_head`` query rows that always include the first and last 128-row
    tile and the rows of the last (possibly short) 32-row block.
    """
    import numpy as np

    rng = np.random.default_rng(seed)
    bh_all = [(b, h) for b in range(B) for h in range(H)]
    picks = {bh_all[0], bh_all[-1]}
    while len(picks) < min(heads, len(bh_all)):
        picks.add(bh_all[int(rng.integers(len(bh_all)))])
    fixed = set(range(min(S, 128))) | set(range(max(0, S - 128), S))
    fixed |= set(range((S - 1) // 32 * 32, S))
    rows = []
    for b, h in sorted(picks):
        need = max(0, rows_per_head - len(fixed))
        pool = np.setdiff1d(np.arange(S), np.fromiter(fixed, dtype=np.int64))
        extra = rng.choice(pool, size=min(need, pool.size), replace=False) if need else []
        for i in sorted(fixed | set(int(x) for x in extra)):
            rows.append((b, h, i))
    return np.asarray(rows, dtype=np.int32)
