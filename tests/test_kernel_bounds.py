"""Host-side bounds check of the quantisation kernels' index arithmetic.

For each launch of the two quantisation kernels (the Q/K + V-maxima pass and
the V^T encoder) this enumerates, with numpy, every global element or byte a
thread reads or writes, from the grid, the block size and the index formulas
the kernels state in their comments, and checks each range against the
buffer it belongs to, including the 16- and 8-byte vector alignment.  No GPU
is used: this is the reading-based check the GPU cannot be asked to do by
faulting.  Shapes: the special-values quantisation shape (B=1, S=200, H=2),
the tail lengths and a multi-head case.
"""
import numpy as np
import pytest

D = 128


def padded(S):
    return (S + 127) // 128 * 128


def check_range(lo, hi, size, what):
    """Half-open [lo, hi) element ranges (arrays) inside [0, size)."""
    assert np.all(lo >= 0), what
    assert np.all(hi <= size), (what, int(hi.max()), size)


def v_encode_accesses(B, S, H):
    """v_encode_kernel: grid (S_pad / 128, B*H), 256 threads; warp w, lane l:
    c4 = 16w + 4(l%4), s0 = 128 blockIdx.x + 16(l/4); loads tokens s0..s0+15
    (only those < S) of channels c4..c4+3 (8 bytes); stores 16 bytes per
    channel row c4+c at token s0 of V^T."""
    Sp, BH = padded(S), B * H
    gx, gy = np.meshgrid(np.arange(Sp // 128), np.arange(BH), indexing="ij")
    t = np.arange(256)
    lane, warp = t & 31, t >> 5
    c4 = warp * 16 + (lane & 3) * 4
    bh = gy.ravel()[:, None]
    s0 = gx.ravel()[:, None] * 128 + (lane >> 2)[None, :] * 16
    b, h = bh // H, bh % H
    loads = []
    for i in range(16):
        s = s0 + i
        ok = s < S
        elem = ((b * S + s) * H + h) * D + c4[None, :]
        loads.append(elem[ok])
    loads = np.concatenate(loads)
    assert np.all(loads % 4 == 0)                             # 8-byte aligned uint2 of bf16
    check_range(loads, loads + 4, B * S * H * D, "V loads")
    amax = bh * D + c4[None, :]
    check_range(amax, amax + 4, BH * D, "channel maxima")
    vt = (bh * D + c4[None, :]) * Sp + s0
    for c in range(4):
        off = vt + c * Sp
        assert np.all(off % 16 == 0)
        check_range(off, off + 16, BH * D * Sp, "V^T stores")
    # every byte of V^T is written exactly once
    cover = np.zeros(BH * D * Sp, dtype=np.int32)
    for c in range(4):
        for k in range(16):
            np.add.at(cover, (vt + c * Sp + k).ravel(), 1)
    assert np.all(cover == 1)


def pass1_accesses(B, S, H):
    """qkv_pass1_kernel for self-attention: grid (ctas, 3), 256 threads.
    Roles 0/1 (Q, K): warp gblk = 8 blockIdx.x + w < B*H*S_pad/32, block
    blk = gblk % nbp of head gblk / nbp; lane l owns tokens 32 blk + l/16 +
    2 it (loads only < S) and channels 8(l%16)..+7 (16 bytes); codes rows
    up to 32 blk + 31 < S_pad; the scale only for blk < nb.  Role 2: CTA idx
    < B*H*nslices reads tokens [256 slice, min(S, 256 slice + 256))."""
    Sp, BH, nb = padded(S), B * H, (S + 31) // 32
    nbp, nslices = Sp // 32, (S + 255) // 256
    ctas = max((BH * nbp + 7) // 8, BH * nslices)
    t = np.arange(256)
    lane, warp = t & 31, t >> 5
    gblk = (np.arange(ctas)[:, None] * 8 + warp[None, :]).ravel()
    lane_r = np.tile(lane, ctas)
    live = gblk < BH * nbp
    gblk, lane_r = gblk[live], lane_r[live]
    blk, bh = gblk % nbp, gblk // nbp
    b, h = bh // H, bh % H
    c8 = (lane_r & 15) * 8
    tok0 = blk * 32 + (lane_r >> 4)
    for it in range(16):
        s = tok0 + 2 * it
        ok = s < S
        elem = ((b * S + s) * H + h) * D + c8
        assert np.all(elem % 8 == 0)                           # 16-byte aligned uint4 of bf16
        check_range(elem[ok], elem[ok] + 8, B * S * H * D, "Q/K loads")
        code = (bh * Sp + s) * D + c8
        check_range(code, code + 8, BH * Sp * D, "Q/K code stores")
    sc = (bh * nb + blk)[(lane_r == 0) & (blk < nb)]
    check_range(sc, sc + 1, BH * nb, "Q/K scales")
    idx = np.arange(ctas)
    idx = idx[idx < BH * nslices]
    bh2, s0 = idx // nslices, (idx % nslices) * 256
    for r in range(16):
        for k in range(16):
            s = s0 + r + 16 * k
            ok = s < np.minimum(S, s0 + 256)
            elem = (((bh2 // H) * S + s) * H + bh2 % H) * D
            check_range(elem[ok], elem[ok] + D, B * S * H * D, "V maxima loads")


@pytest.mark.parametrize("B,S,H", [(1, 200, 2), (1, 1, 2), (1, 31, 2), (2, 33, 1), (1, 127, 1),
                                   (1, 129, 3), (2, 300, 3), (1, 1000, 1)])
def test_quantisation_kernels_stay_in_bounds(B, S, H):
    v_encode_accesses(B, S, H)
    pass1_accesses(B, S, H)
