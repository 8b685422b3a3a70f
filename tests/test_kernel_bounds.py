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


GRID_Y_MAX = 65535


def heads_grid_blocks(x_blocks, heads):
    """(bh, x) of every live block of a grid from heads_grid(x_blocks,
    heads): dim3(x, min(heads, 65535), ceil(heads / 65535)), head index
    z * 65535 + y, blocks with bh >= heads returning at once."""
    gy, gz = min(heads, GRID_Y_MAX), (heads + GRID_Y_MAX - 1) // GRID_Y_MAX
    assert gy <= 65535 and gz <= 65535
    out = []
    for z in range(gz):
        for y in range(gy):
            bh = z * GRID_Y_MAX + y
            if bh < heads:
                out.extend((bh, x) for x in range(x_blocks))
    return out


def test_heads_grid_covers_every_head_once():
    for heads in (1, 2, 65534, 65535, 65536, 65600, 131071, 200000):
        gy, gz = min(heads, GRID_Y_MAX), (heads + GRID_Y_MAX - 1) // GRID_Y_MAX
        bhs = np.add.outer(np.arange(gz) * GRID_Y_MAX, np.arange(gy)).ravel()
        live = bhs[bhs < heads]
        assert np.array_equal(np.sort(live), np.arange(heads)), heads
    # the largest B*H the ABI takes still fits the y and z limits
    assert (2 ** 31 - 1 + GRID_Y_MAX - 1) // GRID_Y_MAX <= 65535


def v_encode_accesses(B, S, H):
    """v_encode_kernel: grid (S_pad / 128, heads) as heads_grid forms it,
    block (x, y, z) for tile x of head bh = z * 65535 + y, 256 threads.  Follows every
    byte: load instruction i (0..7) of lane l in warp w reads token
    128 x + 8 tg + i (tg = 2w + l/16; only tokens < S) at channels
    8g .. 8g+7 (g = l % 16, 16 bytes); the register transposes give channel
    8g + c the tokens 8 tg .. 8 tg + 7, stored as 8 bytes at
    tile[(8g + c) * 128 + 8 (tg ^ (g & 14))]; thread t then reads, for
    it = 0..3, channel row c = 32 it + t/8, 16 bytes at 16 (m ^ (gc / 2))
    (m = t % 8, gc = (c / 8) % 16) and writes them to V^T row (bh, c) at
    tokens 128 x + 16 m .. +15.  A lane with an out-of-range channel scale
    rewrites byte i of its chunk in row 8g + c (c = 0..7, i = 0..7): those
    are bytes the same lane stored.  Checks
    bounds, alignment, that every tile byte is written once and every V^T
    byte once, that V^T gets the transpose of the tokens' codes, and that
    each tile store instruction takes two bank wavefronts."""
    Sp, BH = padded(S), B * H
    assert Sp % 128 == 0
    ntiles = Sp // 128
    written = np.full(BH * D * Sp, -1, dtype=np.int64)        # V^T byte -> (token * D + channel)
    blocks = heads_grid_blocks(ntiles, BH)
    for bh, x in blocks:
        b, h = bh // H, bh % H
        tile = np.full(D * 128, -1, dtype=np.int64)
        for t in range(256):
            lane, warp = t & 31, t >> 5
            g, tg = lane & 15, 2 * warp + (lane >> 4)
            for i in range(8):
                s = 128 * x + 8 * tg + i
                if s < S:
                    elem = ((b * S + s) * H + h) * D + 8 * g
                    assert elem % 8 == 0 and 0 <= elem and elem + 8 <= B * S * H * D
            mine = set()
            for c in range(8):
                addr = (8 * g + c) * 128 + ((tg ^ (g & 14)) << 3)
                assert addr % 8 == 0 and 0 <= addr and addr + 8 <= D * 128
                for j in range(8):
                    assert tile[addr + j] == -1, "tile byte written twice"
                    tile[addr + j] = (128 * x + 8 * tg + j) * D + 8 * g + c
                    mine.add(addr + j)
            chunk = 8 * g * 128 + ((tg ^ (g & 14)) << 3)
            for c in range(8):
                for i in range(8):
                    assert chunk + c * 128 + i in mine          # division rewrite of its own byte
                    assert tile[chunk + c * 128 + i] == (128 * x + 8 * tg + i) * D + 8 * g + c
        assert np.all(tile >= 0)
        for t in range(256):
            m = t & 7
            for it in range(4):
                c = it * 32 + (t >> 3)
                gc = (c >> 3) & 15
                a = c * 128 + ((m ^ (gc >> 1)) << 4)
                assert a % 16 == 0 and a + 16 <= D * 128
                piece = tile[a:a + 16]
                dst = (bh * D + c) * Sp + 128 * x + 16 * m
                assert dst % 16 == 0 and dst + 16 <= BH * D * Sp
                assert np.all(written[dst:dst + 16] == -1), "V^T byte written twice"
                written[dst:dst + 16] = piece
    tok = np.arange(Sp)[None, :]
    ch = np.arange(D)[:, None]
    expect = np.broadcast_to(tok * D + ch, (D, Sp))
    assert np.array_equal(written.reshape(BH, D, Sp), np.broadcast_to(expect, (BH, D, Sp)))
    # bank wavefronts of one tile store instruction (fixed c) of warp w: 32 lanes x 8 bytes
    for w in range(8):
        for c in range(8):
            pairs = [(((8 * (l & 15) + c) * 128 + (((2 * w + (l >> 4)) ^ (l & 14)) << 3)) // 8) % 16
                     for l in range(32)]
            assert max(np.bincount(pairs, minlength=16)) == 2


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
                                   (1, 129, 3), (2, 300, 3), (1, 400, 1)])
def test_quantisation_kernels_stay_in_bounds(B, S, H):
    v_encode_accesses(B, S, H)
    pass1_accesses(B, S, H)
