"""The phase-map scheme of the phased TMA kernel, modelled on the CPU (no GPU):
an operand whose rows are only 4-byte aligned is read as four matrices of the
rows of one residue mod 4, each starting at the 16-byte boundary d_s floats
below its first row and d_s floats wider than the operand, in boxes 4 floats
wider than the tile at x-coordinates that are multiples of 4; shifting every
landed row left by d_s must give exactly the tile, with zeros past the
operand's last row and column, and never use a float outside the operand.
The model follows the kernel's description (box shapes, phase-major shared
rows, the shifted reads of the FMA loop) and checks the invariants the
hardware imposes: 16-byte aligned starts, row pitches that are multiples of 16
bytes, and x-coordinates that are multiples of 4."""

import numpy as np
import pytest

BM, BN, BK = 128, 128, 32


def phase_maps(base, rows, cols, ld):
    """(start, width, height, pitch, d) of each phase, in floats of the flat memory."""
    maps = []
    for s in range(4):
        row = base + s * ld
        d = row % 4
        maps.append((row - d, cols + d, (rows - s + 3) // 4, 4 * ld, d))
    return maps


def box(mem, m, x0, y0, bw, bh):
    start, width, height, pitch, _ = m
    assert start % 4 == 0 and pitch % 4 == 0 and x0 % 4 == 0 and (bw * 4) % 16 == 0
    out = np.zeros((bh, bw))
    for r in range(bh):
        for c in range(bw):
            if x0 + c < width and y0 + r < height:
                out[r, c] = mem[start + (y0 + r) * pitch + x0 + c]
    return out


def landed_tile(mem, maps, r0, c0, tile_rows, tile_cols):
    """Rows r0 .. r0 + tile_rows - 1 (r0 a multiple of 4), columns c0 .. c0 +
    tile_cols - 1, through the phase maps and the shift, in tile order."""
    out = np.zeros((tile_rows, tile_cols))
    for s, m in enumerate(maps):
        b = box(mem, m, c0, r0 // 4, tile_cols + 4, tile_rows // 4)
        shifted = b[:, m[4]:m[4] + tile_cols]             # the in-place shift left by d_s
        out[s::4] = shifted                                 # phase-major rows back to tile rows
    return out


@pytest.mark.parametrize("rows,cols,ld,off", [(130, 37, 39, 1), (9, 140, 141, 2), (64, 33, 33, 3), (4, 5, 7, 0),
                                              (200, 64, 67, 2)])
def test_every_tile_lands_exactly(rows, cols, ld, off):
    rng = np.random.default_rng(rows * 7 + ld)
    mem = np.full(off + rows * ld + 8, np.nan)               # NaN everywhere outside the operand
    M = rng.integers(-9, 10, (rows, cols)).astype(float)
    for r in range(rows):
        mem[off + r * ld: off + r * ld + cols] = M[r]
    maps = phase_maps(off, rows, cols, ld)
    # A-shaped tiles (BM rows x BK columns) and B-shaped tiles (BK rows x BN columns)
    for tr, tc in ((BM, BK), (BK, BN)):
        for r0 in range(0, rows, tr):
            for c0 in range(0, cols, tc):
                got = landed_tile(mem, maps, r0, c0, tr, tc)
                want = np.zeros((tr, tc))
                blk = M[r0:r0 + tr, c0:c0 + tc]
                want[:blk.shape[0], :blk.shape[1]] = blk
                assert not np.isnan(got).any(), "a float outside the operand reached the tile"
                assert np.array_equal(got, want)


def test_shift_offsets_follow_the_row_addresses():
    # lda = 2047 floats from a 16-byte aligned base: phases 1, 2, 3 start 3, 2, 1 floats late
    assert [m[4] for m in phase_maps(0, 3001, 2047, 2047)] == [0, 3, 2, 1]
    assert [m[4] for m in phase_maps(0, 2047, 4999, 4999)] == [0, 3, 2, 1]
    # an aligned operand needs no shift at all
    assert [m[4] for m in phase_maps(0, 100, 64, 64)] == [0, 0, 0, 0]
    # a base one float past a boundary shifts every phase
    assert [m[4] for m in phase_maps(1, 100, 64, 64)] == [1, 1, 1, 1]


def test_epilogue_row_map_is_a_bijection():
    # the thread of lane bits lm, warp row warp_m holds shared rows
    # rho = 64 warp_m + lm + 8 i; shared row rho holds tile row 4 (rho % 32) + rho // 32
    seen = set()
    for warp_m in range(2):
        for lm in range(8):
            base = 64 * warp_m // 32 + 4 * lm
            for i in range(8):
                rho = 64 * warp_m + lm + 8 * i
                row = 4 * (rho % 32) + rho // 32
                assert row == base + 4 * ((8 * i) % 32) + (8 * i) // 32
                seen.add(row)
    assert seen == set(range(BM))
