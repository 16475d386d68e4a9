"""CPU checks of how the tensor-core consumer stages a 32-token value block in
shared memory (no GPU, no attention arithmetic).

The page's value layout [D][BS] gives each dim a row of BS tokens; at 32
tokens a row is 64 bytes, so an ldmatrix row group of 8 consecutive dims falls
in 2 of the 8 sixteen-byte bank groups (a 4-way conflict).  The kernel copies
the block in kVPieces pieces of D / kVPieces dims, piece p placed 16 p bytes
past its contiguous place, and builds each fragment matrix from 8 / kVPieces
dims of every piece, rotated by kVRot dims per piece.  These tests restate
that placement rule and check, for every head size the kernel takes, that the
tile rows cover each dim once, that every piece stays inside its stage on
16-byte boundaries, how many ways the fragment loads conflict, and that the
accumulator hand-over stores are spread no worse than with contiguous rows.
The piece count and rotations are read from the CUDA source, so a change there
is checked here.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MMA = os.path.join(ROOT, "decode_attention_paged_pa_gb300", "csrc", "pa_mma.cuh")
HEAD_SIZES = (64, 80, 96, 112, 128, 256)
ESZ = 2  # 16-bit caches


def _source_constants():
    src = open(MMA).read()
    pieces = int(re.search(r"#define PA_V_PIECES32 (\d+)", src).group(1))
    m = re.search(r"kVRot = kVPieces == 4 \? (\d+) : kVPieces == 2 \? (\d+) : 0;", src)
    return pieces, {4: int(m.group(1)), 2: int(m.group(2)), 1: 0}


PIECES, ROT = _source_constants()


def _layout(D, BS, npc):
    """(vdim, vrow): the dim row i of value tile mt holds, and a dim's byte offset."""
    per, r = D // npc, 8 // npc
    piece_bytes = per * BS * ESZ

    def vdim(mt, i):
        if npc == 1:
            return mt * 16 + i
        h, ri = i >> 3, i & 7
        p = ri // r
        return p * per + (mt * 2 * r + h * r + ri % r + ROT[npc] * p) % per

    def vrow(d):
        p = d // per
        return p * (piece_bytes + 16) + (d - p * per) * BS * ESZ

    return vdim, vrow


def _worst(values):
    return max(values.count(v) for v in values)


def _check(D, BS, npc):
    vdim, vrow = _layout(D, BS, npc)
    kbytes = D * BS * ESZ
    dims, worst_load, worst_store = [], 0, 0
    for mt in range(D // 16):
        for h in range(2):
            rows = [vdim(mt, 8 * h + ri) for ri in range(8)]
            dims += rows
            # One fragment matrix: 8 rows of 16 bytes at token chunk c.
            for c in range(BS * ESZ // 16):
                groups = [((vrow(d) + 16 * c) // 16) % 8 for d in rows]
                worst_load = max(worst_load, _worst(groups))
                assert all(vrow(d) + 16 * c + 16 <= kbytes + 16 * (npc - 1) for d in rows)
            # finish(): lane (r, hq) stores float rows hq * D + dim for hq in 0, 2, 4, 6.
            worst_store = max(worst_store, _worst([(hq * D + d) % 32 for d in rows for hq in (0, 2, 4, 6)]))
    assert sorted(dims) == list(range(D)), "tile rows must hold every dim exactly once"
    piece_bytes = kbytes // npc
    assert piece_bytes % 16 == 0 and all((p * (piece_bytes + 16)) % 16 == 0 for p in range(npc))
    return worst_load, worst_store


def test_source_takes_two_pieces_for_32_token_blocks():
    assert PIECES == 2


@pytest.mark.parametrize("D", HEAD_SIZES)
def test_contiguous_32_token_rows_conflict_four_ways(D):
    assert _check(D, 32, 1) == (4, 4)


@pytest.mark.parametrize("npc", [2, 4])
@pytest.mark.parametrize("D", HEAD_SIZES)
def test_pieces_cut_the_load_conflict_and_keep_the_stores_spread(D, npc):
    worst_load, worst_store = _check(D, 32, npc)
    assert worst_load == 4 // npc
    assert worst_store <= 4


def test_a_dropped_rotation_is_caught():
    """Without the per-piece rotation the hand-over stores of head size 128
    pile onto the same banks: the check above must notice."""
    saved = dict(ROT)
    try:
        ROT[4] = 0
        assert _check(128, 32, 4)[1] > 4
    finally:
        ROT.clear()
        ROT.update(saved)
