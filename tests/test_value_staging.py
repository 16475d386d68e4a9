"""CPU checks of how the tensor-core consumer addresses a staged value block
(no GPU, no attention arithmetic).

A value block is the page's value layout [D][BS] for one kv head: rows of
R = 2 BS bytes (16-bit elements), copied into shared memory by a tensor copy
in the R-byte swizzle (32, 64 or 128 bytes for blocks of 16, 32 or 64
tokens), which XORs the 16-byte chunk index of an address (bits 4..) with
its bits 7.. (one, two or three of them).  The consumer's ``vchunk(d, c)``
gives the byte offset of the 16-byte chunk c (tokens 8c .. 8c + 7) of dim d.
These tests read that expression from the CUDA source and check, for every
head size and block size the kernel takes, that it is the swizzle rule
applied to the unswizzled offset, that it maps the block's (dim, chunk)
pairs one to one onto its 16-byte slots, and that every ldmatrix row group
(8 consecutive dims, one chunk) falls in 8 distinct bank groups, i.e. is
free of bank conflicts -- which the unswizzled rows are not.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MMA = os.path.join(ROOT, "decode_attention_paged_pa_gb300", "csrc", "pa_mma.cuh")
HEAD_SIZES = (64, 80, 96, 112, 128, 256)
BLOCK_SIZES = (16, 32, 64)
CASES = [(D, BS) for D in HEAD_SIZES for BS in BLOCK_SIZES]


def _vchunk_from_source():
    src = open(MMA).read()
    body = src[src.index("static uint32_t vchunk(int d, int c)"):]
    expr = re.search(r"if constexpr \(kTma\) \{\s*return (.*?);", body, re.S).group(1)
    py = re.sub(r"\(uint32_t\)", "", expr)
    py = re.sub(r"(\d+)u\b", r"\1", py)
    py = py.replace("/", "//")
    return eval("lambda d, c, VROW: " + py)  # noqa: S307 - an arithmetic expression of the kernel source


VCHUNK = _vchunk_from_source()


def swizzle(addr: int, row_bytes: int) -> int:
    """The tensor copy's swizzle of `row_bytes` (32, 64, 128) bytes: the
    16-byte chunk index XOR address bits 7.. (1, 2 or 3 of them)."""
    mask = row_bytes // 16 - 1
    return addr ^ (((addr >> 7) & mask) << 4)


@pytest.mark.parametrize("D,BS", CASES)
def test_vchunk_is_the_row_width_swizzle(D, BS):
    R = 2 * BS
    for d in range(D):
        for c in range(BS // 8):
            assert VCHUNK(d, c, R) == swizzle(d * R + c * 16, R), (d, c)


@pytest.mark.parametrize("D,BS", CASES)
def test_vchunk_is_one_to_one_inside_the_block(D, BS):
    R = 2 * BS
    slots = sorted(VCHUNK(d, c, R) for d in range(D) for c in range(BS // 8))
    assert slots == list(range(0, D * R, 16))


@pytest.mark.parametrize("D,BS", CASES)
def test_ldmatrix_row_groups_are_conflict_free(D, BS):
    # ldmatrix .x4 reads four 8x8 matrices; each is 8 rows of 16 bytes from 8
    # lanes: dims mt*16 + 8*h + (0..7), one chunk.  32 banks of 4 bytes = 8
    # groups of 16 bytes; 8 distinct groups means one wavefront.
    R = 2 * BS
    for mt in range(D // 16):
        for h in range(2):
            for c in range(BS // 8):
                groups = [(VCHUNK(mt * 16 + 8 * h + i, c, R) // 16) % 8 for i in range(8)]
                assert len(set(groups)) == 8, (mt, h, c, groups)


@pytest.mark.parametrize("BS", BLOCK_SIZES)
def test_unswizzled_rows_would_conflict(BS):
    # Without the swizzle, 8 rows R bytes apart fill only 8 R / 128 bank groups.
    R = 2 * BS
    groups = [((d * R) // 16) % 8 for d in range(8)]
    assert len(set(groups)) == max(1, 8 * 16 // R) and len(set(groups)) < 8


def test_row_consumer_uses_the_same_value_addressing():
    """The 16-row consumer (pa_mma_rows.cuh) addresses a staged value block by
    the same expression, so every check above holds for it too."""
    rows = open(os.path.join(ROOT, "decode_attention_paged_pa_gb300", "csrc", "pa_mma_rows.cuh")).read()
    body = rows[rows.index("static uint32_t vchunk(int d, int c)"):]
    expr = re.search(r"\{\s*return (.*?);", body, re.S).group(1)
    src = open(MMA).read()
    mma_body = src[src.index("static uint32_t vchunk(int d, int c)"):]
    mma_expr = re.search(r"if constexpr \(kTma\) \{\s*return (.*?);", mma_body, re.S).group(1)
    assert " ".join(expr.split()) == " ".join(mma_expr.split())
