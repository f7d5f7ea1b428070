"""The launch planner, on the CPU: hq_debug_plan runs the library's own
policy choice and make_plan for a described device and returns the geometry a
launch would get, touching no GPU.

Two kinds of checks:
  * pins: the geometry of the bench's launches as ncu recorded them on a GB300
    (grid x block and dynamic shared memory in the committed ncu summaries), for a
    device of 152 SMs with 227 KB (232,448 B) of opt-in shared memory per CTA
    and the kernels' register counts from `ptxas -v` of the sm_103a build;
  * invariants over a sweep of shapes, vector counts and formats: every stage
    has one owner (or, with column-split stages, at least two stages), the ring
    fits the opt-in shared memory, a K split is one wave of whole clusters with
    at least one K chunk per CTA, and every row tile is covered.
"""
import itertools
import math

import pytest

from quantized_weight_matvec_hq_gb300 import build as hq_build

GB300 = dict(num_sms=152, smem_optin=232448)


@pytest.fixture(scope="module")
def hq():
    hq_build.build()
    import quantized_weight_matvec_hq_gb300 as hq
    hq.lib()
    return hq


def plan(hq, fmt, n_vec, rows, cols, regs):
    return hq.hq_debug_plan(fmt, n_vec, rows, cols, GB300["num_sms"], GB300["smem_optin"], regs)


# (fmt, n_vec, rows, cols, regs) -> (grid, threads per CTA, K split, dynamic smem bytes or None),
# as ncu recorded them for the 8B-shaped Q8_0 and Q4_0 tokens, the Qwen3-0.6B-shaped token and the
# full captures of single matrices (the ncu summaries committed beside the benchmark).
PINS = [
    ((8, 1, 28672, 4096, 78), (448, 96, 1, 58880)),      # Q8_0 gate|up: 2 tiles per CTA, 6-stage ring
    ((8, 1, 4096, 14336, 78), (512, 96, 4, None)),       # down: clusters of 4
    ((8, 1, 6144, 4096, 78), (384, 96, 2, None)),        # q|k|v: clusters of 2
    ((8, 1, 4096, 4096, 78), (512, 96, 4, None)),        # o: clusters of 4
    ((8, 1, 128256, 4096, 78), (668, 96, 1, None)),      # lm_head: 6 tiles per CTA
    ((8, 1, 4096, 1024, 78), (256, 160, 2, None)),       # Qwen3-0.6B q|k|v, short rows
    ((8, 1, 1024, 2048, 78), (256, 160, 8, None)),       # Qwen3-0.6B o
    ((8, 1, 6144, 1024, 78), (192, 160, 1, 39648)),      # Qwen3-0.6B gate|up (full capture)
    ((8, 1, 1024, 3072, 78), (256, 160, 8, None)),       # Qwen3-0.6B down
    ((8, 1, 151936, 1024, 78), (297, 160, 1, None)),     # Qwen3-0.6B lm_head
    ((8, 8, 28672, 4096, 104), (448, 160, 1, 59584)),    # Q8_0 n_vec 8, column-split stages (full capture)
    ((4, 1, 28672, 4096, 72), (448, 160, 1, 72976)),     # Q4_0 gate|up, column-split stages (full capture)
    ((75, 1, 28672, 4096, 120), (448, 160, 1, 72976)),   # Q4_K gate|up, column-split stages (full capture)
    ((8, 1, 4096, 4096, 80), (512, 96, 4, 39904)),       # Q8_0 o (full capture)
    ((4, 1, 4096, 14336, 97), (256, 160, 4, None)),
    ((4, 1, 6144, 4096, 97), (384, 160, 4, None)),
    ((4, 1, 4096, 4096, 97), (448, 160, 7, None)),      # Q4_0 o: the K split that fills one wave
    ((4, 1, 128256, 4096, 97), (456, 160, 1, None)),
]


@pytest.mark.parametrize("args,want", PINS)
def test_plan_matches_the_recorded_launches(hq, args, want):
    p = plan(hq, *args)
    grid, threads, ks, smem = want
    assert p["grid"] == grid
    assert 32 * (p["cons_warps"] + 1) == threads
    assert p["ksplit"] == ks
    if smem is not None:
        assert p["smem"] == smem


def expected_policy(fmt, n_vec, rows, cols):
    if fmt == 8 and n_vec == 1:
        return 1 if cols <= 3072 else 0
    if fmt == 8:
        return 4                # n_vec >= 2: column-split stages, two rows per lane
    if fmt in (4, 75) and n_vec >= 4:
        return 4                # column-split stages, two rows per lane
    if fmt in (4, 75) and n_vec <= 2:
        # column-split stages unless K is split over clusters (64-row tiles too
        # few to give each of the 152 x 3 CTA slots two)
        return 4 if math.ceil(rows / 64) * 2 > GB300["num_sms"] * 3 else 0
    return 0


ROWS = [1, 31, 33, 100, 257, 1000, 4096, 6144, 28672, 128256]
COLS = [256, 1024, 2048, 3072, 3328, 4096, 14336]


@pytest.mark.parametrize("fmt", [8, 4, 75, 1])
def test_plan_invariants(hq, fmt):
    chunk = 128 if fmt == 1 else 256
    for rows, cols, n_vec in itertools.product(ROWS, COLS, range(1, 9)):
        regs = 80 if n_vec <= 2 else 128
        p = plan(hq, fmt, n_vec, rows, cols, regs)
        what = f"fmt {fmt} {rows}x{cols} n_vec={n_vec}: {p}"
        n_chunks = cols // chunk
        if fmt in (4, 75) and n_vec == 3:
            # one owner per stage, or eight column-split warps on a K-split launch
            assert p["policy"] == 0 or (p["policy"] == 4 and p["cons_warps"] == 8 and p["ksplit"] > 1), what
        else:
            assert p["policy"] == expected_policy(fmt, n_vec, rows, cols), what
        rpl = 2 if (fmt in (4, 75) and (n_vec != 3 or p["policy"] == 4)) or (fmt == 8 and n_vec >= 2) else 1
        assert p["tile_rows"] == 32 * rpl, what
        assert p["tiles"] == math.ceil(rows / p["tile_rows"]), what
        # the ring: one owner per stage (a multiple of the consumer warps), or at
        # least a double buffer when every warp consumes every stage
        if p["policy"] == 4:
            assert p["stages"] >= 2, what
        else:
            assert p["stages"] >= p["cons_warps"] and p["stages"] % p["cons_warps"] == 0, what
        assert 0 < p["smem"] <= GB300["smem_optin"], what
        assert p["slots"] <= GB300["num_sms"] * p["ctas_per_sm"], what
        # K split: whole clusters of at most 8 CTAs in one wave, each with a K chunk
        assert 1 <= p["ksplit"] <= 8, what
        if p["ksplit"] > 1:
            assert p["grid"] == p["tiles"] * p["ksplit"], what
            assert p["grid"] <= p["slots"], what
            assert p["ksplit"] <= n_chunks, what
        else:
            assert 1 <= p["grid"] <= min(p["tiles"], p["slots"]), what


@pytest.mark.parametrize("rows,cols,n_vec,warps", [
    (1024, 3072, 8, 8),     # short rows, K split kept with eight warps
    (4096, 1024, 4, 8),
    (4096, 14336, 4, 8),    # four vectors, long rows
    (4096, 14336, 8, 4),    # eight vectors on long rows: four warps
    (6144, 4096, 4, 4),     # eight warps would halve the K split (2 instead of 4)
    (28672, 4096, 4, 4),    # no K split
    (128256, 4096, 8, 4),
])
def test_q8_0_wide_warps(hq, rows, cols, n_vec, warps):
    """Q8_0 at two or more vectors takes eight consumer warps of one block
    each only on K-split launches that keep their split with them, on rows of
    at most 3072 columns or at four vectors or fewer; four warps otherwise."""
    p = plan(hq, 8, n_vec, rows, cols, 100)
    assert p["policy"] == 4 and p["tile_rows"] == 64
    assert p["cons_warps"] == warps, p
    if warps == 8:
        assert p["ksplit"] > 1 and p["ctas_per_sm"] == 2


@pytest.mark.parametrize("rows,cols,n_vec,warps", [
    (4096, 14336, 3, 8), (4096, 14336, 4, 8), (4096, 4096, 5, 8), (4096, 14336, 6, 4), (28672, 4096, 4, 4),
])
def test_q4_0_wide_warps(hq, rows, cols, n_vec, warps):
    """Q4_0 at three to five vectors takes eight warps on K-split launches that
    keep their split; four warps from six vectors on and without a K split."""
    p = plan(hq, 4, n_vec, rows, cols, 100)
    assert p["policy"] == 4 and p["tile_rows"] == 64
    assert p["cons_warps"] == warps, p


@pytest.mark.parametrize("rows,cols,n_vec,warps", [
    (4096, 14336, 3, 8), (4096, 14336, 4, 8), (4096, 14336, 5, 4), (28672, 4096, 4, 4),
])
def test_q4_k_wide_warps(hq, rows, cols, n_vec, warps):
    """Q4_K takes eight warps on K-split launches that keep their split at three
    and four vectors only."""
    p = plan(hq, 75, n_vec, rows, cols, 100)
    assert p["policy"] == 4 and p["tile_rows"] == 64
    assert p["cons_warps"] == warps, p


def test_plan_rejects_bad_arguments(hq):
    with pytest.raises(hq.HQError):
        hq.hq_debug_plan(3, 1, 64, 256, 152, 232448, 80)        # no such format
    with pytest.raises(hq.HQError):
        hq.hq_debug_plan(8, 1, 64, 320, 152, 232448, 80)        # not a multiple of 256: the plain kernel
    with pytest.raises(hq.HQError):
        hq.hq_debug_plan(8, 9, 64, 256, 152, 232448, 80)        # n_vec out of range
    with pytest.raises(hq.HQError):
        hq.hq_debug_plan(8, 1, 0, 256, 152, 232448, 80)         # no rows
    with pytest.raises(hq.HQError):
        hq.hq_debug_plan(8, 1, 64, 256, 0, 232448, 80)          # no SMs
