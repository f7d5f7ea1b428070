"""Compile-time resources of the sm_103a kernels (ptxas -v of the kernel
translation units, built into a temporary directory; the installed library is
not touched): no kernel spills registers to local memory, and the launch plans
computed with the registers the build actually uses reproduce the grids and
shared memory ncu recorded for the bench's launches."""
import pytest

from quantized_weight_matvec_hq_gb300 import build as hq_build


@pytest.fixture(scope="module")
def resources(tmp_path_factory):
    return hq_build.kernel_resources(str(tmp_path_factory.mktemp("ptxas")))


@pytest.fixture(scope="module")
def hq():
    hq_build.build()
    import quantized_weight_matvec_hq_gb300 as hq
    hq.lib()
    return hq


def regs_of(resources, fragment):
    hits = [v[0] for k, v in resources.items() if fragment in k]
    assert len(hits) == 1, (fragment, hits)
    return hits[0]


def test_no_kernel_spills(resources):
    assert len(resources) >= 30
    spilled = {k: v for k, v in resources.items() if v[1] or v[2]}
    assert not spilled, spilled


# (mangled-name fragment of the kernel, fmt, n_vec, rows, cols) -> (grid, dynamic smem bytes)
RECORDED = [
    ("INS_7PolQ8_0ELi1ELi1ELb0E", 8, 1, 28672, 4096, 448, 58880),
    ("INS_12PolQ8_0ShortELi1ELi1ELb0E", 8, 1, 6144, 1024, 192, 39648),
    ("INS_11PolColSplitINS_11PolQ8_0WideEEELi8ELi2ELb0E", 8, 8, 28672, 4096, 448, 59584),
    ("INS_11PolColSplitINS_11PolQ4_0PairEEELi1ELi2ELb0E", 4, 1, 28672, 4096, 448, 72976),
    ("INS_11PolColSplitINS_11PolQ4_KWideEEELi1ELi2ELb0E", 75, 1, 28672, 4096, 448, 72976),
]


@pytest.mark.parametrize("fragment,fmt,n_vec,rows,cols,grid,smem", RECORDED)
def test_plans_with_the_built_registers(resources, hq, fragment, fmt, n_vec, rows, cols, grid, smem):
    regs = regs_of(resources, fragment)
    p = hq.hq_debug_plan(fmt, n_vec, rows, cols, 152, 232448, regs)
    assert (p["grid"], p["smem"]) == (grid, smem)
