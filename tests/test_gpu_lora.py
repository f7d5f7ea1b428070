"""GPU parity of the QLoRA entry points against the oracle ("One Native Stack
...", section "The Central Efficiency Thesis", Lemma "QLoRA over the unified
core is exact": y = What x + (alpha/r) B_A (A x), A and B_A in bf16)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_weight_matvec_hq_gb300 import synthetic

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def hq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_weight_matvec_hq_gb300 import build
    build.build()
    import quantized_weight_matvec_hq_gb300 as hq
    return hq


@pytest.fixture(autouse=True)
def no_device_fault(hq):
    yield
    assert hq.hq_device_fault() == 0


def bf16_bits(a):
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, T, what):
    y = np.asarray(y, dtype=np.float64)
    excess = np.abs(y - y_ref) - (1e-3 * T + 1e-5)
    if not np.all(excess <= 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: {np.sum(excess > 0)} outputs out of tolerance; worst at {i}: "
                             f"gpu {y[i]!r} ref {y_ref[i]!r} T {T[i]!r}")


def case(fmt, rows, cols, rank, n_vec, seed):
    g = synthetic.rng(seed)
    W = synthetic.weights(g, rows, cols)
    blocks = oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)
    A = bf16_bits(g.standard_normal((rank, cols)) * 0.02)
    B = bf16_bits(g.standard_normal((rows, rank)) * 0.02)
    x = synthetic.activations(g, n_vec, cols)
    return blocks, A, B, x


def run(hq, fmt, blocks, A, B, x, scale, rows, cols):
    rank, n_vec = A.shape[0], x.shape[0]
    y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(rank * n_vec, dtype=torch.float32, device="cuda")
    fn = hq.hq_matvec_q8_0_lora if fmt == "q8_0" else hq.hq_matvec_q4_0_lora
    fn(dev(blocks), dev(x), dev(A), dev(B), scale, rank, ws, y, rows, cols, n_vec)
    torch.cuda.synchronize()
    return y.cpu().numpy(), ws


def reference(fmt, blocks, A, B, x, scale, rows, cols):
    y_b, T_b = oracle.matvec(fmt, blocks, x, rows, cols)
    d, T_d = oracle.lora_delta(A, B, x, scale)
    return y_b + d, T_b + T_d


# (rows, cols): few tiles (K split over a cluster), many tiles, ragged rows,
# and a cols % 256 != 0 shape on the plain-load kernel
SHAPES = [(100, 4096), (1000, 2048), (257, 3072), (64, 14336), (130, 320)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_lora_parity(hq, fmt, rows, cols):
    for rank, n_vec, scale in ((1, 1, 0.5), (16, 2, 2.0), (64, 4, -0.125), (8, 8, 1.0)):
        blocks, A, B, x = case(fmt, rows, cols, rank, n_vec, 500 + rows + rank)
        y, _ = run(hq, fmt, blocks, A, B, x, scale, rows, cols)
        y_ref, T = reference(fmt, blocks, A, B, x, scale, rows, cols)
        assert_within(y, y_ref, T, f"{fmt} {rows}x{cols} rank={rank} n_vec={n_vec}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_lora_zero_adapter_is_the_served_output(hq, fmt):
    """With B = 0 the output is bit for bit the plain matvec of the same bytes
    (the Lemma's "frozen base" term is the served decode output)."""
    rows, cols = 513, 4096
    blocks, A, B, x = case(fmt, rows, cols, 16, 1, 77)
    y, _ = run(hq, fmt, blocks, A, np.zeros_like(B), x, 1.0, rows, cols)
    y0 = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    (hq.hq_matvec_q8_0 if fmt == "q8_0" else hq.hq_matvec_q4_0)(dev(blocks), dev(x), y0, rows, cols, 1)
    torch.cuda.synchronize()
    assert np.array_equal(y.view(np.uint32), y0.cpu().numpy().view(np.uint32))


def test_lora_workspace_holds_down_projection_and_is_deterministic(hq):
    rows, cols, rank, n_vec = 300, 2048, 16, 3
    blocks, A, B, x = case("q8_0", rows, cols, rank, n_vec, 78)
    y1, ws = run(hq, "q8_0", blocks, A, B, x, 0.75, rows, cols)
    u = ws.cpu().numpy().reshape(n_vec, rank).astype(np.float64)
    Af = np.array([[oracle.bf16_to_float(int(h)) for h in row] for row in A])
    u_ref = x.astype(np.float64) @ Af.T
    u_mag = np.abs(x.astype(np.float64)) @ np.abs(Af).T
    assert np.all(np.abs(u - u_ref) <= 1e-5 * u_mag + 1e-12)
    y2, _ = run(hq, "q8_0", blocks, A, B, x, 0.75, rows, cols)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_launch_count_per_call(hq):
    """The library's launch counter: one kernel per plain matvec, two per
    adapted matvec (the down projection, then the matvec)."""
    rows, cols, rank = 256, 2048, 16
    blocks, A, B, x = case("q8_0", rows, cols, rank, 1, 1600)
    Wd, xd, Ad, Bd = dev(blocks), dev(x), dev(A), dev(B)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(rank, dtype=torch.float32, device="cuda")
    n0 = hq.hq_launch_count()
    hq.hq_matvec_q8_0(Wd, xd, y, rows, cols, 1)
    n1 = hq.hq_launch_count()
    hq.hq_matvec_q8_0_lora(Wd, xd, Ad, Bd, 1.0, rank, ws, y, rows, cols, 1)
    n2 = hq.hq_launch_count()
    torch.cuda.synchronize()
    assert (n1 - n0, n2 - n1) == (1, 2)


def test_lora_one_workspace_for_every_shape(hq):
    """One workspace of the largest size (rank 64 x 8 vectors) serves calls of
    different ranks, widths and shapes in turn, on both the TMA kernel and the
    plain-load kernel (cols % 256 != 0)."""
    ws = torch.empty(64 * 8, dtype=torch.float32, device="cuda")
    for k, (fmt, rows, cols, rank, n_vec) in enumerate([("q8_0", 500, 4096, 16, 1), ("q4_0", 257, 3072, 1, 2),
                                                        ("q8_0", 1000, 2048, 64, 8), ("q4_0", 4096, 14336, 16, 1),
                                                        ("q8_0", 300, 2336, 8, 3)]):
        blocks, A, B, x = case(fmt, rows, cols, rank, n_vec, 1500 + k)
        y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
        fn = hq.hq_matvec_q8_0_lora if fmt == "q8_0" else hq.hq_matvec_q4_0_lora
        fn(dev(blocks), dev(x), dev(A), dev(B), 1.25, rank, ws, y, rows, cols, n_vec)
        torch.cuda.synchronize()
        y_ref, T = reference(fmt, blocks, A, B, x, 1.25, rows, cols)
        assert_within(y.cpu().numpy(), y_ref, T, f"shared workspace call {k}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", [(28672, 4096), (4096, 14336)])
def test_lora_full_size_8b_sampled(hq, fmt, rows, cols):
    """Rank-16 adapters on full 8B decode shapes, in the bench's launch
    configuration; sampled rows against the oracle."""
    rank = 16
    g = synthetic.rng(synthetic.SEED_BASE + 11)
    W = synthetic.weights(g, rows, cols)
    blocks = oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)
    del W
    A = bf16_bits(g.standard_normal((rank, cols)) * 0.02)
    B = bf16_bits(g.standard_normal((rows, rank)) * 0.02)
    x = synthetic.activations(g, 1, cols)
    y, _ = run(hq, fmt, blocks, A, B, x, 2.0, rows, cols)
    for lo in np.linspace(0, rows - 5, 16).astype(int):
        lo = int(lo)
        y_b, T_b = oracle.matvec_rows(fmt, blocks, x, rows, cols, lo, lo + 5)
        d, T_d = oracle.lora_delta(A, B[lo:lo + 5], x, 2.0)
        assert_within(y[:, lo:lo + 5], y_b + d, T_b + T_d, f"{fmt} {rows}x{cols} rows {lo}")


def test_lora_chain_in_graph(hq):
    """Two adapted matvecs chained (the second's x is the first's y), captured
    in a CUDA graph and replayed with new inputs: the down projection and the
    matvec both start early under programmatic launch and must still read
    their inputs only after the kernels that write them."""
    rows, cols, rank = 4096, 4096, 16
    stages = []
    for k, fmt in enumerate(("q8_0", "q4_0")):
        blocks, A, B, _ = case(fmt, rows, cols, rank, 1, 900 + k)
        stages.append((fmt, blocks, A, B, dev(blocks), dev(A), dev(B),
                       torch.empty(rank, dtype=torch.float32, device="cuda")))
    x0 = torch.empty((1, cols), dtype=torch.float32, device="cuda")
    ys = [torch.empty((1, rows), dtype=torch.float32, device="cuda") for _ in stages]

    def launch(stream):
        x = x0
        for (fmt, _, _, _, Wd, Ad, Bd, ws), y in zip(stages, ys):
            fn = hq.hq_matvec_q8_0_lora if fmt == "q8_0" else hq.hq_matvec_q4_0_lora
            fn(Wd, x, Ad, Bd, 0.5, rank, ws, y, rows, cols, 1, stream=stream)
            x = y

    s = torch.cuda.Stream()
    g = synthetic.rng(901)
    x0.copy_(torch.from_numpy(synthetic.activations(g, 1, cols)))
    with torch.cuda.stream(s):
        launch(s.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch(torch.cuda.current_stream().cuda_stream)
    for trial in range(2):
        x_np = synthetic.activations(g, 1, cols)
        x0.copy_(torch.from_numpy(x_np))
        for y in ys:
            y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        x_in = x_np
        for (fmt, blocks, A, B, *_), y in zip(stages, ys):
            y_np = y.cpu().numpy()
            y_ref, T = reference(fmt, blocks, A, B, x_in, 0.5, rows, cols)
            assert_within(y_np, y_ref, T, f"trial {trial} {fmt}")
            x_in = y_np
