"""The QLoRA entry point for callers that cannot allocate device memory,
hq_matvec_q8_0_lora_noalloc.  Such callers cannot hand the library a
workspace: an engine that keeps all device memory in its own pool, or a path
that must not call cudaMalloc, which may synchronize the device.  The call
keeps u = A x in the library's static per-device scratch instead.  Two calls
in a row (different inputs, so the second must overwrite the first's scratch)
must give the same bits as hq_matvec_q8_0_lora with a caller workspace and
match the oracle within the tests' tolerance.  Repeated calls must leave the
free device memory unchanged.  Collected last, so that a run which stops at
the first failure has run every other test; it also passes run alone.
"""
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


def bf16_bits(a):
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def make(rows, cols, rank, n_vec, seed):
    g = synthetic.rng(seed)
    blocks = oracle.quantize_q8_0(synthetic.weights(g, rows, cols))
    A = bf16_bits(g.standard_normal((rank, cols)) * 0.02)
    B = bf16_bits(g.standard_normal((rows, rank)) * 0.02)
    x = synthetic.activations(g, n_vec, cols)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return blocks, A, B, x, d(blocks), d(A), d(B), d(x)


@pytest.mark.parametrize("rows,cols,rank,n_vec", [(100, 4096, 16, 1), (1000, 2048, 64, 8), (257, 3072, 1, 2),
                                                  (130, 320, 8, 3)])
def test_noalloc_matches_oracle_and_workspace_call(hq, rows, cols, rank, n_vec):
    blocks, A, B, x, Wd, Ad, Bd, xd = make(rows, cols, rank, n_vec, 1200 + rows + rank)
    g = synthetic.rng(1900 + rows + rank)
    x2 = synthetic.activations(g, n_vec, cols)
    xd2 = torch.from_numpy(x2).cuda()
    ws = torch.empty(rank * n_vec, dtype=torch.float32, device="cuda")
    y_ws = [torch.empty((n_vec, rows), dtype=torch.float32, device="cuda") for _ in range(2)]
    y_na = [torch.empty((n_vec, rows), dtype=torch.float32, device="cuda") for _ in range(2)]
    # the workspace call on both inputs, then two allocation-free calls in a row
    for xi, yi in zip((xd, xd2), y_ws):
        hq.hq_matvec_q8_0_lora(Wd, xi, Ad, Bd, 1.5, rank, ws, yi, rows, cols, n_vec)
    for xi, yi in zip((xd, xd2), y_na):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xi, Ad, Bd, 1.5, rank, yi, rows, cols, n_vec)
    torch.cuda.synchronize()
    for xh, a_t, b_t in zip((x, x2), y_ws, y_na):
        a, b = a_t.cpu().numpy(), b_t.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        y_b, T_b = oracle.matvec("q8_0", blocks, xh, rows, cols)
        dl, T_d = oracle.lora_delta(A, B, xh, 1.5)
        excess = np.abs(b.astype(np.float64) - (y_b + dl)) - (1e-3 * (T_b + T_d) + 1e-5)
        assert np.all(excess <= 0)
    assert hq.hq_device_fault() == 0


def test_noalloc_rejects_sizes_beyond_the_scratch(hq):
    blocks, A, B, x, Wd, Ad, Bd, xd = make(64, 256, 65, 1, 1250)
    y = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(hq.HQError):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 1.0, 65, y, 64, 256, 1)


def test_noalloc_takes_no_device_memory(hq):
    rows, cols, rank = 4096, 4096, 16
    blocks, A, B, x, Wd, Ad, Bd, xd = make(rows, cols, rank, 1, 1300)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 2.0, rank, y, rows, cols, 1)      # the device's set-up
    torch.cuda.synchronize()
    ref = y.clone()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 2.0, rank, y, rows, cols, 1)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.equal(y, ref)
    assert hq.hq_device_fault() == 0


def test_noalloc_in_captured_graph(hq):
    """After one eager call (the device's set-up), the allocation-free call is
    captured in a CUDA graph; two replays with different x give the eager
    call's bits on the same x."""
    rows, cols, rank, n_vec = 1000, 4096, 16, 2
    blocks, A, B, x, Wd, Ad, Bd, xd = make(rows, cols, rank, n_vec, 1400)
    g = synthetic.rng(1401)
    xs = [synthetic.activations(g, n_vec, cols) for _ in range(2)]
    y = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    eager = []
    with torch.cuda.stream(s):
        for xi in xs:
            xd.copy_(torch.from_numpy(xi))
            hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 0.5, rank, y, rows, cols, n_vec,
                                          stream=s.cuda_stream)
            eager.append(y.clone())
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 0.5, rank, y, rows, cols, n_vec,
                                      stream=torch.cuda.current_stream().cuda_stream)
    for xi, ref in zip(xs, eager):
        xd.copy_(torch.from_numpy(xi))
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, ref)
    assert hq.hq_device_fault() == 0
