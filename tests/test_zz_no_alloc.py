"""The allocation-free QLoRA entry point, hq_matvec_q8_0_lora_noalloc: its
down projection u = A x lives in the library's static per-device scratch, so
the call takes no workspace and allocates nothing.  It must give the same
bits as hq_matvec_q8_0_lora with a caller workspace (the same kernels), match
the oracle, leave device memory untouched, and run inside a captured graph.
(Collected last: it runs after every other GPU test.)"""
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
    y0 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    y1 = torch.empty((n_vec, rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(rank * n_vec, dtype=torch.float32, device="cuda")
    hq.hq_matvec_q8_0_lora(Wd, xd, Ad, Bd, 1.5, rank, ws, y0, rows, cols, n_vec)
    hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 1.5, rank, y1, rows, cols, n_vec)
    torch.cuda.synchronize()
    a, b = y0.cpu().numpy(), y1.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    y_b, T_b = oracle.matvec("q8_0", blocks, x, rows, cols)
    dl, T_d = oracle.lora_delta(A, B, x, 1.5)
    excess = np.abs(b.astype(np.float64) - (y_b + dl)) - (1e-3 * (T_b + T_d) + 1e-5)
    assert np.all(excess <= 0)
    assert hq.hq_device_fault() == 0


def test_noalloc_takes_no_device_memory_and_captures(hq):
    rows, cols, rank = 4096, 4096, 16
    blocks, A, B, x, Wd, Ad, Bd, xd = make(rows, cols, rank, 1, 1300)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 2.0, rank, y, rows, cols, 1)      # warm (module set-up)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 2.0, rank, y, rows, cols, 1)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ref = y.clone()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        hq.hq_matvec_q8_0_lora_noalloc(Wd, xd, Ad, Bd, 2.0, rank, y, rows, cols, 1,
                                       stream=torch.cuda.current_stream().cuda_stream)
    y.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert hq.hq_device_fault() == 0
