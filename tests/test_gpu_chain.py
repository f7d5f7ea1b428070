"""GPU tests of what a decode step relies on beyond single-call parity:
matvecs chained through their outputs inside a captured CUDA graph (every
launch allows programmatic dependent launch, so a kernel may start before
the previous one ends and must not read x, or MoE expert ids, before it has
waited for it), and the bounded-wait failure path of the fault word."""
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


def assert_within(y, y_ref, T, what):
    y = np.asarray(y, dtype=np.float64)
    excess = np.abs(y - y_ref) - (1e-3 * T + 1e-5)
    assert np.all(excess <= 0), f"{what}: {np.sum(excess > 0)} outputs out of tolerance"


def quant(fmt, W):
    return oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)


def test_dense_chain_in_graph(hq):
    """x0 -> Q8_0 4096x4096 -> Q4_0 4096x4096 -> Q8_0 1024x4096, each launch's x
    the previous launch's y, captured once and replayed with two different x0.
    Each stage is checked against the oracle on the GPU's own input to it."""
    g = synthetic.rng(4242)
    stages = [("q8_0", 4096, 4096), ("q4_0", 4096, 4096), ("q8_0", 1024, 4096)]
    blocks = [quant(f, synthetic.weights(g, r, c)) for (f, r, c) in stages]
    Wd = [torch.from_numpy(b).cuda() for b in blocks]
    x0 = torch.empty((1, 4096), dtype=torch.float32, device="cuda")
    ys = [torch.empty((1, r), dtype=torch.float32, device="cuda") for (_, r, _) in stages]

    def launch(stream):
        x = x0
        for (f, r, c), w, y in zip(stages, Wd, ys):
            fn = hq.hq_matvec_q8_0 if f == "q8_0" else hq.hq_matvec_q4_0
            fn(w, x, y, r, c, 1, stream=stream)
            x = y

    s = torch.cuda.Stream()
    x0.copy_(torch.from_numpy(synthetic.activations(g, 1, 4096)))
    with torch.cuda.stream(s):
        launch(s.cuda_stream)                      # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch(torch.cuda.current_stream().cuda_stream)
    for trial in range(2):
        x_np = synthetic.activations(g, 1, 4096)
        x0.copy_(torch.from_numpy(x_np))
        for y in ys:
            y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        x_in = x_np
        for k, ((f, r, c), b, y) in enumerate(zip(stages, blocks, ys)):
            y_np = y.cpu().numpy()
            y_ref, T = oracle.matvec(f, b, x_in, r, c)
            assert_within(y_np, y_ref, T, f"trial {trial} stage {k} {f} {r}x{c}")
            x_in = y_np


@pytest.mark.parametrize("down_flags", [0, 1])
def test_moe_chain_with_device_ids_in_graph(hq, down_flags):
    """A small kernel writes the expert ids right before the MoE gate launch,
    and the down launch reads the gate launch's output as its per-slot x; the
    whole chain is captured and replayed with two different routings.  With
    HQ_MOE_IDS_READY on the down launch (its ids were written before the gate
    launch), the down kernel reads the ids and starts its weight copies while
    the gate launch still runs, and must still take x only after it ends."""
    E, A, H, F = 128, 8, 2048, 768
    g = synthetic.rng(4343)
    gate = np.empty((E * F, H // 32 * 34), np.uint8)
    down = np.empty((E * H, F // 32 * 34), np.uint8)
    for e in range(E):
        gate[e * F:(e + 1) * F] = oracle.quantize_q8_0(synthetic.weights(g, F, H))
        down[e * H:(e + 1) * H] = oracle.quantize_q8_0(synthetic.weights(g, H, F))
    gate_d, down_d = torch.from_numpy(gate).cuda(), torch.from_numpy(down).cuda()
    x = torch.from_numpy(synthetic.activations(g, 1, H)).cuda()
    seed = torch.zeros(A, dtype=torch.int32, device="cuda")
    ids = torch.empty((1, A), dtype=torch.int32, device="cuda")
    step = torch.arange(A, dtype=torch.int32, device="cuda") * 17
    y_gate = torch.empty((1, A, F), dtype=torch.float32, device="cuda")
    y_down = torch.empty((1, A, H), dtype=torch.float32, device="cuda")

    def launch(stream):
        torch.remainder(seed + step, E, out=ids.view(-1))          # ids written on the device
        hq.hq_moe_matvec_q8_0(gate_d, ids, x, 0, y_gate, E, A, F, H, 1, stream=stream)
        hq.hq_moe_matvec_q8_0_ex(down_d, ids, y_gate, 1, None, y_down, E, A, H, F, 1, hq.HQ_MOE_EPI_NONE,
                                 down_flags, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch(s.cuda_stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        launch(torch.cuda.current_stream().cuda_stream)
    for base in (3, 90):
        seed.fill_(base)
        y_gate.fill_(float("nan"))
        y_down.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        ids_np = ((base + 17 * np.arange(A)) % E).astype(np.int32).reshape(1, A)
        assert np.array_equal(ids.cpu().numpy(), ids_np)
        yg = y_gate.cpu().numpy()
        yg_ref, Tg = oracle.moe_matvec_q8_0(gate, ids_np, x.cpu().numpy(), False, E, A, F, H, 1)
        assert_within(yg, yg_ref, Tg, f"moe gate, routing {base}")
        yd_ref, Td = oracle.moe_matvec_q8_0(down, ids_np, yg.reshape(A, F), True, E, A, H, F, 1)
        assert_within(y_down.cpu().numpy(), yd_ref, Td, f"moe down (flags {down_flags}), routing {base}")
    assert hq.hq_device_fault() == 0


def test_wait_timeout_sets_fault_word_and_context_survives(hq):
    """A bounded wait that nothing completes gives up after its limit, records
    the timeout (CTA 0, consumer bit) in the fault word and returns; the next
    matvec on the same context is exact."""
    assert hq.hq_device_fault() == 0
    hq.hq_selftest_wait_timeout(2_000_000)          # about a millisecond of SM cycles
    torch.cuda.synchronize()
    word = hq.hq_device_fault()
    assert word & hq.HQ_FAULT_WAIT_TIMEOUT
    assert (word >> 9) == 0 and (word & 0x100)      # CTA 0, a consumer-side wait
    assert hq.hq_device_fault() == 0                # reading clears it
    g = synthetic.rng(7)
    rows, cols = 64, 512
    b = oracle.quantize_q8_0(synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, 1, cols)
    y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
    hq.hq_matvec_q8_0(torch.from_numpy(b).cuda(), torch.from_numpy(x).cuda(), y, rows, cols, 1)
    y_ref, T = oracle.matvec("q8_0", b, x, rows, cols)
    assert_within(y.cpu().numpy(), y_ref, T, "matvec after the self-test")
