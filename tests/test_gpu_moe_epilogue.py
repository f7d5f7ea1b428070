"""GPU parity of the MoE epilogues against the oracle, through the C ABI:
hq_moe_matvec_q8_0_swiglu (SwiGLU over interleaved gate/up rows, "Blue --
porting zen-nano ...", section "Architecture") and hq_moe_matvec_q8_0_combine
(router-weighted sum over a token's slots, "Economical Serving ...",
paragraph "MoE is the cheapest-per-quality tier").

Tolerances.  Every matvec output is within e = 1e-3 * T + 1e-5 of the f64
oracle (T = sum_j |w_deq x_j|).  SwiGLU: |silu'| <= 1.1 everywhere, so h is
within 1.1 * e_g * (|u| + e_u) + |silu(g)| * e_u of silu(g) * u, plus fp32
rounding of the gate itself (taken as 1e-6 of the magnitude).  Combine:
within 1e-3 * sum_k |w_k| T_k + 1e-5."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from quantized_weight_matvec_hq_gb300 import synthetic

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def hq():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_weight_matvec_hq_gb300 import build
    build.build()
    import quantized_weight_matvec_hq_gb300 as hq
    hq.hq_device_fault()
    yield hq
    assert hq.hq_device_fault() == 0


@pytest.fixture(autouse=True)
def no_device_fault(request, hq):
    yield
    f = hq.hq_device_fault()
    assert f == 0, f"{request.node.name} left device fault word {f:#x}"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bank_of(g, n_experts, rows, cols):
    bank = np.empty((n_experts * rows, cols // 32 * 34), np.uint8)
    for e in range(n_experts):
        bank[e * rows:(e + 1) * rows] = oracle.quantize_q8_0(synthetic.weights(g, rows, cols))
    return bank


def swiglu_ref(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec):
    """(h_ref, tol) from the oracle's matvec outputs and the derived bound."""
    y, T = oracle.moe_matvec_q8_0(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    h = oracle.swiglu_pairs(y)
    g_, u_ = y[..., 0::2], y[..., 1::2]
    eg, eu = 1e-3 * T[..., 0::2] + 1e-5, 1e-3 * T[..., 1::2] + 1e-5
    sg = np.abs(h / np.where(u_ == 0, 1.0, u_))                  # |silu(g)|
    sg = np.where(u_ == 0, np.abs(g_), sg)
    tol = 1.1 * eg * (np.abs(u_) + eu) + sg * eu + 1e-6 * (sg + 1.1 * eg) * (np.abs(u_) + eu) + 1e-30
    return h, tol


def assert_close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    excess = np.abs(got - ref) - tol
    if not np.all(excess <= 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: {np.sum(excess > 0)} out of tolerance; worst at {i}: "
                             f"gpu {got[i]!r} ref {ref[i]!r} tol {tol[i]!r}")


def run_swiglu(hq, bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec):
    h = torch.full((n_vec, n_active, rows // 2), -7.0, dtype=torch.float32, device="cuda")
    hq.hq_moe_matvec_q8_0_swiglu(dev(bank), dev(ids), dev(x), int(x_per_slot), h, n_experts, n_active,
                                 rows, cols, n_vec)
    torch.cuda.synchronize()
    return h.cpu().numpy()


def run_combine(hq, bank, ids, x, x_per_slot, w, n_experts, n_active, rows, cols, n_vec):
    y = torch.full((n_vec, rows), -7.0, dtype=torch.float32, device="cuda")
    hq.hq_moe_matvec_q8_0_combine(dev(bank), dev(ids), dev(x), int(x_per_slot), dev(w), y,
                                  n_experts, n_active, rows, cols, n_vec)
    torch.cuda.synchronize()
    return y.cpu().numpy()


# (n_experts, n_active, rows, cols, n_vec, x_per_slot): the 128-expert top-8 bench
# shapes, K-split shapes (few row tiles), ragged row tails and duplicate experts
SWIGLU_CASES = [(128, 8, 1536, 2048, 1, False), (128, 8, 1536, 2048, 4, False), (16, 4, 200, 512, 8, False),
                (4, 2, 64, 2048, 1, False), (6, 3, 66, 256, 5, True), (3, 3, 1536, 2048, 2, False)]


@pytest.mark.parametrize("case", SWIGLU_CASES)
def test_swiglu_parity(hq, case):
    n_experts, n_active, rows, cols, n_vec, x_per_slot = case
    g = synthetic.rng(5000 + rows + n_vec)
    bank = bank_of(g, n_experts, rows, cols)
    ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    x = synthetic.activations(g, n_vec * (n_active if x_per_slot else 1), cols) * np.float32(8.0)
    h = run_swiglu(hq, bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    h_ref, tol = swiglu_ref(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    assert_close(h, h_ref, tol, f"swiglu {case}")
    # both tails of the gate were exercised
    y, _ = oracle.moe_matvec_q8_0(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    assert (y[..., 0::2] < -1.0).any() and (y[..., 0::2] > 1.0).any()


# the 128-expert top-8 down projection at every bench width (clusters of 8 and
# of 7 CTAs per row tile), fewer groups than cluster CTAs, more groups than
# cluster CTAs (n_vec 8: up to 64), ragged row tails, and more row tiles than
# one wave of CTAs (one CTA per tile, no cluster)
COMBINE_CASES = [(128, 8, 2048, 768, 1), (128, 8, 2048, 768, 4), (128, 8, 2048, 768, 8), (8, 4, 100, 512, 3),
                 (4, 2, 64, 2048, 1), (5, 5, 33, 256, 2), (64, 32, 96, 256, 8), (2, 2, 40000, 256, 1)]


@pytest.mark.parametrize("case", COMBINE_CASES)
def test_combine_parity_and_determinism(hq, case):
    n_experts, n_active, rows, cols, n_vec = case
    g = synthetic.rng(6000 + rows + n_vec)
    bank = bank_of(g, n_experts, rows, cols)
    ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    x = synthetic.activations(g, n_vec * n_active, cols)
    w = synthetic.router_weights(g, n_vec, n_active)
    y = run_combine(hq, bank, ids, x, True, w, n_experts, n_active, rows, cols, n_vec)
    y_slots, T = oracle.moe_matvec_q8_0(bank, ids, x, True, n_experts, n_active, rows, cols, n_vec)
    out, Tout = oracle.moe_combine(y_slots, T, w)
    assert_close(y, out, 1e-3 * Tout + 1e-5, f"combine {case}")
    y2 = run_combine(hq, bank, ids, x, True, w, n_experts, n_active, rows, cols, n_vec)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_combine_shared_x(hq):
    """x shared by a token's slots (x_per_slot = 0): the weighted sum of the
    chosen experts applied to one input."""
    n_experts, n_active, rows, cols, n_vec = 16, 4, 256, 1024, 3
    g = synthetic.rng(6050)
    bank = bank_of(g, n_experts, rows, cols)
    ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    x = synthetic.activations(g, n_vec, cols)
    w = synthetic.router_weights(g, n_vec, n_active)
    y = run_combine(hq, bank, ids, x, False, w, n_experts, n_active, rows, cols, n_vec)
    y_slots, T = oracle.moe_matvec_q8_0(bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    out, Tout = oracle.moe_combine(y_slots, T, w)
    assert_close(y, out, 1e-3 * Tout + 1e-5, "combine, shared x")


def test_combine_signed_weights_and_duplicates(hq):
    """Signed weights (not a softmax) and slots that share experts: the sum is
    still the plain weighted sum of the slots."""
    n_experts, n_active, rows, cols, n_vec = 6, 3, 96, 512, 4
    g = synthetic.rng(6100)
    bank = bank_of(g, n_experts, rows, cols)
    ids = np.array([[0, 1, 2], [2, 2, 2], [5, 0, 5], [1, 4, 3]], dtype=np.int32)
    x = synthetic.activations(g, n_vec * n_active, cols)
    w = g.standard_normal((n_vec, n_active)).astype(np.float32)
    y = run_combine(hq, bank, ids, x, True, w, n_experts, n_active, rows, cols, n_vec)
    y_slots, T = oracle.moe_matvec_q8_0(bank, ids, x, True, n_experts, n_active, rows, cols, n_vec)
    out, Tout = oracle.moe_combine(y_slots, T, w)
    assert_close(y, out, 1e-3 * Tout + 1e-5, "signed weights")


def test_invalid_ids_in_epilogues(hq):
    n_experts, n_active, rows, cols, n_vec = 4, 2, 64, 256, 2
    g = synthetic.rng(6200)
    bank = bank_of(g, n_experts, rows, cols)
    ids = np.array([[1, 2], [3, 9]], dtype=np.int32)
    xs = synthetic.activations(g, n_vec, cols)
    h = run_swiglu(hq, bank, ids, xs, False, n_experts, n_active, rows, cols, n_vec)
    assert hq.hq_device_fault() == hq.HQ_FAULT_EXPERT_ID
    assert np.all(np.isnan(h[1, 1])) and not np.isnan(h[0]).any()
    ok = np.array([[1, 2], [3, 0]], dtype=np.int32)
    h_ref, tol = swiglu_ref(bank, ok, xs, False, n_experts, n_active, rows, cols, n_vec)
    assert_close(h[0], h_ref[0], tol[0], "valid token beside an invalid id")
    xp = synthetic.activations(g, n_vec * n_active, cols)
    w = synthetic.router_weights(g, n_vec, n_active)
    y = run_combine(hq, bank, ids, xp, True, w, n_experts, n_active, rows, cols, n_vec)
    assert hq.hq_device_fault() == hq.HQ_FAULT_EXPERT_ID
    assert np.all(np.isnan(y[1])) and not np.isnan(y[0]).any()
    y_slots, T = oracle.moe_matvec_q8_0(bank, ok, xp, True, n_experts, n_active, rows, cols, n_vec)
    out, Tout = oracle.moe_combine(y_slots, T, w)
    assert_close(y[0], out[0], 1e-3 * Tout[0] + 1e-5, "valid token beside an invalid id")
    # every id invalid: no group forms and every sum is NaN
    bad = np.array([[7, 8], [-1, 4]], dtype=np.int32)
    y = run_combine(hq, bank, bad, xp, True, w, n_experts, n_active, rows, cols, n_vec)
    assert hq.hq_device_fault() == hq.HQ_FAULT_EXPERT_ID
    assert np.all(np.isnan(y))


@pytest.mark.parametrize("down_flags", [0, 1])
def test_moe_ffn_chain_in_graph(hq, down_flags):
    """Two MoE feed-forward layers, each gate|up + SwiGLU then down + combine,
    the next layer reading the previous layer's combined output, captured in a
    CUDA graph and replayed with two different inputs and routings.  Each stage
    is checked against the oracle on the GPU's own input to that stage.  With
    HQ_MOE_IDS_READY the down launches (their ids were written before the
    gate|up launch) start their weight copies before gate|up ends."""
    n_experts, n_active, hidden, inter, n_vec = 16, 4, 512, 256, 2
    g = synthetic.rng(6300)
    layers = []
    for _ in range(2):
        gu = bank_of(g, n_experts, 2 * inter, hidden)
        down = bank_of(g, n_experts, hidden, inter)
        layers.append((gu, down, dev(gu), dev(down)))
    x0 = torch.zeros((n_vec, hidden), dtype=torch.float32, device="cuda")
    ids_d = [torch.zeros((n_vec, n_active), dtype=torch.int32, device="cuda") for _ in layers]
    w_d = [torch.zeros((n_vec, n_active), dtype=torch.float32, device="cuda") for _ in layers]
    h_d = [torch.empty((n_vec, n_active, inter), dtype=torch.float32, device="cuda") for _ in layers]
    out_d = [torch.empty((n_vec, hidden), dtype=torch.float32, device="cuda") for _ in layers]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def step():
        xin = x0
        for li, (_, _, gud, downd) in enumerate(layers):
            hq.hq_moe_matvec_q8_0_swiglu(gud, ids_d[li], xin, 0, h_d[li], n_experts, n_active, 2 * inter, hidden,
                                         n_vec, stream=s.cuda_stream)
            hq.hq_moe_matvec_q8_0_ex(downd, ids_d[li], h_d[li], 1, w_d[li], out_d[li], n_experts, n_active,
                                     hidden, inter, n_vec, hq.HQ_MOE_EPI_COMBINE, down_flags, stream=s.cuda_stream)
            xin = out_d[li]

    with torch.cuda.stream(s):
        step()                                                  # warm (module set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for rep in range(2):
        x = synthetic.activations(g, n_vec, hidden)
        ids = [synthetic.expert_ids(g, n_vec, n_active, n_experts) for _ in layers]
        ws = [synthetic.router_weights(g, n_vec, n_active) for _ in layers]
        x0.copy_(torch.from_numpy(x))
        for li in range(len(layers)):
            ids_d[li].copy_(torch.from_numpy(ids[li]))
            w_d[li].copy_(torch.from_numpy(ws[li]))
        graph.replay()
        torch.cuda.synchronize()
        xin = x
        for li, (gu, down, _, _) in enumerate(layers):
            h_ref, tol = swiglu_ref(gu, ids[li], xin, False, n_experts, n_active, 2 * inter, hidden, n_vec)
            h = h_d[li].cpu().numpy()
            assert_close(h, h_ref, tol, f"replay {rep} layer {li} swiglu")
            y_slots, T = oracle.moe_matvec_q8_0(down, ids[li], h, True, n_experts, n_active, hidden, inter, n_vec)
            out, Tout = oracle.moe_combine(y_slots, T, ws[li])
            y = out_d[li].cpu().numpy()
            assert_close(y, out, 1e-3 * Tout + 1e-5, f"replay {rep} layer {li} combine")
            xin = y
