"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: quantized bytes, int8 weights and int8 outputs bit-exact; float outputs
within |y - y_ref| <= 1e-3 * sum_j |w_deq x_j| + 1e-5 per output (the oracle
accumulates in f64 and returns the |w x| sum).  Inputs are seeded synthetic
draws (W ~ N(0, 0.02), x ~ N(0, 1)); quantized inputs come from the oracle's
quantizer, never from the GPU.
"""
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
    """Every test leaves the device fault word clear (the invalid-id test clears
    the bit it expects itself): no bounded wait may ever time out."""
    yield
    f = hq.hq_device_fault()
    assert f == 0, f"{request.node.name} left device fault word {f:#x}: {hq.hq_last_error()}"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def assert_within(y, y_ref, T, what=""):
    y = np.asarray(y, dtype=np.float64)
    excess = np.abs(y - y_ref) - (1e-3 * T + 1e-5)
    if not np.all(excess <= 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(f"{what}: {np.sum(excess > 0)} outputs out of tolerance; worst at {i}: "
                             f"gpu {y[i]!r} ref {y_ref[i]!r} T {T[i]!r}")


def gpu_matvec(hq, fmt, blocks, x, rows, cols, stream=None):
    n_vec = x.shape[0]
    y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    fn = hq.hq_matvec_q8_0 if fmt == "q8_0" else hq.hq_matvec_q4_0
    fn(dev(blocks), dev(x), y, rows, cols, n_vec, stream=stream)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def quant(fmt, W):
    return oracle.quantize_q8_0(W) if fmt == "q8_0" else oracle.quantize_q4_0(W)


# ---------------------------------------------------------------- quantizers

def _special_weights(rows, cols, seed):
    g = synthetic.rng(seed)
    W = synthetic.weights(g, rows, cols)
    W[0, :] = 0                                            # all-zero blocks
    W[1, :32] = np.float32(-1e-30)                         # tiny: d underflows in fp16
    W[2, 0], W[2, 5] = np.float32(0.8), np.float32(-0.8)   # |max| tie, clamps to 15 in Q4_0
    W[3, ::7] *= np.float32(300)                           # outliers
    W[4, :32] = np.float32(0.25)                           # equal elements
    W[5, :32] = np.arange(32, dtype=np.float32) * np.float32(0.0625) - np.float32(1)  # exact ratios
    return W


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_quantizer_bytes_bit_exact(hq, fmt):
    rows, cols = 301, 1024 + 96
    W = _special_weights(rows, cols, 31)
    out = torch.empty((rows, cols // 32 * (34 if fmt == "q8_0" else 18)), dtype=torch.uint8, device="cuda")
    (hq.hq_quantize_q8_0 if fmt == "q8_0" else hq.hq_quantize_q4_0)(dev(W), out, rows, cols)
    torch.cuda.synchronize()
    got, ref = out.cpu().numpy(), quant(fmt, W)
    bpb = 34 if fmt == "q8_0" else 18
    g3, r3 = got.reshape(rows, -1, bpb), ref.reshape(rows, -1, bpb)
    bad_d = np.argwhere(np.any(g3[:, :, :2] != r3[:, :, :2], axis=2))
    bad_q = np.argwhere(np.any(g3[:, :, 2:] != r3[:, :, 2:], axis=2))
    assert len(bad_d) == 0 and len(bad_q) == 0, (
        f"{len(bad_d)} blocks with a different scale (first {bad_d[:3].tolist()}: gpu "
        f"{g3[tuple(bad_d[0])][:2].tolist() if len(bad_d) else None} ref "
        f"{r3[tuple(bad_d[0])][:2].tolist() if len(bad_d) else None}), {len(bad_q)} with different quants")


def test_quantizer_i8_rows_bit_exact(hq):
    rows, cols = 97, 3000
    W = _special_weights(rows, cols, 32)
    Wq = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    hq.hq_quantize_i8_rows(dev(W), Wq, s, rows, cols)
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quantize_i8_rows(W)
    assert np.array_equal(Wq.cpu().numpy(), q_ref)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_ref.view(np.uint32))


# ---------------------------------------------------------------- float matvecs

# (rows, cols): tiles of 32/64 rows with ragged tails; cols % 256 == 0 use the
# TMA kernel (few row tiles -> K split over a cluster, many -> persistent
# CTAs); other multiples of 32 use the plain-load kernel.
SHAPES = [(1, 256), (31, 512), (33, 1024), (100, 4096), (257, 3072), (1000, 2048),
          (64, 14336), (5000, 256), (7, 32), (45, 96), (130, 320), (64, 992)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_matvec_parity(hq, fmt, rows, cols):
    g = synthetic.rng(1000 + rows + cols)
    W = synthetic.weights(g, rows, cols)
    blocks = quant(fmt, W)
    for n_vec in (1, 2, 3, 4, 5, 8) if rows * cols <= 1 << 20 else (1, 4, 8):
        x = synthetic.activations(g, n_vec, cols)
        y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
        y = gpu_matvec(hq, fmt, blocks, x, rows, cols)
        assert_within(y, y_ref, T, f"{fmt} {rows}x{cols} n_vec={n_vec}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_all_n_vec_and_column_independence(hq, fmt):
    rows, cols = 200, 2048
    g = synthetic.rng(77)
    blocks = quant(fmt, synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, 8, cols)
    y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
    for n_vec in range(1, 9):
        y = gpu_matvec(hq, fmt, blocks, x[:n_vec], rows, cols)
        assert_within(y, y_ref[:n_vec], T[:n_vec], f"{fmt} n_vec={n_vec}")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_closed_forms_on_gpu(hq, fmt):
    rows, cols = 96, 1024
    g = synthetic.rng(78)
    W = synthetic.weights(g, rows, cols)
    W[10] = 0
    blocks = quant(fmt, W)
    Wd = oracle.dequant(fmt, blocks, rows, cols)
    # one-hot x: exactly one column (d*q is exact in fp32, no rounding happens)
    for j in (0, 33, 511, 1023):
        e = np.zeros((1, cols), np.float32)
        e[0, j] = 1
        y = gpu_matvec(hq, fmt, blocks, e, rows, cols)
        assert np.array_equal(y[0].astype(np.float64), Wd[:, j])
    y = gpu_matvec(hq, fmt, blocks, synthetic.activations(g, 2, cols), rows, cols)
    assert np.all(y[:, 10] == 0)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("scale", [1e-40, 1e-30, 1e-6, 1e6, 1e15, 1e29])
def test_x_magnitudes(hq, fmt, scale):
    """x far from N(0, 1), up to the header's |x| < 2^100 (1e29) and down into
    fp32 subnormals (1e-40): every decode reads x as stored, and tiny x falls
    back on the tolerance's absolute term."""
    rows, cols = 300, 2048
    g = synthetic.rng(90)
    blocks = quant(fmt, synthetic.weights(g, rows, cols))
    for n_vec in (1, 2, 3, 4, 8):
        x = (synthetic.activations(g, n_vec, cols).astype(np.float64) * scale).astype(np.float32)
        y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
        y = gpu_matvec(hq, fmt, blocks, x, rows, cols)
        assert np.all(np.isfinite(y))
        assert_within(y, y_ref, T, f"{fmt} x*{scale:g} n_vec={n_vec}")


def _outlier_x(g, outlier_cols, n_vec, cols, kind):
    """x for sparse outlier blocks.  "tiny": 1 everywhere except +-1e-4 at the
    outlier columns, so sum_j |w x| is 1e-4 * |w| per block against
    sum_j |x| of about 31; "neg": the same with alternating +-1 elsewhere;
    "mean": N(20, 1), a large common mean."""
    if kind == "mean":
        return (g.standard_normal((n_vec, cols)) + 20.0).astype(np.float32)
    x = np.ones((n_vec, cols), np.float32)
    if kind == "neg":
        x[:, 1::2] = -1
    x[:, outlier_cols] = np.float32(1e-4) * np.where(
        g.integers(0, 2, size=(n_vec, outlier_cols.size)) == 0, -1, 1).astype(np.float32)
    return x


# (rows, cols): many row tiles, few row tiles (K split over a cluster), the
# plain-load kernel (cols % 256 != 0), a long row
OUTLIER_SHAPES = [(1000, 4096), (40, 4096), (100, 992), (64, 14336)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", OUTLIER_SHAPES)
@pytest.mark.parametrize("kind", ["tiny", "neg", "mean"])
def test_sparse_outlier_blocks(hq, fmt, rows, cols, kind):
    """Blocks of one +-outlier and 31 zeros (Q8_0: q = +-127 and 0; Q4_0: the
    outlier at n = 0, the zeros at n = 8), with x chosen so that
    sum_j |w x| is small against sum_j |x|.  A decode that carries the quant
    offset (q + 128, or the nibble n) through its products rounds relative to
    128 |x| (or 8 |x|) and fails here; the bound has to hold relative to
    |w x|, at every n_vec."""
    g = synthetic.rng(4200 + rows + cols)
    W, oc = synthetic.sparse_outlier_weights(g, rows, cols)
    blocks = quant(fmt, W)
    Wd = oracle.dequant(fmt, blocks, rows, cols)            # the zeros decode to exact zeros
    mask = np.zeros((rows, cols), bool)
    mask[:, oc] = True
    assert np.all(Wd[~mask] == 0) and np.all(np.abs(Wd[mask]) > 0.99)
    for n_vec in range(1, 9):
        x = _outlier_x(g, oc, n_vec, cols, kind)
        y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
        y = gpu_matvec(hq, fmt, blocks, x, rows, cols)
        assert_within(y, y_ref, T, f"{fmt} {rows}x{cols} {kind} n_vec={n_vec}")


@pytest.mark.parametrize("n_vec", [1, 2, 4, 8])
def test_sparse_outlier_moe(hq, n_vec):
    """The expert-indexed kernel (groups of one and of several tokens) on
    sparse outlier experts, x = 1 except +-1e-4 at the outlier columns."""
    n_experts, n_active, rows, cols = 16, 4, 96, 2048
    g = synthetic.rng(4400 + n_vec)
    W, oc = synthetic.sparse_outlier_weights(g, n_experts * rows, cols)
    bank = quant("q8_0", W)
    ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    x = _outlier_x(g, oc, n_vec, cols, "tiny")
    y_ref, T = oracle.moe_matvec_q8_0(bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    y = torch.full((n_vec, n_active, rows), float("nan"), dtype=torch.float32, device="cuda")
    hq.hq_moe_matvec_q8_0(dev(bank), dev(ids), dev(x), 0, y, n_experts, n_active, rows, cols, n_vec)
    torch.cuda.synchronize()
    assert_within(y.cpu().numpy(), y_ref, T, f"MoE sparse outliers n_vec={n_vec}")


def test_deterministic_and_stream(hq):
    rows, cols = 4096, 4096
    g = synthetic.rng(79)
    blocks = quant("q8_0", synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, 2, cols)
    s = torch.cuda.Stream()
    y1 = gpu_matvec(hq, "q8_0", blocks, x, rows, cols)
    with torch.cuda.stream(s):
        y2 = gpu_matvec(hq, "q8_0", blocks, x, rows, cols, stream=s)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def _sampled_rows(rows, n=24, width=5):
    starts = np.linspace(0, rows - width, n).astype(int)
    return [(int(s), int(s) + width) for s in starts]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", [(28672, 4096), (6144, 4096), (4096, 4096), (14336, 4096),
                                       (4096, 14336), (1024, 4096)])
def test_full_size_8b_shapes_sampled(hq, fmt, rows, cols):
    """The 8B-dense decode shapes at full size -- the fused gate|up and q|k|v
    and o, down of the bench's decode token, and the unfused gate, k -- in the
    bench's launch configuration; the oracle computes sampled rows one range
    at a time."""
    g = synthetic.rng(synthetic.SEED_BASE + 2)
    W = synthetic.weights(g, rows, cols)
    blocks = quant(fmt, W)
    del W
    for n_vec in (1, 2, 4, 8):
        x = synthetic.activations(g, n_vec, cols)
        y = gpu_matvec(hq, fmt, blocks, x, rows, cols)
        assert np.all(np.isfinite(y))
        for lo, hi in _sampled_rows(rows):
            y_ref, T = oracle.matvec_rows(fmt, blocks, x, rows, cols, lo, hi)
            assert_within(y[:, lo:hi], y_ref, T, f"{fmt} {rows}x{cols} n_vec={n_vec} rows {lo}:{hi}")


@pytest.mark.parametrize("fmt,rows,cols", [("q8_0", 151936, 1024), ("q8_0", 128256, 4096),
                                           ("q4_0", 128256, 4096)])
def test_full_size_lm_heads_sampled(hq, fmt, rows, cols):
    """The tied Qwen3-0.6B lm_head (151936 x 1024) and the 8B lm_head
    (128256 x 4096: 558 MB of Q8_0, 296 MB of Q4_0), n_vec = 1, sampled rows."""
    g = synthetic.rng(synthetic.SEED_BASE + 7)
    blocks = np.empty((rows, cols // 32 * (34 if fmt == "q8_0" else 18)), np.uint8)
    step = 8192
    for r0 in range(0, rows, step):                        # quantize in slabs to bound host memory
        r1 = min(rows, r0 + step)
        blocks[r0:r1] = quant(fmt, synthetic.weights(g, r1 - r0, cols))
    x = synthetic.activations(g, 1, cols)
    y = gpu_matvec(hq, fmt, blocks, x, rows, cols)
    f = hq.hq_device_fault()
    assert f == 0, f"{rows}x{cols}: fault word {f:#x} ({hq.hq_last_error()})"
    for lo, hi in _sampled_rows(rows, n=40):
        y_ref, T = oracle.matvec_rows(fmt, blocks, x, rows, cols, lo, hi)
        assert_within(y[:, lo:hi], y_ref, T, f"{fmt} lm_head {rows}x{cols} rows {lo}:{hi}")


@pytest.mark.parametrize("rows,cols", sorted({(r, c) for (_, r, c) in
                                              synthetic.QWEN3_0_6B_LAYER + synthetic.fuse_same_input(synthetic.QWEN3_0_6B_LAYER)}))
def test_qwen3_0_6b_layer_shapes_full(hq, rows, cols):
    """Every Qwen3-0.6B-shaped decode matvec (unfused and with q|k|v, gate|up
    row-fused), Q8_0, every output checked, n_vec 1, 2, 4 and 8 (the short-row
    K-split launches take eight consumer warps from two vectors on)."""
    g = synthetic.rng(synthetic.SEED_BASE + 1)
    blocks = quant("q8_0", synthetic.weights(g, rows, cols))
    for n_vec in (1, 2, 4, 8):
        x = synthetic.activations(g, n_vec, cols)
        y_ref, T = oracle.matvec("q8_0", blocks, x, rows, cols)
        y = gpu_matvec(hq, "q8_0", blocks, x, rows, cols)
        assert_within(y, y_ref, T, f"qwen3 {rows}x{cols} n_vec={n_vec}")


# ---------------------------------------------------------------- int8 requant

@pytest.mark.parametrize("rows,cols", [(1024, 3072), (3072, 1024), (77, 100), (40, 4), (300, 640),
                                       (50, 200), (33, 128)])
def test_int8_requant_bit_exact(hq, rows, cols):
    g = synthetic.rng(2000 + rows + cols)
    W = synthetic.weights(g, rows, cols)
    x = synthetic.activations(g, 8, cols)
    Wq, xq, mult, shift = oracle.int8_workload(W, x)
    for n_vec in (1, 2, 3, 4, 8):
        y_ref, _ = oracle.matvec_i8_requant(Wq, xq[:n_vec], mult, shift)
        y = torch.full((n_vec, rows), 99, dtype=torch.int8, device="cuda")
        hq.hq_matvec_i8_requant(dev(Wq), dev(xq[:n_vec]), dev(mult), dev(shift), y, rows, cols, n_vec)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), y_ref), f"int8 {rows}x{cols} n_vec={n_vec}"


def test_int8_extreme_weights_bit_exact(hq):
    """All +-127 weights and activations: the largest accumulators the path can form."""
    rows, cols = 64, 3072
    g = np.random.Generator(np.random.PCG64(5))
    Wq = np.where(g.random((rows, cols)) < 0.5, -127, 127).astype(np.int8)
    Wq[0] = 127
    xq = np.full((2, cols), 127, np.int8)
    xq[1] = -127
    mult = g.integers(2 ** 30, 2 ** 31 - 1, size=rows, dtype=np.int64).astype(np.int32)
    shift = g.integers(0, 32, size=rows).astype(np.int32)
    y_ref, _ = oracle.matvec_i8_requant(Wq, xq, mult, shift)
    y = torch.empty((2, rows), dtype=torch.int8, device="cuda")
    hq.hq_matvec_i8_requant(dev(Wq), dev(xq), dev(mult), dev(shift), y, rows, cols, 2)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), y_ref)


def test_requant_epilogue_edge_values(hq):
    I32_MIN, I32_MAX = -(2 ** 31), 2 ** 31 - 1
    g = np.random.Generator(np.random.PCG64(6))
    acc = np.concatenate([np.array([I32_MIN, I32_MIN + 1, -1, 0, 1, I32_MAX - 1, I32_MAX,
                                    2 ** 30, -(2 ** 30), -(2 ** 30) - 1], np.int64),
                          g.integers(I32_MIN, I32_MAX, 50000, endpoint=True, dtype=np.int64)]).astype(np.int32)
    rows = 64
    mult = g.integers(I32_MIN, I32_MAX, rows, endpoint=True, dtype=np.int64).astype(np.int32)
    mult[:4] = [I32_MIN, I32_MAX, 0, 1]
    shift = g.integers(0, 32, rows).astype(np.int32)
    shift[:3] = [0, 31, 1]
    y = torch.empty(acc.size, dtype=torch.int8, device="cuda")
    hq.hq_requant_i32_debug(dev(acc), dev(mult), dev(shift), y, acc.size, rows)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.requant_array(acc, mult, shift))


# ---------------------------------------------------------------- MoE

def _moe_case(n_experts, n_active, rows, cols, n_vec, seed, x_per_slot, ids=None):
    g = synthetic.rng(seed)
    bank = np.empty((n_experts * rows, cols // 32 * 34), np.uint8)
    for e in range(n_experts):
        bank[e * rows:(e + 1) * rows] = oracle.quantize_q8_0(synthetic.weights(g, rows, cols))
    if ids is None:
        ids = synthetic.expert_ids(g, n_vec, n_active, n_experts)
    x = synthetic.activations(g, n_vec * (n_active if x_per_slot else 1), cols)
    return bank, ids, x


def gpu_moe(hq, bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec):
    y = torch.full((n_vec, n_active, rows), -7.0, dtype=torch.float32, device="cuda")
    hq.hq_moe_matvec_q8_0(dev(bank), dev(ids), dev(x), int(x_per_slot), y, n_experts, n_active, rows, cols, n_vec)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("x_per_slot,rows,cols", [(False, 768, 2048), (True, 2048, 768), (False, 1536, 2048)])
@pytest.mark.parametrize("n_vec", [1, 4, 8])
def test_moe_128_experts_top8(hq, x_per_slot, rows, cols, n_vec):
    """128 experts, top-8: gate (768x2048, x shared by the slots), down
    (2048x768, x per slot) and the row-fused gate|up (1536x2048) the bench
    launches."""
    n_experts, n_active = 128, 8
    bank, ids, x = _moe_case(n_experts, n_active, rows, cols, n_vec, 3000 + n_vec, x_per_slot)
    y = gpu_moe(hq, bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    y_ref, T = oracle.moe_matvec_q8_0(bank, ids, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
    assert_within(y, y_ref, T, f"moe n_vec={n_vec} x_per_slot={x_per_slot}")


def test_moe_shared_and_duplicate_experts(hq):
    n_experts, n_active, rows, cols, n_vec = 6, 3, 40, 256, 5
    ids = np.array([[0, 1, 2], [2, 1, 0], [5, 5, 5], [2, 2, 3], [4, 0, 2]], dtype=np.int32)
    for x_per_slot in (False, True):
        bank, ids_, x = _moe_case(n_experts, n_active, rows, cols, n_vec, 4000, x_per_slot, ids=ids)
        y = gpu_moe(hq, bank, ids_, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
        y_ref, T = oracle.moe_matvec_q8_0(bank, ids_, x, x_per_slot, n_experts, n_active, rows, cols, n_vec)
        assert_within(y, y_ref, T, f"moe duplicates x_per_slot={x_per_slot}")


def test_moe_all_same_expert_equals_dense(hq):
    """Every slot routed to one expert: each slot equals the dense matvec of that
    expert (to the float tolerance; the grouped kernel sums in another order),
    and two calls give bit-identical outputs."""
    n_experts, n_active, rows, cols, n_vec = 4, 2, 100, 512, 3
    bank, _, x = _moe_case(n_experts, n_active, rows, cols, n_vec, 4001, False)
    ids = np.full((n_vec, n_active), 3, np.int32)
    y = gpu_moe(hq, bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    y_again = gpu_moe(hq, bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    assert np.array_equal(y.view(np.uint32), y_again.view(np.uint32))
    expert = bank[3 * rows:4 * rows]
    y_dense = gpu_matvec(hq, "q8_0", expert, x, rows, cols)
    y_ref, T = oracle.matvec("q8_0", expert, x, rows, cols)
    assert_within(y_dense, y_ref, T, "dense expert 3")
    for k in range(n_active):
        assert_within(y[:, k], y_ref, T, f"moe slot {k}")


@pytest.mark.parametrize("flags", [0, 1])
def test_moe_invalid_id_sets_fault_and_nan(hq, flags):
    """An out-of-range expert id: NaN rows for its slots, the fault bit, exact
    neighbours -- also when the launch reads its ids before waiting for the
    previous kernel (HQ_MOE_IDS_READY), where the NaN rows must still be
    written only after that wait."""
    n_experts, n_active, rows, cols, n_vec = 4, 2, 64, 256, 2
    bank, _, x = _moe_case(n_experts, n_active, rows, cols, n_vec, 4002, False)
    ids = np.array([[1, 9], [3, -1]], dtype=np.int32)
    if flags:
        yd = torch.full((n_vec, n_active, rows), 7.0, dtype=torch.float32, device="cuda")
        hq.hq_moe_matvec_q8_0_ex(dev(bank), dev(ids), dev(x), 0, None, yd, n_experts, n_active, rows, cols,
                                 n_vec, hq.HQ_MOE_EPI_NONE, hq.HQ_MOE_IDS_READY)
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
    else:
        y = gpu_moe(hq, bank, ids, x, False, n_experts, n_active, rows, cols, n_vec)
    assert hq.hq_device_fault() == hq.HQ_FAULT_EXPERT_ID
    assert np.all(np.isnan(y[0, 1])) and np.all(np.isnan(y[1, 1]))
    ok = np.array([[1, 0], [3, 0]], dtype=np.int32)
    y_ref, T = oracle.moe_matvec_q8_0(bank, ok, x, False, n_experts, n_active, rows, cols, n_vec)
    assert_within(y[:, 0], y_ref[:, 0], T[:, 0], "valid slots beside invalid ones")
    assert hq.hq_device_fault() == 0


# ---------------------------------------------------------------- launch-policy boundaries

@pytest.mark.parametrize("rows,cols,n_vec", [
    (97, 3072, 1),      # Q8_0 short rows (four consumer warps), ragged last tile
    (97, 3328, 1),      # one K chunk past the short-row limit: two warps, K split over a cluster
    (1000, 1024, 1),    # short rows, many tiles
    (4100, 4096, 3),    # column-split stages (64-row tiles, two rows per lane), ragged last tile
    (14593, 512, 2),    # two vectors: column-split stages without a K split, ragged last tile
    (97, 3328, 2),      # two vectors, K split over a cluster
    (4100, 4096, 6),
    (333, 14336, 7),    # column-split stages with a K split over a cluster
    (4100, 4096, 3),    # eight consumer warps of one block each (K split kept), ragged last tile
    (1000, 2048, 5),    # eight warps on short rows, clusters of 8
    (300, 14336, 4),    # eight warps, clusters of 8 over long rows, ragged last tile
    (1024, 3072, 8),    # eight warps at eight vectors (short rows)
])
def test_q8_0_launch_policy_boundaries(hq, rows, cols, n_vec):
    """Each Q8_0 launch policy at and around its switch point (rows of at most
    3072 columns at one vector; column-split stages at two or more vectors,
    with four or eight consumer warps), element by element against the oracle."""
    g = synthetic.rng(4242 + rows + cols + n_vec)
    blocks = quant("q8_0", synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, n_vec, cols)
    y_ref, T = oracle.matvec("q8_0", blocks, x, rows, cols)
    y = gpu_matvec(hq, "q8_0", blocks, x, rows, cols)
    assert_within(y, y_ref, T, f"q8_0 {rows}x{cols} n_vec={n_vec}")


@pytest.mark.parametrize("fmt,rows,cols,n_vec", [
    ("q4_0", 4100, 4096, 1), ("q4_0", 333, 14336, 1), ("q4_0", 4100, 4096, 5),
    # one vector: K split over clusters up to 228 tiles of 64 rows on 152 SMs,
    # column-split stages from 229 tiles on (ragged last tiles both sides)
    ("q4_0", 14592, 512, 1), ("q4_0", 14593, 512, 1), ("q4_0", 20000, 768, 1),
    ("q4_k", 14592, 512, 1), ("q4_k", 14593, 512, 1),
    # two vectors: column-split stages without a K split too
    ("q4_0", 14592, 512, 2), ("q4_0", 14593, 512, 2), ("q4_k", 14592, 512, 2), ("q4_k", 14593, 512, 2),
    # four and five vectors: two rows per lane, eight warps on K-split launches
    ("q4_0", 300, 14336, 4), ("q4_0", 1000, 2048, 5), ("q4_0", 4100, 4096, 6), ("q4_k", 333, 14336, 4)])
def test_nibble_launch_policy_boundaries(hq, fmt, rows, cols, n_vec):
    """Q4_0 / Q4_K at one vector (four consumer warps: one stage per warp with a
    K split, column-split stages without) and at five vectors (three CTAs per
    SM), ragged last tiles, against the oracle."""
    g = synthetic.rng(5151 + rows + cols + n_vec)
    blocks = oracle.quantize(fmt, synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, n_vec, cols)
    y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
    n = x.shape[0]
    y = torch.full((n, rows), float("nan"), dtype=torch.float32, device="cuda")
    fn = {"q4_0": hq.hq_matvec_q4_0, "q4_k": hq.hq_matvec_q4_k}[fmt]
    fn(dev(blocks), dev(x), y, rows, cols, n)
    torch.cuda.synchronize()
    assert_within(y.cpu().numpy(), y_ref, T, f"{fmt} {rows}x{cols} n_vec={n_vec}")
