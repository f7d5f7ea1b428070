"""GPU parity of the Q4_K path (hq_quantize_q4_k, hq_matvec_q4_k) against the
CPU oracle ("One Native Stack ...", sections "The Unified Quant Core" and
"Ported Versus Novel": ggml's Q4_K super-block, 256 weights in 144 bytes).

Bar: the GPU encoder's bytes bit-exact against the oracle's; the matvec within
|y - y_ref| <= 1e-3 * sum_j |w_deq x_j| + 1e-5 per output, the same bar as the
symmetric formats: every weight d*sc*q - dmin*m is formed in fp32 before it
multiplies x, so sub-blocks whose weights nearly cancel (d*sc*q close to
dmin*m) meet it too."""
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


def gpu_q4_k(hq, blocks, x, rows, cols):
    n_vec = x.shape[0]
    y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
    hq.hq_matvec_q4_k(dev(blocks), dev(x), y, rows, cols, n_vec)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def special_weights(rows, cols, seed):
    g = synthetic.rng(seed)
    W = synthetic.weights(g, rows, cols)
    W[::5] *= np.float32(40.0)
    W[1::7, :32] = np.abs(W[1::7, :32]) + 0.01
    W[2::7, 32:64] = -np.abs(W[2::7, 32:64]) - 0.01
    W[3::7, 64:96] = 0
    W[4::7, :] = 0
    W[5::7, 100 % cols] = 3.0
    return W


@pytest.mark.parametrize("rows,cols", [(1, 256), (64, 512), (333, 1024), (40, 4096)])
def test_quantizer_bytes_bit_exact(hq, rows, cols):
    W = special_weights(rows, cols, 800 + rows)
    out = torch.empty((rows, cols // 256 * 144), dtype=torch.uint8, device="cuda")
    hq.hq_quantize_q4_k(dev(W), out, rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.quantize_q4_k(W))


@pytest.mark.parametrize("rows,cols", [(1, 256), (31, 256), (96, 512), (200, 1024), (1000, 2048), (333, 2816),
                                       (2048, 768), (64, 14336)])
def test_matvec_parity(hq, rows, cols):
    g = synthetic.rng(900 + rows + cols)
    blocks = oracle.quantize_q4_k(special_weights(rows, cols, 901 + rows))
    for n_vec in range(1, 9):
        x = synthetic.activations(g, n_vec, cols)
        y_ref, T = oracle.matvec("q4_k", blocks, x, rows, cols)
        assert_within(gpu_q4_k(hq, blocks, x, rows, cols), y_ref, T, f"{rows}x{cols} n_vec={n_vec}")


def _cancelling_blocks(rows, cols, seed):
    """Super-blocks whose weights are mostly exactly zero through cancellation:
    d = dmin, sc_j = m_j, and q = 1 gives w = d*sc - dmin*m = 0; one element per
    sub-block gets q = 2 (w = d*sc).  Large d and scales make each term big
    while the weight is 0, which only an exact per-weight decode survives."""
    g = np.random.Generator(np.random.PCG64(seed))
    nsb = cols // 256
    b = np.zeros((rows, nsb, 144), np.uint8)
    d = np.float16(g.uniform(0.5, 8.0)).view(np.uint16)
    for r in range(rows):
        for s in range(nsb):
            sc = g.integers(1, 64, size=8)
            b[r, s, 0:2] = [int(d) & 0xFF, int(d) >> 8]
            b[r, s, 2:4] = [int(d) & 0xFF, int(d) >> 8]
            for j in range(4):
                b[r, s, 4 + j] = sc[j] | ((sc[j + 4] >> 4) << 6)
                b[r, s, 8 + j] = sc[j] | ((sc[j + 4] >> 4) << 6)
                b[r, s, 12 + j] = (sc[j + 4] & 15) | ((sc[j + 4] & 15) << 4)
            q = np.ones(256, np.int64)
            q[np.arange(8) * 32 + g.integers(0, 32, size=8)] = 2
            for gq in range(4):
                b[r, s, 16 + 32 * gq:48 + 32 * gq] = q[64 * gq:64 * gq + 32] | (q[64 * gq + 32:64 * gq + 64] << 4)
    return b.reshape(rows, nsb * 144)


@pytest.mark.parametrize("n_vec", [1, 2, 4, 8])
def test_cancelling_weights(hq, n_vec):
    rows, cols = 96, 1024
    blocks = _cancelling_blocks(rows, cols, 1000 + n_vec)
    Wd = oracle.dequant("q4_k", blocks, rows, cols)
    assert np.mean(Wd == 0) > 0.9
    g = synthetic.rng(1100 + n_vec)
    x = synthetic.activations(g, n_vec, cols) * np.float32(1e4)
    x[:, Wd[0] != 0] *= np.float32(1e-8)              # tiny x where row 0's weights are nonzero
    y_ref, T = oracle.matvec("q4_k", blocks, x, rows, cols)
    assert_within(gpu_q4_k(hq, blocks, x, rows, cols), y_ref, T, f"cancelling n_vec={n_vec}")


@pytest.mark.parametrize("scale", [1e-30, 1e-6, 1e6, 1e15])
def test_x_magnitudes(hq, scale):
    rows, cols = 128, 1024
    g = synthetic.rng(1200)
    blocks = oracle.quantize_q4_k(synthetic.weights(g, rows, cols))
    for n_vec in (1, 3, 5, 8):
        x = (synthetic.activations(g, n_vec, cols).astype(np.float64) * scale).astype(np.float32)
        y_ref, T = oracle.matvec("q4_k", blocks, x, rows, cols)
        assert_within(gpu_q4_k(hq, blocks, x, rows, cols), y_ref, T, f"x scale {scale} n_vec={n_vec}")


def test_deterministic_and_shape_checks(hq):
    rows, cols = 4096, 4096
    g = synthetic.rng(1300)
    blocks = oracle.quantize_q4_k(synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, 1, cols)
    y1 = gpu_q4_k(hq, blocks, x, rows, cols)
    y2 = gpu_q4_k(hq, blocks, x, rows, cols)
    assert np.array_equal(y1, y2)
    W = torch.zeros((8, 9 * 18), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((1, 288), dtype=torch.float32, device="cuda")
    ys = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(hq.HQError):
        hq.hq_matvec_q4_k(W, xs, ys, 8, 288, 1)            # 288 is not a multiple of 256


def _sampled_rows(rows, n=24, width=40):
    starts = np.linspace(0, rows - width, n).astype(int)
    return [(int(s), int(s) + width) for s in starts] + [(rows - 7, rows)]


@pytest.mark.parametrize("rows,cols", [(28672, 4096), (6144, 4096), (4096, 4096), (4096, 14336), (128256, 4096)])
def test_full_size_8b_shapes_sampled(hq, rows, cols):
    """The 8B decode shapes (gate|up, q|k|v, o, down, lm_head) at full size,
    quantized on the GPU (bytes checked against the oracle's encoder on a
    slab), with the oracle on sampled row ranges at n_vec 1, 2 and 8."""
    g = synthetic.rng(synthetic.SEED_BASE + 13)
    Wt = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    step = 8192
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        Wt[r0:r1] = torch.from_numpy(synthetic.weights(g, r1 - r0, cols))
    blocks_d = torch.empty((rows, cols // 256 * 144), dtype=torch.uint8, device="cuda")
    hq.hq_quantize_q4_k(Wt, blocks_d, rows, cols)
    torch.cuda.synchronize()
    assert np.array_equal(blocks_d[:64].cpu().numpy(), oracle.quantize_q4_k(Wt[:64].cpu().numpy()))
    del Wt
    blocks = blocks_d.cpu().numpy()
    for n_vec in (1, 2, 8):
        x = synthetic.activations(g, n_vec, cols)
        y = torch.full((n_vec, rows), float("nan"), dtype=torch.float32, device="cuda")
        hq.hq_matvec_q4_k(blocks_d, dev(x), y, rows, cols, n_vec)
        torch.cuda.synchronize()
        y = y.cpu().numpy()
        assert np.all(np.isfinite(y))
        for lo, hi in _sampled_rows(rows):
            y_ref, T = oracle.matvec_rows("q4_k", blocks, x, rows, cols, lo, hi)
            assert_within(y[:, lo:hi], y_ref, T, f"{rows}x{cols} n_vec={n_vec} rows {lo}:{hi}")
