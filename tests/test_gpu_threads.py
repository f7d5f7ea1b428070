"""The library's first calls made from several host threads at once.  The
per-device set-up (device attributes, the fault word's and the scratch's
device addresses, kernel attributes) happens lazily on the first call; eight
threads start their first matvec together, each on its own stream, in a fresh
process, and every result must match the oracle.  Run in a subprocess so that
the calls really are the process's first."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import oracle
import quantized_weight_matvec_hq_gb300 as hq
from quantized_weight_matvec_hq_gb300 import synthetic

N = 8
g = synthetic.rng(7)
cases = []
for i in range(N):
    fmt = "q8_0" if i % 2 == 0 else "q4_0"
    rows, cols, n_vec = 300 + 17 * i, 2048 if i < 4 else 4096, 1 + i % 3
    blocks = (oracle.quantize_q8_0 if fmt == "q8_0" else oracle.quantize_q4_0)(synthetic.weights(g, rows, cols))
    x = synthetic.activations(g, n_vec, cols)
    cases.append((fmt, rows, cols, n_vec, blocks, x))
dev = [(torch.from_numpy(b).cuda(), torch.from_numpy(x).cuda(), torch.empty((n, r), device="cuda"))
       for (f, r, c, n, b, x) in cases]
streams = [torch.cuda.Stream() for _ in range(N)]
torch.cuda.synchronize()
barrier = threading.Barrier(N)
errors = []

def run(i):
    try:
        torch.cuda.set_device(0)
        fmt, rows, cols, n_vec, _, _ = cases[i]
        W, x, y = dev[i]
        fn = hq.hq_matvec_q8_0 if fmt == "q8_0" else hq.hq_matvec_q4_0
        barrier.wait()
        fn(W, x, y, rows, cols, n_vec, stream=streams[i])
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=run, args=(i,)) for i in range(N)]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
for (fmt, rows, cols, n_vec, blocks, x), (_, _, y) in zip(cases, dev):
    y_ref, T = oracle.matvec(fmt, blocks, x, rows, cols)
    excess = np.abs(y.cpu().numpy().astype(np.float64) - y_ref) - (1e-3 * T + 1e-5)
    assert np.all(excess <= 0), (fmt, rows, cols, n_vec, float(excess.max()))
assert hq.hq_device_fault() == 0
print("threads-ok")
"""


def test_first_calls_from_eight_threads():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads-ok" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
