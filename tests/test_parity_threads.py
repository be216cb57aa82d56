"""Several host threads calling the library at once, in a fresh process.

Each thread drives its own CUDA stream through shapes that use the same
kernels with different dynamic shared-memory sizes (tensor-core plans with
different stage counts, CUDA-core GEMVs with different x chunks), starting from
a process where no kernel has been set up yet, so the per-device set-up runs
concurrently. Every output must equal, bit for bit, the output of the same call
made alone on one thread (the kernels are deterministic).
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import sys, threading
import numpy as np
import torch
sys.path.insert(0, ROOT)
import gemm_q4_q8_gb300 as qg
import synth
from gemm_q4_q8_gb300 import build
build.build()

# (qtype, rows, k, ncols, residual): tensor-core plans of different stage
# counts, CUDA-core GEMVs of different x chunks, a 16-column prefill
SHAPES = [(synth.Q4_0, 5120, 5120, 1, True), (synth.Q4_0, 17408, 5120, 8, False),
          (synth.Q8_0, 2048, 2048, 1, False), (synth.Q8_0, 2048, 2048, 8, False),
          (synth.Q4_0, 1040, 1280, 16, True), (synth.Q8_0, 96, 65536, 3, True)]
cases = []
for i, (t, rows, k, nc, res) in enumerate(SHAPES):
    c = synth.gemv_case(t, rows, k, nc, residual=res, seed=60 + i)
    blocks = torch.from_numpy(synth.to_gguf_blocks(t, c["q"], c["scl"])).cuda()
    q = torch.empty(c["q"].shape, dtype=torch.uint8, device="cuda")
    s = torch.empty(c["scl"].shape, dtype=torch.int16, device="cuda")
    qg.qrepack(t, blocks, rows, k, q, s)
    x = torch.from_numpy(c["x"].view(np.int16)).cuda().view(torch.float16)
    y0 = torch.from_numpy(c["y0"]).cuda() if res else None
    cases.append((t, q, s, x, y0, nc, rows))
torch.cuda.synchronize()

def run(case, stream):
    t, q, s, x, y0, nc, rows = case
    y = torch.empty((nc, rows), dtype=torch.float32, device="cuda")
    if nc > 8:
        qg.qgemm_cols(t, q, s, x, y, y0, stream)
    else:
        (qg.qgemv_q4_0 if t == synth.Q4_0 else qg.qgemv_q8_0)(q, s, x, y, y0, stream)
    return y

NT, REPS = 6, 8
results = [[] for _ in range(NT)]
errors = []
def worker(tid):
    try:
        stream = torch.cuda.Stream()
        order = [(tid + j) % len(cases) for j in range(len(cases))]
        for _ in range(REPS):
            for ci in order:
                results[tid].append((ci, run(cases[ci], stream)))
        stream.synchronize()
    except Exception as e:  # reported below
        errors.append(repr(e))
threads = [threading.Thread(target=worker, args=(i,)) for i in range(NT)]
for th in threads:
    th.start()
for th in threads:
    th.join()
torch.cuda.synchronize()
assert not errors, errors
ref = []
st = torch.cuda.Stream()
for case in cases:
    ref.append(run(case, st))
torch.cuda.synchronize()
n = 0
for tid in range(NT):
    for ci, y in results[tid]:
        assert torch.equal(y, ref[ci]), (tid, ci)
        n += 1
assert qg.qg_device_error() == 0
print("THREADS_OK", n)
'''


def test_concurrent_host_threads_fresh_process():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    code = "ROOT = " + repr(ROOT) + "\n" + WORKER
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    assert "THREADS_OK" in r.stdout
