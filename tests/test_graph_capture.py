"""Every entry point called for the first time inside CUDA-graph stream capture.

A serving loop captures its step into a CUDA graph, often before any kernel
of the library has run. In a fresh process (nothing set up yet: no kernel
attribute raised, no occupancy figure cached, no tensor map encoded, the
library's own MoE workspace never looked up), each call below is first made
while torch captures a graph on its stream, in torch's default (global)
capture mode. The graph is replayed twice; then the same calls run eagerly on
fresh outputs, and every output must match the replayed one bit for bit (the
kernels are deterministic). Only the load-time repack runs before capture."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import gemm_q4_q8_gb300 as qg
import synth
from gemm_q4_q8_gb300 import build
build.build()

def dq(t, q, s):
    blocks = torch.from_numpy(synth.to_gguf_blocks(t, q, s)).cuda()
    qd = torch.empty(q.shape, dtype=torch.uint8, device="cuda")
    sd = torch.empty(s.shape, dtype=torch.int16, device="cuda")
    qg.qrepack(t, blocks, q.shape[0], s.shape[1] * 32, qd, sd)
    return qd, sd

def f16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)

def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()

g = synth.rng(77)
calls = []   # (name, fn(outputs) -> None, output factory)

# GEMV: tensor cores with a K-split cluster and a residual; CUDA cores at 8 columns
for name, t, rows, k, nc, res in (("gemv q4 5120x5120 c1 y0", synth.Q4_0, 5120, 5120, 1, True),
                                  ("gemv q8 2048x2048 c8", synth.Q8_0, 2048, 2048, 8, False),
                                  ("cols q4 1040x1280 c16 y0", synth.Q4_0, 1040, 1280, 16, True)):
    q, s = synth.draw_matrix(g, t, rows, k)
    qd, sd = dq(t, q, s)
    x = f16(synth.draw_x(g, nc, k))
    y0 = dev(synth.draw_y0(g, nc, rows)) if res else None
    def fn(out, t=t, qd=qd, sd=sd, x=x, y0=y0, nc=nc):
        if nc > 8:
            qg.qgemm_cols(t, qd, sd, x, out[0], y0)
        else:
            (qg.qgemv_q4_0 if t == synth.Q4_0 else qg.qgemv_q8_0)(qd, sd, x, out[0], y0)
    calls.append((name, fn, lambda nc=nc, rows=rows: [torch.empty((nc, rows), device="cuda")]))

# fused gate/up: tensor cores (16 columns) and CUDA cores (1 column)
for name, t, rows, k, nc in (("gate/up q4 1000x2048 c16", synth.Q4_0, 1000, 2048, 16),
                             ("gate/up q8 300x1056 c1", synth.Q8_0, 300, 1056, 1)):
    a = dq(t, *synth.draw_matrix(g, t, rows, k))
    b = dq(t, *synth.draw_matrix(g, t, rows, k))
    x = f16(synth.draw_x(g, nc, k))
    def fn(out, t=t, a=a, b=b, x=x):
        qg.qffn_gate_up_silu(t, a[0], a[1], b[0], b[1], x, out[0])
    calls.append((name, fn, lambda nc=nc, rows=rows: [torch.empty((nc, rows), dtype=torch.float16,
                                                                   device="cuda")]))

# MoE: staged down kernel (2 columns), register down kernel (8), library workspace (1)
for name, nc, noalloc in (("moe c2", 2, False), ("moe c8", 8, False), ("moe noalloc c1", 1, True)):
    c = synth.moe_case(synth.Q8_0, 24, 512, 1024, nc, topk=8, shared=True, residual=True, seed=nc)
    t = c["qtype"]
    m = {}
    for a_, b_ in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
        m[a_], m[b_] = dq(t, c[a_], c[b_])
    sh = {}
    for a_, b_ in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
        sh[a_], sh[b_] = dq(t, c["shared"][a_], c["shared"][b_])
    ids, rw, x, y0 = dev(c["ids"].astype(np.int32)), dev(c["rw"]), f16(c["x"]), dev(c["y0"])
    ws = torch.empty(qg.qmoe_workspace_bytes(24, 512, 1024, nc, 8), dtype=torch.uint8, device="cuda")
    def fn(out, t=t, m=m, sh=sh, ids=ids, rw=rw, x=x, y0=y0, ws=ws, noalloc=noalloc):
        args = (t, m["qg"], m["sg"], m["qu"], m["su"], m["qd"], m["sd"], 24, 512, 1024, ids, rw, x,
                out[0])
        if noalloc:
            qg.qmoe_experts_noalloc(*args, y0=y0, shared=sh, err_flag=out[1], uniq_ids_out=out[2])
        else:
            qg.qmoe_experts(*args, ws, y0=y0, shared=sh, err_flag=out[1], uniq_ids_out=out[2])
    def mk(nc=nc):
        return [torch.empty((nc, 1024), device="cuda"), torch.zeros(1, dtype=torch.int32, device="cuda"),
                torch.empty(nc * 8, dtype=torch.int32, device="cuda")]
    calls.append((name, fn, mk))

# router, argmax, top-k
w = dev((g.standard_normal((256, 2048)) * 0.02).astype(np.float32))
xr = f16(synth.draw_x(g, 8, 2048))
calls.append(("router 256x2048 c8", lambda out: qg.qmoe_router(w, xr, 8, out[0], out[1], logits_out=out[2]),
              lambda: [torch.empty((8, 8), dtype=torch.int32, device="cuda"),
                       torch.empty((8, 8), device="cuda"), torch.empty((8, 256), device="cuda")]))
lg = dev(g.standard_normal((2, 248320)).astype(np.float32))
calls.append(("argmax 248320 c2", lambda out: qg.qargmax_f32(lg, out[0], out[1]),
              lambda: [torch.empty(2, dtype=torch.int32, device="cuda"), torch.empty(2, device="cuda")]))
calls.append(("top-40 248320 c2", lambda out: qg.qtopk_f32(lg, 40, out[0], out[1]),
              lambda: [torch.empty((2, 40), dtype=torch.int32, device="cuda"),
                       torch.empty((2, 40), device="cuda")]))
torch.cuda.synchronize()

launches_before = qg.qg_kernel_launches()
outs_g = [mk() for _, _, mk in calls]
torch.cuda.synchronize()
graph = torch.cuda.CUDAGraph()
with torch.cuda.graph(graph):
    for (name, fn, _), out in zip(calls, outs_g):
        fn(out)
for _ in range(2):
    graph.replay()
torch.cuda.synchronize()
outs_e = [mk() for _, _, mk in calls]
for (name, fn, _), out in zip(calls, outs_e):
    fn(out)
torch.cuda.synchronize()
for (name, _, _), og, oe in zip(calls, outs_g, outs_e):
    for a, b in zip(og, oe):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name
    if og[0].is_floating_point():
        assert torch.isfinite(og[0].float()).all(), name
assert qg.qg_device_error() == 0
print("GRAPH_OK", len(calls), qg.qg_kernel_launches() - launches_before)
'''


def test_first_calls_inside_graph_capture_fresh_process():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    code = "ROOT = " + repr(ROOT) + "\n" + WORKER
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, (r.stdout[-2000:], r.stderr[-3000:])
    assert "GRAPH_OK" in r.stdout
