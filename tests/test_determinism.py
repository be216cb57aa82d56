"""Run-to-run bit identity under back-to-back launches.

Each call below is launched eight times in a row on one stream with no
synchronisation between them (so consecutive calls overlap through early
dependent launch and every run sees different timing), each into its own
output; all eight outputs must be identical bit for bit. The shapes are the
workload's tensor-core plans at full size (K-split clusters, one and two
n-tiles, single and dual matrices, Q4_0 and Q8_0), where a stage refilled
while a consumer still reads it, or a partial tile handed over too early, would
show up as run-to-run differences. Values are checked against the oracle by the
parity tests; here only the identity of the runs is checked."""
import numpy as np
import pytest

import synth
from helpers import dev, dev_q, dev_u16_as_f16

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q4_q8_gb300 import build
    build.build()
    import oracle
    oracle.build()


import gemm_q4_q8_gb300 as qg  # noqa: E402

REPS = 8


def _same(outs, what):
    ref = outs[0].view(torch.int32) if outs[0].dtype != torch.float16 else outs[0].view(torch.int16)
    for i, o in enumerate(outs[1:], 1):
        v = o.view(torch.int32) if o.dtype != torch.float16 else o.view(torch.int16)
        diff = int((v != ref).sum())
        assert diff == 0, f"{what}: run {i} differs from run 0 in {diff} elements"


@pytest.mark.parametrize("qtype,rows,k,ncols,residual", [
    (synth.Q4_0, 5120, 5120, 1, True),      # K-split cluster of 3, residual
    (synth.Q4_0, 17408, 5120, 8, False),    # verify twins
    (synth.Q8_0, 17408, 5120, 8, False),    # Q8_0 twins (early release)
    (synth.Q8_0, 65536, 5120, 1, False),    # LM-head plan, 65,536-row cut
    (synth.Q4_0, 5120, 17408, 16, True),    # FFN down: two n-tiles, K split
])
def test_gemm_runs_bit_identical(qtype, rows, k, ncols, residual):
    g = synth.rng(rows + k + ncols)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    dq, ds = dev_q(qtype, q, s)
    x = dev_u16_as_f16(synth.draw_x(g, ncols, k))
    y0 = dev(synth.draw_y0(g, ncols, rows)) if residual else None
    outs = [torch.empty((ncols, rows), dtype=torch.float32, device="cuda") for _ in range(REPS)]
    torch.cuda.synchronize()
    for y in outs:
        if ncols > 8:
            qg.qgemm_cols(qtype, dq, ds, x, y, y0)
        else:
            (qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0)(dq, ds, x, y, y0)
    torch.cuda.synchronize()
    _same(outs, f"{qtype} {rows}x{k} C={ncols}")


def test_in_place_down_runs_bit_identical():
    """The FFN down projection with y += W h in place, each run on a fresh copy
    of the residual (the copies are queued between the calls)."""
    g = synth.rng(99)
    q, s = synth.draw_matrix(g, synth.Q4_0, 5120, 17408)
    dq, ds = dev_q(synth.Q4_0, q, s)
    h = dev_u16_as_f16(synth.draw_x(g, 16, 17408))
    y0 = dev(synth.draw_y0(g, 16, 5120))
    outs = [torch.empty_like(y0) for _ in range(REPS)]
    torch.cuda.synchronize()
    for y in outs:
        y.copy_(y0)
        qg.qgemm_cols(synth.Q4_0, dq, ds, h, y, y)
    torch.cuda.synchronize()
    _same(outs, "in-place down 5120x17408 C=16")


@pytest.mark.parametrize("qtype,rows,k,ncols", [
    (synth.Q4_0, 17408, 5120, 16),   # the workload's fused gate/up
    (synth.Q8_0, 8192, 2048, 8),     # dual Q8_0, one n-tile
])
def test_gate_up_runs_bit_identical(qtype, rows, k, ncols):
    g = synth.rng(rows + k + ncols + 1)
    a = dev_q(qtype, *synth.draw_matrix(g, qtype, rows, k))
    b = dev_q(qtype, *synth.draw_matrix(g, qtype, rows, k))
    x = dev_u16_as_f16(synth.draw_x(g, ncols, k))
    outs = [torch.empty((ncols, rows), dtype=torch.float16, device="cuda") for _ in range(REPS)]
    torch.cuda.synchronize()
    for h in outs:
        qg.qffn_gate_up_silu(qtype, a[0], a[1], b[0], b[1], x, h)
    torch.cuda.synchronize()
    _same(outs, f"gate/up {qtype} {rows}x{k} C={ncols}")


def test_moe_runs_bit_identical():
    """The MoE layer at 1, 8 and 16 columns, eight back-to-back runs each."""
    for ncols in (1, 8, 16):
        c = synth.moe_case(synth.Q8_0, 64, 512, 2048, ncols, topk=8, shared=True, residual=True,
                           seed=ncols)
        t = c["qtype"]
        m = {}
        for a_, b_ in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
            m[a_], m[b_] = dev_q(t, c[a_], c[b_])
        sh = {}
        for a_, b_ in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
            sh[a_], sh[b_] = dev_q(t, c["shared"][a_], c["shared"][b_])
        ids, rw = dev(np.ascontiguousarray(c["ids"], np.int32)), dev(c["rw"])
        x, y0 = dev_u16_as_f16(c["x"]), dev(c["y0"])
        ws = [torch.empty(qg.qmoe_workspace_bytes(64, 512, 2048, ncols, 8), dtype=torch.uint8,
                          device="cuda") for _ in range(REPS)]
        outs = [torch.empty((ncols, 2048), dtype=torch.float32, device="cuda") for _ in range(REPS)]
        torch.cuda.synchronize()
        for y, w in zip(outs, ws):
            qg.qmoe_experts(t, m["qg"], m["sg"], m["qu"], m["su"], m["qd"], m["sd"], 64, 512, 2048,
                            ids, rw, x, y, w, y0=y0, shared=sh)
        torch.cuda.synchronize()
        _same(outs, f"MoE C={ncols}")


def test_step_graph_soak():
    """The benchmark's whole step (GEMV + residual, LM head, twins, fused
    gate/up, down with residual, MoE layer) captured in one CUDA graph and
    replayed 3,000 times; after every replay a device-side comparison of all
    its outputs with the first replay's, counted on the device (no host
    synchronisation until the end)."""
    import bench
    gs = bench.GpuStep(bench.make_workload(0), torch)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            gs.step(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gs.step(s)
    g.replay()
    torch.cuda.synchronize()
    out = gs.dout_flat[0].view(torch.int32)
    ref = out.clone()
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(3000):
        g.replay()
        bad += ((out != ref).sum() > 0).long()
    torch.cuda.synchronize()
    assert int(bad) == 0, f"{int(bad)} of 3000 replays differ from the first"
    assert qg.qg_device_error() == 0 and int(gs.m_err.item()) == 0
