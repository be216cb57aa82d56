"""Verify twins are bit-identical to single-column decode ("Architecture",
sections "Speculative decoding" and "Models without a draft block": the
batched verify kernels share the decode kernel's work shape, so every checked
column reproduces the logits of a plain decoding step exactly, and a verified
token is exactly a decoded one).

Each multi-column call is compared bit for bit, column by column, with the
1-column call on that column alone: the GEMV twins (tensor-core plan when K is
a multiple of 256, CUDA cores otherwise, including x staged in several
chunks), the residual form, the fused gate/up, the MoE layer and the router.
The values themselves are checked against the oracle by the other parity
tests."""
import numpy as np
import pytest

import synth
from helpers import dev, dev_q, dev_u16_as_f16, host

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


def gemv(qtype, qd, sd, x, y0):
    ncols, rows = x.shape[0], sd.shape[0]
    y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    fn = qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0
    fn(qd, sd, x, y, y0)
    torch.cuda.synchronize()
    return host(y)


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k", [
    (5120, 5120),     # tensor-core plan
    (2048, 2048),     # CUDA cores (small matrix)
    (17408, 5120),    # tensor-core plan, cluster split-K
    (333, 1056),      # CUDA cores (K not a multiple of 256)
    (200, 4128),      # CUDA cores, x staged in chunks for 5-8 columns
])
@pytest.mark.parametrize("residual", [False, True])
def test_gemv_twins_bit_identical(qtype, rows, k, residual):
    g = synth.rng(rows + k + qtype)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    qd, sd = dev_q(qtype, q, s)
    x8 = synth.draw_x(g, 8, k)
    y08 = synth.draw_y0(g, 8, rows) if residual else None
    singles = [gemv(qtype, qd, sd, dev_u16_as_f16(x8[c:c + 1]),
                    dev(y08[c:c + 1]) if residual else None)[0] for c in range(8)]
    for n in range(2, 9):
        yn = gemv(qtype, qd, sd, dev_u16_as_f16(x8[:n]), dev(y08[:n]) if residual else None)
        for c in range(n):
            assert np.array_equal(yn[c].view(np.uint32), singles[c].view(np.uint32)), \
                f"{rows}x{k} columns={n}: column {c} differs from its 1-column GEMV"


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k", [(1024, 2048), (300, 1056)])
def test_gate_up_twins_bit_identical(qtype, rows, k):
    g = synth.rng(7 * rows + k)
    qg_, sg = synth.draw_matrix(g, qtype, rows, k)
    qu, su = synth.draw_matrix(g, qtype, rows, k)
    dg, dsg = dev_q(qtype, qg_, sg)
    du, dsu = dev_q(qtype, qu, su)
    x8 = synth.draw_x(g, 8, k)

    def run(x):
        h = torch.full((x.shape[0], rows), float("nan"), dtype=torch.float16, device="cuda")
        qg.qffn_gate_up_silu(qtype, dg, dsg, du, dsu, dev_u16_as_f16(x), h)
        torch.cuda.synchronize()
        return host(h.view(torch.int16))
    singles = [run(x8[c:c + 1])[0] for c in range(8)]
    for n in (2, 3, 4, 8):
        hn = run(x8[:n])
        for c in range(n):
            assert np.array_equal(hn[c], singles[c]), f"gate/up columns={n}: column {c}"


@pytest.mark.parametrize("ffn", [128, 512])
def test_moe_twins_bit_identical(ffn):
    """ffn 512 runs both down kernels: the staged one (1-2 columns) and the
    register kernel (more columns); ffn 128 the register kernel throughout."""
    case = synth.moe_case(synth.Q8_0, 32, ffn, 512, 16, topk=4, shared=True, residual=True,
                          seed=21)
    t, E, ffn, hidden = case["qtype"], case["n_expert"], case["ffn"], case["hidden"]
    mats = [dev_q(t, case[a], case[b]) for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd"))]
    sh = {}
    for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
        sh[a], sh[b] = dev_q(t, case["shared"][a], case["shared"][b])

    def run(cols):
        n = len(cols)
        ws = torch.empty(qg.qmoe_workspace_bytes(E, ffn, hidden, n, case["topk"]),
                         dtype=torch.uint8, device="cuda")
        y = torch.full((n, hidden), float("nan"), dtype=torch.float32, device="cuda")
        qg.qmoe_experts(t, *mats[0], *mats[1], *mats[2], E, ffn, hidden,
                        dev(case["ids"][cols]), dev(case["rw"][cols]),
                        dev_u16_as_f16(case["x"][cols]), y, ws, y0=dev(case["y0"][cols]),
                        shared=sh)
        torch.cuda.synchronize()
        return host(y)
    singles = [run([c])[0] for c in range(16)]
    for n in (2, 6, 8, 16):
        yn = run(list(range(n)))
        for c in range(n):
            assert np.array_equal(yn[c].view(np.uint32), singles[c].view(np.uint32)), \
                f"MoE columns={n}: column {c}"


def test_router_twins_bit_identical():
    g = np.random.Generator(np.random.PCG64(31))
    E, hidden, k = 256, 2048, 8
    w = dev((g.standard_normal((E, hidden)) * 0.02).astype(np.float32))
    x16 = g.standard_normal((16, hidden)).astype(np.float16)

    def run(x):
        n = x.shape[0]
        lg = torch.empty((n, E), dtype=torch.float32, device="cuda")
        ids = torch.empty((n, k), dtype=torch.int32, device="cuda")
        rw = torch.empty((n, k), dtype=torch.float32, device="cuda")
        qg.qmoe_router(w, dev(x), k, ids, rw, logits_out=lg)
        torch.cuda.synchronize()
        return host(lg), host(ids), host(rw)
    singles = [run(x16[c:c + 1]) for c in range(16)]
    for n in (2, 5, 8, 16):
        lg, ids, rw = run(x16[:n])
        for c in range(n):
            assert np.array_equal(lg[c].view(np.uint32), singles[c][0][0].view(np.uint32))
            assert np.array_equal(ids[c], singles[c][1][0])
            assert np.array_equal(rw[c].view(np.uint32), singles[c][2][0].view(np.uint32))
