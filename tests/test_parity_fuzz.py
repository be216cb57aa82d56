"""Seeded random shapes for every entry point, checked against the oracle.

The other parity files pick their shapes by hand; this one draws them from a
fixed-seed generator (so a failure reproduces exactly) across the whole
accepted range: row counts log-uniform from 1 to ~30,000, K any multiple of 32
(K a multiple of 256 in 60% of the cases, so both engines are drawn), 1-16
columns, no residual / a separate y0 / y += W x in place, both entry points of
the GEMV, the fused gate/up, MoE layers with random expert counts, widths,
top-k, shared expert on or off, duplicate and out-of-range ids, the router,
argmax and top-k. Tolerances are the product's: 1e-3 sum|w||x| + 1e-6 per
element for the products, the h bound for the gate/up, the staged and end-to-end
MoE bounds, bit-exact for every index and for the sampled values."""
import numpy as np
import pytest

import oracle
import synth
from helpers import NTHREADS, assert_within, dev, dev_q, dev_u16_as_f16, gemv_bound, host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q4_q8_gb300 import build
    build.build()
    oracle.build()


import gemm_q4_q8_gb300 as qg  # noqa: E402


def _rows(g, top):
    return int(np.exp(g.uniform(0.0, np.log(top))))


def _k(g, kmax_units):
    if g.random() < 0.6:
        return 256 * int(g.integers(1, kmax_units // 8 + 1))
    return 32 * int(g.integers(1, kmax_units + 1))


def gemv_shapes(n, seed=2024):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < n:
        qtype = int(g.choice([synth.Q4_0, synth.Q8_0]))
        k = _k(g, 256)                     # up to 8,192
        rows = _rows(g, 30000)
        if rows * k > (1 << 26):
            continue
        ncols = int(g.integers(1, 17))
        residual = str(g.choice(["none", "y0", "inplace"]))
        api = "cols" if ncols > 8 or g.random() < 0.3 else "gemv"
        out.append((qtype, rows, k, ncols, residual, api))
    return out


@pytest.mark.parametrize("i,shape", list(enumerate(gemv_shapes(240))))
def test_fuzz_gemv(i, shape):
    qtype, rows, k, ncols, residual, api = shape
    g = synth.rng(10000 + i)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    x = synth.draw_x(g, ncols, k)
    y0 = synth.draw_y0(g, ncols, rows) if residual != "none" else None
    dq, ds = dev_q(qtype, q, s)
    y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    dy0 = None
    if residual == "inplace":
        y.copy_(torch.from_numpy(y0))
        dy0 = y
    elif residual == "y0":
        dy0 = dev(y0)
    if api == "gemv":
        (qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0)(dq, ds, dev_u16_as_f16(x), y, dy0)
    else:
        qg.qgemm_cols(qtype, dq, ds, dev_u16_as_f16(x), y, dy0)
    torch.cuda.synchronize()
    got = host(y)
    assert np.isfinite(got).all(), shape
    sel = None
    if rows > 2048:
        r = np.random.Generator(np.random.PCG64(i))
        sel = np.unique(np.concatenate([np.arange(64), rows - 64 + np.arange(64),
                                        r.integers(0, rows, 512)]))
    yr, S = oracle.matmul(qtype, q, s, x, y0, rows_sel=sel, nthreads=NTHREADS)
    assert_within(got if sel is None else got[:, sel], yr, gemv_bound(S), f"fuzz gemv {shape}")


def gate_up_shapes(n, seed=2025):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < n:
        qtype = int(g.choice([synth.Q4_0, synth.Q8_0]))
        k = _k(g, 160)                     # up to 5,120
        rows = _rows(g, 20000)
        if rows * k > (1 << 23):
            continue
        out.append((qtype, rows, k, int(g.integers(1, 17))))
    return out


@pytest.mark.parametrize("i,shape", list(enumerate(gate_up_shapes(64))))
def test_fuzz_gate_up(i, shape):
    qtype, rows, k, ncols = shape
    g = synth.rng(20000 + i)
    qg_, sg = synth.draw_matrix(g, qtype, rows, k)
    qu, su = synth.draw_matrix(g, qtype, rows, k)
    x = synth.draw_x(g, ncols, k)
    h = torch.full((ncols, rows), float("nan"), dtype=torch.float16, device="cuda")
    qg.qffn_gate_up_silu(qtype, *dev_q(qtype, qg_, sg), *dev_q(qtype, qu, su),
                         dev_u16_as_f16(x), h)
    torch.cuda.synchronize()
    got = host(h).astype(np.float64)
    href, gg, uu, Sg, Su = oracle.ffn_gate_up_silu(qtype, qg_, sg, qu, su, x, nthreads=NTHREADS)
    assert np.isfinite(got).all(), shape
    assert_within(got, href, oracle.h_bound(gg, uu, Sg, Su), f"fuzz gate/up {shape}")


def moe_shapes(n, seed=2026):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    while len(out) < n:
        E = int(g.integers(1, 49))
        ffn = 32 * int(g.integers(1, 25))
        ncols = int(g.integers(1, 17))
        hidden = 32 * int(g.integers(1, 65))
        topk = int(g.integers(1, min(16, E, 256 // ncols) + 1))
        if ncols * hidden > 32768 or (topk + 1) * ffn > 32768:
            continue
        out.append((int(g.choice([synth.Q4_0, synth.Q8_0])), E, ffn, hidden, ncols, topk,
                    bool(g.random() < 0.7), bool(g.random() < 0.5), str(g.choice(
                        ["distinct", "distinct", "duplicate", "invalid"]))))
    return out


@pytest.mark.parametrize("i,shape", list(enumerate(moe_shapes(48))))
def test_fuzz_moe(i, shape):
    from test_parity_ffn_moe import check_moe
    qtype, E, ffn, hidden, ncols, topk, shared, residual, ids_kind = shape
    case = synth.moe_case(qtype, E, ffn, hidden, ncols, topk=topk, shared=shared,
                          residual=residual, seed=30000 + i)
    ids = case["ids"].copy()
    r = np.random.Generator(np.random.PCG64(i))
    c = int(r.integers(0, ncols))
    if ids_kind == "duplicate" and topk > 1:
        ids[c, -1] = ids[c, 0]
    elif ids_kind == "invalid":
        ids[c, int(r.integers(0, topk))] = int(r.choice([-1, E, E + 7]))
    check_moe(case, ids=ids, what=f"fuzz MoE {shape}")


def router_shapes(n, seed=2027):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        E = int(np.exp(g.uniform(0.0, np.log(1024))))
        out.append((E, int(g.integers(1, 6000)), int(g.integers(1, 17)),
                    int(g.integers(1, min(32, E) + 1))))
    return out


@pytest.mark.parametrize("i,shape", list(enumerate(router_shapes(32))))
def test_fuzz_router(i, shape):
    from test_parity_router import check
    E, hidden, ncols, k = shape
    g = np.random.Generator(np.random.PCG64(40000 + i))
    w = (g.standard_normal((E, hidden)) * 0.02).astype(np.float32)
    x = g.standard_normal((ncols, hidden)).astype(np.float16)
    check(w, x, k)


def sampling_shapes(n, seed=2028):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        nn = int(np.exp(g.uniform(0.0, np.log(300000))))
        out.append((nn, int(g.integers(1, 17)), int(g.integers(1, min(256, nn) + 1)),
                    str(g.choice(["normal", "ties", "specials"]))))
    return out


@pytest.mark.parametrize("i,shape", list(enumerate(sampling_shapes(32))))
def test_fuzz_sampling(i, shape):
    from test_parity_sampling import check, logits
    nn, ncols, k, kind = shape
    check(logits(nn, ncols, 50000 + i, kind), k)
