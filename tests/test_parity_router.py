"""GPU parity of the MoE router ("Engine and kernels", section "Kernel families":
router, top-k and the expert kernels all on the GPU, no routing readback).

The logits are floating point and take the product tolerance; the expert ids
are an integer decision taken on the kernel's own f32 logits, so they are
compared bit for bit against the oracle's top-k of those same f32 values; the
routing weights are compared with the oracle's f64 softmax of the selected f32
logits."""
import numpy as np
import pytest

import oracle
from helpers import dev, host

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


def inputs(E, hidden, ncols, seed, kind="normal"):
    g = np.random.Generator(np.random.PCG64(seed))
    w = (g.standard_normal((E, hidden)) * 0.02).astype(np.float32)
    x = g.standard_normal((ncols, hidden)).astype(np.float16)
    if kind == "dup":  # duplicated router rows: equal logits, ties go to the lower id
        w[1::2] = w[0::2][: w[1::2].shape[0]]
    elif kind == "zero":  # zero router: every logit 0, ids 0..k-1, uniform weights
        w[:] = 0
    elif kind == "ascending":  # row e = (e+1) * row 0: logits ordered by expert id
        w[:] = np.abs(w[0])[None, :] * np.arange(1, E + 1, dtype=np.float32)[:, None]
        x = np.abs(x)
    return w, x


def run(w, x, k):
    E, hidden = w.shape
    ncols = x.shape[0]
    lg = torch.empty((ncols, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((ncols, k), dtype=torch.int32, device="cuda")
    rw = torch.empty((ncols, k), dtype=torch.float32, device="cuda")
    qg.qmoe_router(dev(w), dev(x), k, ids, rw, logits_out=lg)
    torch.cuda.synchronize()
    return host(lg), host(ids), host(rw)


def check(w, x, k):
    lg, ids, rw = run(w, x, k)
    ref, S = oracle.router_logits(w, x.view(np.uint16))
    err = np.abs(lg.astype(np.float64) - ref)
    tol = 1e-3 * S + 1e-6
    assert (err <= tol).all(), f"logits: worst {np.max(err - tol):.3e} over tolerance"
    rid, rv = oracle.topk(lg, k)
    assert np.array_equal(ids, rid)
    for c in range(x.shape[0]):
        p = oracle.softmax(rv[c])
        np.testing.assert_allclose(rw[c], p, rtol=2e-6, atol=1e-7)
        assert abs(float(np.sum(rw[c], dtype=np.float64)) - 1.0) < 1e-5
    return lg, ids, rw


@pytest.mark.parametrize("E,hidden,ncols,k", [
    (256, 2048, 1, 8),      # the 256-expert top-8 MoE at decode
    (256, 2048, 8, 8),      # verify width
    (256, 2048, 16, 8),     # prefill width
    (128, 5120, 4, 4),
    (1024, 768, 3, 32),     # largest expert count and k
    (7, 33, 2, 7),          # ragged: k == E, hidden not a multiple of 32
    (1, 5, 1, 1),           # one expert
    (300, 2048, 5, 1),      # E not a multiple of the cluster
    (64, 8192, 16, 8),      # x too large for shared memory: read from global memory
    (64, 8190, 13, 8),      # the same with rows that are not float4-aligned
    (256, 2048, 2, 32),     # k above the number of key segments that hold experts
])
def test_router_parity(E, hidden, ncols, k):
    w, x = inputs(E, hidden, ncols, seed=E * 31 + hidden + ncols)
    check(w, x, k)


def test_router_x_offset_by_one_element():
    """x starting 2 bytes past an 8-byte boundary (the documented alignment
    is 2 bytes): the global-memory path must take scalar loads."""
    E, hidden, ncols, k = 32, 8192, 16, 4
    w, x = inputs(E, hidden, ncols, seed=77)
    buf = torch.empty(ncols * hidden + 1, dtype=torch.float16, device="cuda")
    buf[1:] = torch.from_numpy(x.reshape(-1)).cuda()
    xd = buf[1:].view(ncols, hidden)
    lg = torch.empty((ncols, E), dtype=torch.float32, device="cuda")
    ids = torch.empty((ncols, k), dtype=torch.int32, device="cuda")
    rw = torch.empty((ncols, k), dtype=torch.float32, device="cuda")
    qg.qmoe_router(dev(w), xd, k, ids, rw, logits_out=lg)
    torch.cuda.synchronize()
    ref, S = oracle.router_logits(w, x.view(np.uint16))
    assert (np.abs(host(lg).astype(np.float64) - ref) <= 1e-3 * S + 1e-6).all()
    assert np.array_equal(host(ids), oracle.topk(host(lg), k)[0])


def test_router_ties_lowest_id():
    w, x = inputs(256, 2048, 4, seed=5, kind="dup")
    _, ids, _ = check(w, x, 8)
    # rows 2j and 2j+1 are equal, so a selected odd id is always preceded by its even twin
    for c in range(ids.shape[0]):
        pos = {int(e): i for i, e in enumerate(ids[c])}
        for e, i in pos.items():
            if e % 2 == 1:
                assert e - 1 in pos and pos[e - 1] < i


@pytest.mark.parametrize("k", [1, 8, 32])
def test_router_ascending_logits(k):
    """Logits increasing with the expert id: the candidates that survive the
    pruning threshold are the most numerous; the top k are the last k ids."""
    w, x = inputs(1024, 256, 2, seed=13, kind="ascending")
    _, ids, _ = check(w, x, k)
    assert (ids == np.arange(1023, 1023 - k, -1, dtype=np.int32)).all()


def test_router_zero_weights():
    w, x = inputs(64, 256, 3, seed=9, kind="zero")
    lg, ids, rw = check(w, x, 8)
    assert (lg == 0).all()
    assert (ids == np.arange(8, dtype=np.int32)).all()
    np.testing.assert_allclose(rw, 1.0 / 8, rtol=1e-6)


def test_router_feeds_experts():
    """The router's device outputs drive qmoe_experts with no host round trip:
    the MoE output equals the oracle's MoE evaluated with the same ids and
    routing weights (read back only for the oracle)."""
    import synth
    from helpers import NTHREADS, assert_within, dev_q, dev_u16_as_f16
    case = synth.moe_layer(ncols=8, seed=3)
    t, E, ffn, hidden, ncols, k = (case["qtype"], case["n_expert"], case["ffn"], case["hidden"],
                                   case["ncols"], case["topk"])
    g = np.random.Generator(np.random.PCG64(11))
    wr = (g.standard_normal((E, hidden)) * 0.02).astype(np.float32)
    x = dev_u16_as_f16(case["x"])
    ids = torch.empty((ncols, k), dtype=torch.int32, device="cuda")
    rw = torch.empty((ncols, k), dtype=torch.float32, device="cuda")
    lg = torch.empty((ncols, E), dtype=torch.float32, device="cuda")
    qg.qmoe_router(dev(wr), x, k, ids, rw, logits_out=lg)
    ws = torch.empty(qg.qmoe_workspace_bytes(E, ffn, hidden, ncols, k), dtype=torch.uint8,
                     device="cuda")
    y = torch.full((ncols, hidden), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s_ = case["shared"]
    sh = {}
    for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
        sh[a], sh[b] = dev_q(t, s_[a], s_[b])
    qg.qmoe_experts(t, *dev_q(t, case["qg"], case["sg"]), *dev_q(t, case["qu"], case["su"]),
                    *dev_q(t, case["qd"], case["sd"]), E, ffn, hidden, ids,
                    rw, x, y, ws, shared=sh, err_flag=err)
    torch.cuda.synchronize()
    rid, rv = oracle.topk(host(lg), k)
    assert np.array_equal(host(ids), rid)
    assert int(host(err)[0]) == 0
    ref_case = dict(case, ids=host(ids), rw=host(rw))
    # stage by stage on the GPU's own h (left in the workspace), then end to end
    from helpers import check_moe_staged, workspace_h
    check_moe_staged(ref_case, host(y), workspace_h(ws, ref_case), what="router -> MoE experts")
    yr, bound, _, _, rc = oracle.moe(ref_case, nthreads=NTHREADS)
    assert rc == 0
    assert_within(host(y), yr, bound, "router -> MoE experts (end to end)")
