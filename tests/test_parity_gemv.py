"""GPU parity of the GEMV / twins / prefill-GEMM entry points against the oracle.

Tolerance (per element): |y_gpu - y_ref| <= 1e-3 * sum_k |w_k||x_k| + 1e-6, with
y_ref and the sum computed by the f64 oracle. Integer-exact cases (x = e_j, zero
blocks) are compared bit for bit.
"""
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


def run_gemv(qtype, q, scl, x, y0=None, api="gemv", inplace=False):
    dq, ds = dev_q(qtype, q, scl)
    dx = dev_u16_as_f16(x)
    ncols, rows = x.shape[0], scl.shape[0]
    y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    dy0 = None
    if y0 is not None:
        if inplace:
            y.copy_(torch.from_numpy(y0))
            dy0 = y
        else:
            dy0 = dev(y0)
    if api == "gemv":
        (qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0)(dq, ds, dx, y, dy0)
    else:
        qg.qgemm_cols(qtype, dq, ds, dx, y, dy0)
    torch.cuda.synchronize()
    return host(y)


def check_case(case, api="gemv", rows_sel=None, inplace=False, what=""):
    y = run_gemv(case["qtype"], case["q"], case["scl"], case["x"], case["y0"], api, inplace)
    yr, S = oracle.matmul(case["qtype"], case["q"], case["scl"], case["x"], case["y0"],
                          rows_sel=rows_sel, nthreads=NTHREADS)
    got = y if rows_sel is None else y[:, rows_sel]
    assert np.isfinite(got).all()
    assert_within(got, yr, gemv_bound(S), what)
    return y


def test_small_q8_gemv_2048():
    check_case(synth.small_q8_gemv(), what="Q8_0 2048x2048 C=1")


def test_q4_gemv_residual_5120():
    check_case(synth.q4_gemv_residual(), what="Q4_0 5120x5120 C=1 + y0")


def test_q4_gemv_residual_in_place():
    check_case(synth.q4_gemv_residual(seed=1), inplace=True, what="Q4_0 in place y += W x")


def test_lm_head_all_rows_and_draft_head():
    """The full 248,320-row Q8_0 LM head against the multithreaded oracle on
    every row, and the draft head: the same call on the first 65,536 rows of
    the same weights (a row prefix, no copy)."""
    case = synth.lm_head()
    qtype, rows = case["qtype"], case["rows"]
    dq, ds = dev_q(qtype, case["q"], case["scl"])
    dx = dev_u16_as_f16(case["x"])
    y = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qg.qgemv_q8_0(dq, ds, dx, y)
    nd = 65536
    yd = torch.full((1, nd), float("nan"), dtype=torch.float32, device="cuda")
    qg.qgemv_q8_0(dq[:nd], ds[:nd], dx, yd)
    torch.cuda.synchronize()
    yr, S = oracle.matmul(qtype, case["q"], case["scl"], case["x"], None, nthreads=NTHREADS)
    got = host(y)
    assert np.isfinite(got).all()
    assert_within(got, yr, gemv_bound(S), "Q8_0 LM head 248320x5120, every row")
    gd = host(yd)
    assert np.isfinite(gd).all()
    assert_within(gd, yr[:, :nd], gemv_bound(S[:, :nd]), "draft head: first 65536 rows")


def test_q4_lm_head_shape_all_rows():
    """One column of a Q4_0 matrix of the LM head's shape (248,320 x 5120, the
    bench's Q4_0 LM-head config) against the multithreaded oracle on every row;
    the output starts as NaN, so an unwritten row fails."""
    rows, k = 248320, 5120
    case = synth.gemv_case(synth.Q4_0, rows, k, 1, residual=False, seed=43)
    dq, ds = dev_q(synth.Q4_0, case["q"], case["scl"])
    y = torch.full((1, rows), float("nan"), dtype=torch.float32, device="cuda")
    qg.qgemv_q4_0(dq, ds, dev_u16_as_f16(case["x"]), y)
    torch.cuda.synchronize()
    yr, S = oracle.matmul(synth.Q4_0, case["q"], case["scl"], case["x"], None, nthreads=NTHREADS)
    got = host(y)
    assert np.isfinite(got).all()
    assert_within(got, yr, gemv_bound(S), "Q4_0 248320x5120 C=1, every row")


@pytest.mark.parametrize("k,engine", [(5120, "tensor cores"), (5152, "CUDA cores")])
def test_q8_matrix_beyond_2_gib(k, engine):
    """A Q8_0 matrix whose quants span more than 2^31 bytes (420,000 rows), at
    1 and 8 columns with a residual: byte offsets past 2 GiB on both engines
    (K = 5152 is not a multiple of 256, so it runs on the CUDA cores). Rows are
    sampled at the start, around the 2 GiB boundary, at the tail and at random;
    the output starts as NaN, so every row is also checked for being written."""
    rows = 420000
    assert rows * k > 2 ** 31
    g = synth.rng(k)
    q, s = synth.draw_matrix(g, synth.Q8_0, rows, k)
    dq, ds = dev_q(synth.Q8_0, q, s)
    edge = 2 ** 31 // k
    r = np.random.Generator(np.random.PCG64(5))
    sel = np.unique(np.concatenate([np.arange(64), edge - 64 + np.arange(128),
                                    rows - 96 + np.arange(96), r.integers(0, rows, 1024)]))
    for ncols in (1, 8):
        x = synth.draw_x(g, ncols, k)
        y0 = synth.draw_y0(g, ncols, rows)
        y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        qg.qgemv_q8_0(dq, ds, dev_u16_as_f16(x), y, dev(y0))
        torch.cuda.synchronize()
        got = host(y)
        assert np.isfinite(got).all(), f"{engine} C={ncols}: unwritten rows"
        yr, S = oracle.matmul(synth.Q8_0, q, s, x, y0, rows_sel=sel, nthreads=NTHREADS)
        assert_within(got[:, sel], yr, gemv_bound(S), f"Q8_0 {rows}x{k} ({engine}) C={ncols}")
    del dq, ds
    torch.cuda.empty_cache()


def test_no_device_error_after_tensor_core_calls():
    """Every tensor-core wait is bounded; none gives up on ordinary calls, so the
    device error word reads 0 afterwards (and reading clears it)."""
    qg.qg_device_error()  # start from a clear word
    for qtype, ncols in ((synth.Q4_0, 1), (synth.Q8_0, 8), (synth.Q4_0, 16)):
        case = synth.gemv_case(qtype, 3000, 5120, ncols, residual=True, seed=50 + ncols)
        check_case(case, api="cols", what=f"tensor-core {qtype} C={ncols}")
    assert qg.qg_device_error() == 0
    assert qg.qg_device_error() == 0


def test_bounded_waits_give_up_and_leave_the_context_usable():
    """The self-test waits on an mbarrier phase that nothing completes, with the
    tensor-core kernel's two wait forms (CTA scope, cluster-scope acquire). Each
    gives up after its bound, sets the wait bit in the device error word (read
    once, then clear), and the context runs a tensor-core call correctly right
    after."""
    qg.qg_device_error()  # start from a clear word
    assert qg.qg_wait_selftest() == (0, 0)
    assert qg.qg_device_error() & qg.QG_DEV_ERR_WAIT
    assert qg.qg_device_error() == 0
    case = synth.gemv_case(synth.Q4_0, 3000, 5120, 8, residual=True, seed=58)
    check_case(case, api="cols", what="tensor-core call after the wait self-test")
    assert qg.qg_device_error() == 0


def test_q4_large_one_column_sampled_rows():
    """One column of a large Q4_0 matrix (the tensor-core plan), ragged row tail."""
    case = synth.gemv_case(synth.Q4_0, 20000, 5120, 1, residual=True, seed=41)
    g = np.random.Generator(np.random.PCG64(7))
    sel = np.unique(np.concatenate([np.arange(64), 20000 - 96 + np.arange(96),
                                    g.integers(0, 20000, 2048)]))
    check_case(case, rows_sel=sel, what="Q4_0 20000x5120 C=1 (sampled rows)")


@pytest.mark.parametrize("rows", [5120, 17408])
@pytest.mark.parametrize("ncols", [2, 4, 8])
def test_twins(rows, ncols):
    check_case(synth.twins(rows, ncols), what=f"Q4_0 twins {rows}x5120 C={ncols}")


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k", [(1, 32), (7, 96), (33, 288), (1000, 2080), (129, 4096)])
@pytest.mark.parametrize("ncols", [1, 3, 8])
def test_ragged_shapes(qtype, rows, k, ncols):
    case = synth.gemv_case(qtype, rows, k, ncols, residual=(ncols != 3), seed=rows + k)
    check_case(case, what=f"ragged {qtype} {rows}x{k} C={ncols}")


# Row counts (k = 2048, 8 units of 256) whose tensor-core plan splits K over
# 8, 7, ..., 1 CTAs: the largest cluster whose clusters all stay resident on a
# GB300 at two CTAs per SM (36, 38, 46, 58, 74, 97, 152 clusters of 8 ... 2).
# Every count is ragged (not a multiple of the 64-row tile) and above 2^22
# weights, so 1-8 columns run on the tensor cores too.
K_SPLIT_ROWS = {8: 2299, 7: 2419, 6: 2943, 5: 3682, 4: 4729, 3: 6158, 2: 9725, 1: 10257}


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("ksplit", sorted(K_SPLIT_ROWS))
@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_every_k_split(qtype, ksplit, ncols):
    """Each K-split cluster size reduces its partial tiles through the one-way
    handoff to rank 0: the result is checked against the oracle, and for 8
    columns every column bit for bit against the 1-column call on it."""
    rows = K_SPLIT_ROWS[ksplit]
    case = synth.gemv_case(qtype, rows, 2048, ncols, residual=True, seed=100 + ksplit)
    y = check_case(case, api="cols", what=f"{qtype} {rows}x2048 C={ncols} (K split {ksplit})")
    if ncols == 8:
        for c in range(ncols):
            y1 = run_gemv(qtype, case["q"], case["scl"], case["x"][c:c + 1],
                          case["y0"][c:c + 1], api="gemv")
            assert np.array_equal(y1[0].view(np.uint32), y[c].view(np.uint32)), c


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("ncols", list(range(1, 17)))
def test_prefill_cols_all_widths(qtype, ncols):
    case = synth.gemv_case(qtype, 1040, 1280, ncols, residual=True, seed=ncols)
    check_case(case, api="cols", what=f"qgemm_cols {qtype} C={ncols}")


def test_large_k_chunked_x():
    case = synth.gemv_case(synth.Q4_0, 96, 65536, 1, residual=True, seed=5)
    check_case(case, what="Q4_0 k=65536")
    case = synth.gemv_case(synth.Q8_0, 40, 32768, 3, residual=False, seed=6)
    check_case(case, what="Q8_0 k=32768 C=3")


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("ncols", [1, 2, 8, 16])
def test_unit_vectors_bit_exact(qtype, ncols):
    rows, k = 300, 512
    g = synth.rng(21)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    cols = [0, 15, 16, 31, 33, 255, 256, 511, 100, 200, 300, 400, 17, 18, 19, 20][:ncols]
    x = np.zeros((ncols, k), dtype=np.float16)
    for c, j in enumerate(cols):
        x[c, j] = 1.0
    y = run_gemv(qtype, q, s, x.view(np.uint16), api="cols")
    w = oracle.dequant(qtype, q, s)
    for c, j in enumerate(cols):
        assert np.array_equal(y[c].astype(np.float64), w[:, j]), (qtype, ncols, j)


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("ncols", [1, 5, 16])
def test_zero_blocks_return_residual(qtype, ncols):
    rows, k = 200, 1024
    g = synth.rng(22)
    x = synth.draw_x(g, ncols, k)
    y0 = synth.draw_y0(g, ncols, rows)
    q = (np.full((rows, k // 2), 0x88, np.uint8) if qtype == synth.Q4_0
         else np.zeros((rows, k), np.int8))
    s = synth.draw_scales(g, qtype, rows, k)
    assert np.array_equal(run_gemv(qtype, q, s, x, y0, api="cols"), y0)
    q2 = synth.draw_quants(g, qtype, rows, k)
    assert np.array_equal(run_gemv(qtype, q2, np.zeros_like(s), x, y0, api="cols"), y0)


@pytest.mark.parametrize("ncols", [1, 4, 16])
def test_extreme_quants_and_scales(ncols):
    rows, k = 256, 768
    g = synth.rng(23)
    q = g.integers(-128, 128, size=(rows, k), dtype=np.int8)
    q[:, :32] = -128
    q[:, 32:64] = 127
    d = np.abs(g.standard_normal((rows, k // 32)))
    d[::3] *= 1e-6          # f16 subnormal scales
    d[1::3] *= 300.0        # large scales
    s = d.astype(np.float16).view(np.uint16)
    x = g.standard_normal((ncols, k)).astype(np.float16).view(np.uint16)
    check_case(dict(qtype=synth.Q8_0, q=q, scl=s, x=x, y0=None), api="cols",
               what="Q8_0 extremes")
    nib = g.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    nib[:, :16] = 0x00
    nib[:, 16:32] = 0xFF
    check_case(dict(qtype=synth.Q4_0, q=nib, scl=s, x=x, y0=None), api="cols",
               what="Q4_0 extremes")


@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_deterministic(ncols):
    case = synth.gemv_case(synth.Q4_0, 3000, 5120, ncols, residual=True, seed=31)
    a = run_gemv(synth.Q4_0, case["q"], case["scl"], case["x"], case["y0"], api="cols")
    b = run_gemv(synth.Q4_0, case["q"], case["scl"], case["x"], case["y0"], api="cols")
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_empty_rows_is_noop():
    y = torch.full((1, 4), 7.0, device="cuda")
    dq = torch.zeros((0, 16), dtype=torch.uint8, device="cuda")
    ds = torch.zeros((0, 1), dtype=torch.int16, device="cuda")
    dx = torch.zeros((1, 32), dtype=torch.float16, device="cuda")
    qg.qgemv_q4_0(dq, ds, dx, y)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
