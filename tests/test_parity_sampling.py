"""GPU parity of greedy argmax and top-k against the oracle: indices and values
bit for bit ("Engine and kernels", section "Fewer passes": lowest-index
tie-breaking)."""
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


def logits(n, ncols, seed, kind):
    g = np.random.Generator(np.random.PCG64(seed))
    if kind == "normal":
        x = g.standard_normal((ncols, n)).astype(np.float32)
    elif kind == "ties":       # few distinct values: long runs of equal keys
        x = (g.integers(-3, 4, size=(ncols, n)) * 0.25).astype(np.float32)
    elif kind == "specials":   # signed zeros, infinities and NaNs mixed in
        x = g.standard_normal((ncols, n)).astype(np.float32)
        m = g.random((ncols, n))
        x[m < 0.05] = np.nan
        x[(m >= 0.05) & (m < 0.1)] = -0.0
        x[(m >= 0.1) & (m < 0.12)] = 0.0
        x[(m >= 0.12) & (m < 0.125)] = -np.inf
        x[(m >= 0.125) & (m < 0.127)] = np.inf
    elif kind == "ascending":  # every element beats the previous: worst case for filtering
        x = np.tile(np.arange(n, dtype=np.float32), (ncols, 1))
    elif kind == "allnan":
        x = np.full((ncols, n), np.nan, dtype=np.float32)
    elif kind.startswith("lanes"):  # the largest values on a few index classes mod 512:
        m = int(kind[5:])          # many keys clear the threshold of thread maxima
        x = g.standard_normal((ncols, n)).astype(np.float32)
        big = (np.arange(n) % 512) < m
        x[:, big] += 1000.0
    return x


def check(x, k):
    ncols, n = x.shape
    dx = dev(x)
    idx = torch.empty(ncols, dtype=torch.int32, device="cuda")
    val = torch.empty(ncols, dtype=torch.float32, device="cuda")
    qg.qargmax_f32(dx, idx, val)
    ti = torch.empty((ncols, k), dtype=torch.int32, device="cuda")
    tv = torch.empty((ncols, k), dtype=torch.float32, device="cuda")
    qg.qtopk_f32(dx, k, ti, tv)
    torch.cuda.synchronize()
    ri, rv = oracle.argmax(x)
    rti, rtv = oracle.topk(x, k)
    assert np.array_equal(host(idx), ri)
    assert np.array_equal(host(val).view(np.uint32), rv.view(np.uint32))
    assert np.array_equal(host(ti), rti)
    assert np.array_equal(host(tv).view(np.uint32), rtv.view(np.uint32))


@pytest.mark.parametrize("kind", ["normal", "ties", "specials"])
def test_lm_head_width(kind):
    check(logits(248320, 2, 1, kind), 40)


@pytest.mark.parametrize("n,ncols,k", [(1, 1, 1), (7, 3, 7), (9, 16, 1), (1000, 5, 256),
                                       (65536, 1, 64), (33333, 4, 17)])
def test_ragged_shapes(n, ncols, k):
    check(logits(n, ncols, n + k, "ties"), k)


@pytest.mark.parametrize("m,k", [(64, 64), (256, 256), (16, 40)])
def test_many_candidates(m, k):
    """Index classes that hold every large value: k = 64 leaves ~2,000 keys
    above the threshold (sorted), k = 256 ~7,800 (the streaming fallback)."""
    check(logits(248320, 2, 5, f"lanes{m}"), k)


def test_unaligned_logits():
    """Logits one float past a 16-byte boundary (and n % 4 == 0): the argmax
    and top-k fall back from float4 to scalar loads and give the same answer."""
    x = logits(248320, 2, 9, "ties")
    buf = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")
    dx = buf[1:].view(x.shape)
    dx.copy_(torch.from_numpy(x))
    assert dx.data_ptr() % 16 == 4
    idx = torch.empty(2, dtype=torch.int32, device="cuda")
    val = torch.empty(2, dtype=torch.float32, device="cuda")
    qg.qargmax_f32(dx, idx, val)
    ti = torch.empty((2, 40), dtype=torch.int32, device="cuda")
    tv = torch.empty((2, 40), dtype=torch.float32, device="cuda")
    qg.qtopk_f32(dx, 40, ti, tv)
    torch.cuda.synchronize()
    ri, rv = oracle.argmax(x)
    rti, rtv = oracle.topk(x, 40)
    assert np.array_equal(host(idx), ri)
    assert np.array_equal(host(val).view(np.uint32), rv.view(np.uint32))
    assert np.array_equal(host(ti), rti)
    assert np.array_equal(host(tv).view(np.uint32), rtv.view(np.uint32))


def test_all_nan_and_ascending():
    check(logits(5000, 2, 3, "allnan"), 5)
    check(logits(70000, 1, 4, "ascending"), 256)


def test_argument_errors():
    x = torch.zeros((2, 10), dtype=torch.float32, device="cuda")
    i = torch.empty((2, 11), dtype=torch.int32, device="cuda")
    with pytest.raises(qg.QGError):
        qg.qtopk_f32(x, 11, i)
    with pytest.raises(qg.QGError):
        qg.qtopk_f32(x, 0, i)
