"""Extreme values through both engines, against the oracle.

The other parity tests draw x from N(0, 1) and scales from |N(0, 0.02)|/8 or
/127. Here the f16 inputs sit at the ends of their range:
  * x all subnormal (|x| < 2^-14): the tensor cores must take f16 subnormals
    exactly (a flush to zero would lose the whole product);
  * x near the f16 maximum (|x| up to 65,504) with scales up to 65,504 and
    Q8_0 quants of -128: large f32 sums, no overflow;
  * subnormal f16 scales;
  * x = +-a in pairs, so the exact sums cancel (the bound's 1e-6 floor).
Tolerance: |y - y_ref| <= 1e-3 sum|w||x| + 1e-6 per element; the oracle is f64."""
import zlib

import numpy as np
import pytest

import oracle
import synth
from helpers import NTHREADS, assert_within, dev_q, dev_u16_as_f16, gemv_bound, host

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

# (rows, k): the first runs on the CUDA cores (K not a multiple of 256), the
# second on the tensor cores at every column count
SHAPES = {"cuda cores": (300, 1056), "tensor cores": (1100, 4096)}


def f16_bits(v):
    return np.asarray(v, dtype=np.float16).view(np.uint16)


def draw(kind, qtype, rows, k, ncols, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    q = synth.draw_quants(g, qtype, rows, k)
    nb = k // 32
    sign = lambda shape: np.where(g.random(shape) < 0.5, -1.0, 1.0)  # noqa: E731
    if kind == "subnormal_x":
        # subnormal f16: m * 2^-24 with 1 <= m < 1024; scales of 1-100 keep the
        # products far above the bound's 1e-6 floor
        x = f16_bits(sign((ncols, k)) * g.integers(1, 1024, (ncols, k)) * 2.0 ** -24)
        s = f16_bits(g.uniform(1.0, 100.0, (rows, nb)))
    elif kind == "huge":
        x = f16_bits(sign((ncols, k)) * g.uniform(30000.0, 65504.0, (ncols, k)))
        s = f16_bits(g.uniform(1.0, 65504.0, (rows, nb)))
        if qtype == synth.Q8_0:
            q[:, ::3] = -128
    elif kind == "subnormal_scales":
        x = synth.draw_x(g, ncols, k)
        s = f16_bits(g.integers(1, 1024, (rows, nb)) * 2.0 ** -24)
    elif kind == "cancel":
        a = g.uniform(0.5, 2.0, (ncols, k // 2))
        x = f16_bits(np.stack([a, -a], axis=-1).reshape(ncols, k))
        s = synth.draw_scales(g, qtype, rows, k)
        q = q.copy()
        if qtype == synth.Q8_0:
            q[:, 1::2] = q[:, 0::2]  # equal weights on each +a/-a pair: exact zeros
    else:
        raise ValueError(kind)
    return q, s, x


@pytest.mark.parametrize("engine", list(SHAPES))
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("kind", ["subnormal_x", "huge", "subnormal_scales", "cancel"])
@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_extreme_values(engine, qtype, kind, ncols):
    rows, k = SHAPES[engine]
    q, s, x = draw(kind, qtype, rows, k, ncols,
                   seed=zlib.crc32(f"{engine}/{qtype}/{kind}/{ncols}".encode()))
    dq, ds = dev_q(qtype, q, s)
    y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
    if ncols <= 8:
        (qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0)(dq, ds, dev_u16_as_f16(x), y)
    else:
        qg.qgemm_cols(qtype, dq, ds, dev_u16_as_f16(x), y)
    torch.cuda.synchronize()
    got = host(y)
    assert np.isfinite(got).all()
    yr, S = oracle.matmul(qtype, q, s, x, None, nthreads=NTHREADS)
    assert_within(got, yr, gemv_bound(S), f"{kind} {engine} {qtype} C={ncols}")
    if kind == "subnormal_x":
        # the check can see a flush to zero: the bound is far below |y|
        assert np.median(gemv_bound(S)) < 0.1 * np.median(np.abs(yr))


@pytest.mark.parametrize("engine", list(SHAPES))
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("kind", ["subnormal_x", "subnormal_scales", "cancel"])
@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_extreme_values_gate_up(engine, qtype, kind, ncols):
    """The fused gate/up on the same inputs (h = f16(SiLU(g) u) stays inside the
    f16 range here; the h bound carries the f16 rounding, subnormal h included)."""
    rows, k = SHAPES[engine]
    seed = zlib.crc32(f"gu/{engine}/{qtype}/{kind}/{ncols}".encode())
    qg_, sg, x = draw(kind, qtype, rows, k, ncols, seed=seed)
    qu, su, _ = draw(kind, qtype, rows, k, ncols, seed=seed + 1)
    h = torch.full((ncols, rows), float("nan"), dtype=torch.float16, device="cuda")
    qg.qffn_gate_up_silu(qtype, *dev_q(qtype, qg_, sg), *dev_q(qtype, qu, su),
                         dev_u16_as_f16(x), h)
    torch.cuda.synchronize()
    got = host(h).astype(np.float64)
    assert np.isfinite(got).all()
    href, gg, uu, Sg, Su = oracle.ffn_gate_up_silu(qtype, qg_, sg, qu, su, x, nthreads=NTHREADS)
    assert_within(got, href, oracle.h_bound(gg, uu, Sg, Su), f"gate/up {kind} {engine} C={ncols}")
