"""Property tests of the oracle's product (CPU; needs hypothesis, skipped
without it).

For random shapes, both quant types, with and without a residual, and scales
drawn as arbitrary finite f16 bit patterns (zero, subnormal, huge), the oracle
must equal, bit for bit, a sequential sum written here from the block format:
weight (q - 8) * d for Q4_0 (low nibble of byte j is element j, high nibble is
element j + 16), q * d for Q8_0, accumulated in f64 in k order, y0 added last.
The quants are packed by this file's own packer, not by any library code.
"""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import synth  # noqa: E402


def _pack_q4(ql):
    """Logical nibbles [rows][k] -> GGUF-order bytes [rows][k/2]."""
    rows, k = ql.shape
    out = np.empty((rows, k // 2), np.uint8)
    for b in range(k // 32):
        lo = ql[:, b * 32:b * 32 + 16]
        hi = ql[:, b * 32 + 16:b * 32 + 32]
        out[:, b * 16:(b + 1) * 16] = (lo | (hi << 4)).astype(np.uint8)
    return out


finite_f16 = st.integers(0, 0xFFFF).filter(lambda b: (b & 0x7C00) != 0x7C00)


@settings(max_examples=60, deadline=None)
@given(qtype=st.sampled_from([synth.Q4_0, synth.Q8_0]), rows=st.integers(1, 5),
       nblk=st.integers(1, 4), ncols=st.integers(1, 3), residual=st.booleans(),
       seed=st.integers(0, 2**31 - 1), scale_bits=st.lists(finite_f16, min_size=20, max_size=20))
def test_product_equals_sequential_sum(oracle_lib, qtype, rows, nblk, ncols, residual, seed,
                                       scale_bits):
    k = 32 * nblk
    g = np.random.Generator(np.random.PCG64(seed))
    if qtype == synth.Q4_0:
        ql = g.integers(0, 16, size=(rows, k))
        packed, wint = _pack_q4(ql), ql - 8
    else:
        ql = g.integers(-128, 128, size=(rows, k))
        packed, wint = ql.astype(np.int8), ql
    scl = np.array(scale_bits[:rows * nblk], np.uint16).reshape(rows, nblk)
    d = scl.view(np.float16).astype(np.float64)
    x = g.standard_normal((ncols, k)).astype(np.float16)
    y0 = g.standard_normal((ncols, rows)).astype(np.float32) if residual else None
    y, S = oracle_lib.matmul(qtype, packed, scl, x.view(np.uint16), y0)
    for c in range(ncols):
        for r in range(rows):
            acc, s = 0.0, 0.0
            for kk in range(k):
                w = float(wint[r, kk]) * float(d[r, kk // 32])
                acc += w * float(x[c, kk])
                s += abs(w) * abs(float(x[c, kk]))
            if residual:
                acc += float(y0[c, r])
            assert y[c, r] == acc or (np.isnan(y[c, r]) and np.isnan(acc))
            assert S[c, r] == s or (np.isnan(S[c, r]) and np.isnan(s))
