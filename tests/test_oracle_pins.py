"""Pins for the CPU oracle, checked against facts that do not come from the oracle.

Each test states what it pins: hand-worked blocks (tests/golden/blocks.json),
the f16 decoder against numpy's, x = e_j returning a dequantised column, zero
blocks, linearity, brute force over logical integer weights packed by an
independent packer, multi-column consistency, SiLU closed forms and MoE
reductions to a single gated FFN.
"""
import json
import math
import os

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.usefixtures("oracle_lib")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "blocks.json")


def f16bits(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


# ------------------------------------------------------------------ packers
# Written here from the format statement, independently of synth and oracle:
# byte j of a Q4_0 block = (element j) | (element j+16) << 4.

def pack_q4_row(qlogical):
    qlogical = np.asarray(qlogical, dtype=np.int64)
    k = qlogical.size
    out = bytearray()
    for b in range(k // 32):
        blk = qlogical[b * 32:(b + 1) * 32]
        for j in range(16):
            out.append(int(blk[j]) | (int(blk[j + 16]) << 4))
    return np.frombuffer(bytes(out), dtype=np.uint8)


def golden_block(case):
    t = case["type"]
    if t == "q4_0":
        spec = case["bytes"]
        if spec.startswith("j | (15-j)<<4"):
            b = [j | ((15 - j) << 4) for j in range(16)]
        elif spec.startswith("j for j=0..15"):
            b = list(range(16))
        elif spec.startswith("0x88"):
            b = [0x88] * 16
        elif spec.startswith("0x99"):
            b = [0x99] * 16
        else:
            raise AssertionError(spec)
        return synth.Q4_0, np.array(b, dtype=np.uint8)
    spec = case["q"]
    if spec.startswith("[-127, 0, 127]"):
        q = [-127, 0, 127] + [0] * 29
    elif spec.startswith("(-1)^i * i"):
        q = [(-1) ** i * i for i in range(32)]
    elif spec.startswith("-128 at index 5"):
        q = [0] * 32
        q[5] = -128
    else:
        raise AssertionError(spec)
    return synth.Q8_0, np.array(q, dtype=np.int8)


def golden_x(spec):
    if spec == "ones":
        v = [1.0] * 32
    elif spec == "k+1":
        v = [k + 1.0 for k in range(32)]
    elif spec == "first16":
        v = [1.0] * 16 + [0.0] * 16
    elif spec == "last16":
        v = [0.0] * 16 + [1.0] * 16
    elif spec.startswith("e:"):
        v = [0.0] * 32
        v[int(spec[2:])] = 1.0
    else:
        raise AssertionError(spec)
    return f16bits(v).reshape(1, 32)


def test_golden_blocks(oracle_lib):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        t, q = golden_block(case)
        scl = np.array([[int(case["d_bits"], 16)]], dtype=np.uint16)
        x = golden_x(case["x"])
        y0 = None
        if "y0" in case:
            y0 = np.array([[case["y0"]]], dtype=np.float32)
        y, S = oracle_lib.matmul(t, q.reshape(1, -1), scl, x, y0)
        assert y[0, 0] == case["expected"], (case["name"], y[0, 0], case["expected"])


def test_golden_repack(oracle_lib):
    rp = json.load(open(GOLDEN))["repack"]
    blk = bytes.fromhex(rp["q4_block_hex"].replace(" ", ""))
    q, s = oracle_lib.repack(synth.Q4_0, np.frombuffer(blk, dtype=np.uint8), 1, 32)
    assert s[0, 0] == int(rp["expected_scale"], 16)
    assert q.tobytes() == bytes.fromhex(rp["expected_nib_hex"])
    blk = bytes.fromhex(rp["q8_block_hex"].replace(" ", ""))
    q, s = oracle_lib.repack(synth.Q8_0, np.frombuffer(blk, dtype=np.uint8), 1, 32)
    assert s[0, 0] == int(rp["expected_q8_scale"], 16)
    assert q.tobytes() == bytes.fromhex(rp["expected_q8_hex"])


def test_f16_decoder_all_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def _logical_case(qtype, rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    if qtype == synth.Q4_0:
        ql = g.integers(0, 16, size=(rows, k))
        packed = np.stack([pack_q4_row(ql[r]) for r in range(rows)])
        wint = ql - 8
    else:
        ql = g.integers(-128, 128, size=(rows, k))
        packed = ql.astype(np.int8)
        wint = ql
    d = (np.abs(g.standard_normal((rows, k // 32))) * 0.02).astype(np.float16)
    return packed, d.view(np.uint16), wint, d.astype(np.float64)


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_brute_force_4x64(oracle_lib, qtype):
    rows, k, ncols = 4, 64, 3
    packed, scl, wint, d = _logical_case(qtype, rows, k, seed=11)
    g = np.random.Generator(np.random.PCG64(12))
    x = g.standard_normal((ncols, k)).astype(np.float16)
    y0 = g.standard_normal((ncols, rows)).astype(np.float32)
    y, S = oracle_lib.matmul(qtype, packed, scl, x.view(np.uint16), y0)
    for c in range(ncols):
        for r in range(rows):
            acc, s = 0.0, 0.0
            for kk in range(k):
                w = float(wint[r, kk]) * float(d[r, kk // 32])
                acc += w * float(x[c, kk])
                s += abs(w) * abs(float(x[c, kk]))
            acc += float(y0[c, r])
            assert y[c, r] == acc
            assert S[c, r] == s


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_unit_vector_returns_column(oracle_lib, qtype):
    rows, k = 8, 96
    packed, scl, wint, d = _logical_case(qtype, rows, k, seed=3)
    for j in (0, 15, 16, 31, 32, 47, 63, 95):
        x = np.zeros((1, k), dtype=np.float16)
        x[0, j] = 1.0
        y, _ = oracle_lib.matmul(qtype, packed, scl, x.view(np.uint16))
        expect = wint[:, j].astype(np.float64) * d[:, j // 32]
        assert np.array_equal(y[0], expect)


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_zero_weights_give_residual(oracle_lib, qtype):
    rows, k = 5, 64
    g = synth.rng(4)
    x = synth.draw_x(g, 2, k)
    y0 = synth.draw_y0(g, 2, rows)
    if qtype == synth.Q4_0:
        q = np.full((rows, k // 2), 0x88, dtype=np.uint8)
    else:
        q = np.zeros((rows, k), dtype=np.int8)
    scl = synth.draw_scales(g, qtype, rows, k)
    y, S = oracle_lib.matmul(qtype, q, scl, x, y0)
    assert np.array_equal(y, y0.astype(np.float64))
    assert np.all(S == 0)
    # scale zero with random quants
    q2 = synth.draw_quants(g, qtype, rows, k)
    y, _ = oracle_lib.matmul(qtype, q2, np.zeros_like(scl), x, y0)
    assert np.array_equal(y, y0.astype(np.float64))


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_linearity(oracle_lib, qtype):
    rows, k = 16, 128
    g = synth.rng(5)
    q, scl = synth.draw_matrix(g, qtype, rows, k)
    x = g.standard_normal((2, k)).astype(np.float16)
    mask = np.arange(k) % 3 == 0
    x1 = np.where(mask, x[0], 0).astype(np.float16)
    x2 = np.where(~mask, x[1], 0).astype(np.float16)
    a, b = 0.5, -4.0
    xs = (a * x1.astype(np.float64) + b * x2.astype(np.float64)).astype(np.float16)
    assert np.array_equal(xs.astype(np.float64),
                          a * x1.astype(np.float64) + b * x2.astype(np.float64))
    y1, S1 = oracle_lib.matmul(qtype, q, scl, x1.view(np.uint16).reshape(1, -1))
    y2, S2 = oracle_lib.matmul(qtype, q, scl, x2.view(np.uint16).reshape(1, -1))
    ys, _ = oracle_lib.matmul(qtype, q, scl, xs.view(np.uint16).reshape(1, -1))
    assert np.all(np.abs(ys - (a * y1 + b * y2)) <= 1e-12 * (abs(a) * S1 + abs(b) * S2) + 1e-300)


def test_multicolumn_equals_single(oracle_lib):
    rows, k = 12, 160
    g = synth.rng(6)
    q, scl = synth.draw_matrix(g, synth.Q4_0, rows, k)
    x = synth.draw_x(g, 5, k)
    y0 = synth.draw_y0(g, 5, rows)
    y, S = oracle_lib.matmul(synth.Q4_0, q, scl, x, y0)
    for c in range(5):
        yc, Sc = oracle_lib.matmul(synth.Q4_0, q, scl, x[c:c + 1], y0[c:c + 1])
        assert np.array_equal(y[c], yc[0]) and np.array_equal(S[c], Sc[0])


def test_row_selection_matches_full(oracle_lib):
    rows, k = 40, 64
    g = synth.rng(7)
    q, scl = synth.draw_matrix(g, synth.Q8_0, rows, k)
    x = synth.draw_x(g, 2, k)
    y0 = synth.draw_y0(g, 2, rows)
    y, S = oracle_lib.matmul(synth.Q8_0, q, scl, x, y0, nthreads=3)
    sel = np.array([39, 0, 17, 17, 5])
    ys, Ss = oracle_lib.matmul(synth.Q8_0, q, scl, x, y0, rows_sel=sel)
    assert np.array_equal(ys, y[:, sel]) and np.array_equal(Ss, S[:, sel])


def test_silu_closed_forms(oracle_lib):
    assert oracle_lib.silu(0.0) == 0.0
    for z in (0.1, 0.5, 1.0, 2.4, 7.0, 30.0):
        # sigmoid(z) = (1 + tanh(z/2)) / 2
        ref = z * (1.0 + math.tanh(z / 2.0)) / 2.0
        assert abs(oracle_lib.silu(z) - ref) <= 1e-15 * abs(ref) + 1e-300
        # SiLU(-z) = SiLU(z) - z
        assert abs(oracle_lib.silu(-z) - (oracle_lib.silu(z) - z)) <= 1e-14 * abs(z)
    assert oracle_lib.silu(60.0) == 60.0 or abs(oracle_lib.silu(60.0) - 60.0) < 1e-20
    assert abs(oracle_lib.silu(-60.0)) < 1e-20


def test_ffn_gate_up_against_parts(oracle_lib):
    rows, k, ncols = 10, 96, 3
    g = synth.rng(8)
    qg, sg = synth.draw_matrix(g, synth.Q4_0, rows, k)
    qu, su = synth.draw_matrix(g, synth.Q4_0, rows, k)
    x = synth.draw_x(g, ncols, k)
    h, gg, uu, Sg, Su = oracle_lib.ffn_gate_up_silu(synth.Q4_0, qg, sg, qu, su, x)
    yg, _ = oracle_lib.matmul(synth.Q4_0, qg, sg, x)
    yu, _ = oracle_lib.matmul(synth.Q4_0, qu, su, x)
    assert np.array_equal(gg, yg) and np.array_equal(uu, yu)
    ref = yg * (1.0 + np.tanh(yg / 2.0)) / 2.0 * yu
    assert np.all(np.abs(h - ref) <= 1e-14 * np.abs(ref) + 1e-300)


def _dense_ffn(qtype, qg, sg, qu, su, qd, sd, xbits, oracle_lib):
    """Gated FFN from dequantised matrices with numpy matmuls (library steps)."""
    x = xbits.view(np.float16).astype(np.float64)
    G = oracle_lib.dequant(qtype, qg, sg)
    U = oracle_lib.dequant(qtype, qu, su)
    D = oracle_lib.dequant(qtype, qd, sd)
    gg, uu = G @ x, U @ x
    hh = gg * (1.0 + np.tanh(gg / 2.0)) / 2.0 * uu
    return D @ hh


def test_moe_reductions(oracle_lib):
    E, ffn, hidden, ncols, topk = 6, 64, 96, 2, 2
    case = synth.moe_case(synth.Q8_0, E, ffn, hidden, ncols, topk=topk, shared=True,
                          residual=True, seed=9)
    # experts 1 and 4 identical
    per_gu = case["qg"].shape[0] // E
    per_d = case["qd"].shape[0] // E
    for n, per in (("qg", per_gu), ("sg", per_gu), ("qu", per_gu), ("su", per_gu),
                   ("qd", per_d), ("sd", per_d)):
        case[n][4 * per:5 * per] = case[n][1 * per:2 * per]
    case["ids"] = np.array([[1, 4], [2, 5]], dtype=np.int32)
    case["rw"] = np.array([[0.25, 0.75], [1.0, 0.0]], dtype=np.float32)

    def sl(n, e, per):
        return case[n][e * per:(e + 1) * per]

    y, bound, uniq, nu, rc = oracle_lib.moe(case)
    assert rc == 0
    assert list(uniq[:nu]) == [1, 2, 4, 5] and np.all(uniq[nu:] == -1)
    sh = case["shared"]
    for c, e in ((0, 1), (1, 2)):
        xb = case["x"][c]
        ref = _dense_ffn(synth.Q8_0, sl("qg", e, per_gu), sl("sg", e, per_gu),
                         sl("qu", e, per_gu), sl("su", e, per_gu), sl("qd", e, per_d),
                         sl("sd", e, per_d), xb, oracle_lib)
        ref = ref + _dense_ffn(synth.Q8_0, sh["qg"], sh["sg"], sh["qu"], sh["su"],
                               sh["qd"], sh["sd"], xb, oracle_lib)
        ref = ref + case["y0"][c].astype(np.float64)
        assert np.all(np.abs(y[c] - ref) <= 1e-12 * (np.abs(ref) + 1.0))
    # an invalid id contributes nothing and is reported
    bad = case["ids"].copy()
    bad[1, 1] = E + 3
    yb, _, uniq_b, nub, rcb = oracle_lib.moe(case, ids=bad)
    assert rcb == 3
    assert list(uniq_b[:nub]) == [1, 2, 4]
    assert np.array_equal(yb, y)  # the dropped slot had weight 0


def test_moe_shared_only_and_empty_routing(oracle_lib):
    E, ffn, hidden = 3, 32, 64
    case = synth.moe_case(synth.Q4_0, E, ffn, hidden, 1, topk=1, shared=True,
                          residual=False, seed=10)
    case["rw"] = np.zeros((1, 1), dtype=np.float32)
    y, bound, uniq, nu, rc = oracle_lib.moe(case)
    sh = case["shared"]
    ref = _dense_ffn(synth.Q4_0, sh["qg"], sh["sg"], sh["qu"], sh["su"], sh["qd"],
                     sh["sd"], case["x"][0], oracle_lib)
    assert np.all(np.abs(y[0] - ref) <= 1e-12 * (np.abs(ref) + 1.0))
    assert np.all(bound > 0)


def test_repack_is_one_group_permutation(oracle_lib):
    """Scales pass through unchanged, and every 16-byte group of every block of
    every row is reordered by the same permutation: the one a block of distinct
    bytes 0..15 reveals (pinned by the golden block above)."""
    probe = np.concatenate([[0, 0], np.arange(16)]).astype(np.uint8)
    perm, _ = oracle_lib.repack(synth.Q4_0, probe, 1, 32)
    perm = perm.view(np.uint8).reshape(16).astype(np.int64)
    assert sorted(perm.tolist()) == list(range(16))
    for qtype in (synth.Q4_0, synth.Q8_0):
        g = synth.rng(13)
        q, s = synth.draw_matrix(g, qtype, 7, 96)
        blocks = synth.to_gguf_blocks(qtype, q, s)
        q2, s2 = oracle_lib.repack(qtype, blocks, 7, 96)
        assert np.array_equal(s2, s)
        a = q.view(np.uint8).reshape(7, -1, 16)
        b = q2.view(np.uint8).reshape(7, -1, 16)
        assert np.array_equal(b, a[:, :, perm])


def test_h_bound_dominates_f16_rounding(oracle_lib):
    """The h tolerance is at least one f16 rounding of h (exact inputs)."""
    g = np.linspace(-8, 8, 41)
    u = np.linspace(-3, 3, 41)
    b = oracle_lib.h_bound(g, u, np.zeros_like(g), np.zeros_like(u))
    h = g * (1.0 + np.tanh(g / 2.0)) / 2.0 * u
    h16 = h.astype(np.float16).astype(np.float64)
    assert np.all(np.abs(h16 - h) <= b)


def _golden_vec(vals):
    return np.array([float(v) for v in vals], dtype=np.float32)


def test_golden_sampling(oracle_lib):
    for case in json.load(open(GOLDEN))["sampling"]["cases"]:
        x = _golden_vec(case["x"])
        idx, val = oracle_lib.argmax(x[None, :])
        assert int(idx[0]) == case["argmax"], case
        tidx, tval = oracle_lib.topk(x[None, :], x.size)
        assert tidx[0].tolist() == case["topk_idx"], case
        assert np.array_equal(tval[0], x[tidx[0]], equal_nan=True)


def test_sampling_matches_numpy_orderings(oracle_lib):
    """Against numpy's first-occurrence argmax and a lexicographic sort on
    (NaN last, value descending, index ascending), with many ties."""
    g = np.random.Generator(np.random.PCG64(5))
    for n in (1, 7, 300, 4096):
        x = g.integers(-6, 6, size=(3, n)).astype(np.float32) * 0.5
        x[1, ::7] = np.nan
        x[2, :] = np.where(g.random(n) < 0.3, -0.0, x[2, :]).astype(np.float32)
        idx, val = oracle_lib.argmax(x)
        k = min(n, 37)
        tidx, tval = oracle_lib.topk(x, k)
        for c in range(3):
            v = x[c]
            order = np.lexsort((np.arange(n), -np.nan_to_num(v, nan=0.0), np.isnan(v)))
            assert tidx[c].tolist() == order[:k].tolist()
            assert int(idx[c]) == int(order[0])
            if not np.isnan(v).all():
                assert int(idx[c]) == int(np.nanargmax(v))


def test_router_logits_against_numpy(oracle_lib):
    g = np.random.Generator(np.random.PCG64(11))
    w = g.standard_normal((37, 96)).astype(np.float32)
    x = g.standard_normal((3, 96)).astype(np.float16)
    lg, S = oracle_lib.router_logits(w, x.view(np.uint16))
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    assert np.allclose(lg, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(S, np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64)).T, rtol=1e-12)
    # one-hot x picks a column of W exactly
    e = np.zeros((1, 96), dtype=np.float16)
    e[0, 5] = 1.0
    lg1, _ = oracle_lib.router_logits(w, e.view(np.uint16))
    assert np.array_equal(lg1[0], w[:, 5].astype(np.float64))


def test_softmax_closed_forms(oracle_lib):
    assert np.allclose(oracle_lib.softmax(np.zeros(8, np.float32)), np.full(8, 0.125), rtol=0, atol=1e-15)
    p = oracle_lib.softmax(np.array([np.log(3.0), 0.0], np.float32))
    l3 = float(np.float32(np.log(3.0)))
    assert abs(p[0] - np.exp(l3) / (np.exp(l3) + 1.0)) < 1e-15 and abs(p.sum() - 1.0) < 1e-15
    big = oracle_lib.softmax(np.array([1000.0, 999.0, -1000.0], np.float32))
    assert abs(big[0] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-12 and big[2] == 0.0
