"""Pins of the oracle's tolerance functions, from below and from above.

The h tolerance (qref_h_bound) carries the GEMV tolerance 1e-3 * S + 1e-6 of
the gate and up projections through SiLU(g) * u ("Engine and kernels", section
"Kernel families", fused gate/up) and adds one f16 rounding. From below it must
cover every perturbation of g and u inside their tolerances (checked here by
brute force over a grid of perturbations); from above it must stay within a
small factor of the first-order formula, written independently below, so that
a bound made looser by a constant factor fails. The MoE bound of qref_moe is
pinned the same way against a first-order propagation written in numpy, and
both the staged and the end-to-end bounds are shown to reject three wrong
routed combines (a dropped expert, uniform weights, swapped weights) with the
oracle standing in for the GPU.
"""
import math

import numpy as np
import pytest

import synth
from helpers import NTHREADS, moe_slot_h, out_of_bound_fraction


def np_silu(z):
    # sigmoid via tanh: sigma(z) = (1 + tanh(z / 2)) / 2
    return z * (1.0 + np.tanh(z / 2.0)) / 2.0


def np_silu_prime(z):
    s = (1.0 + np.tanh(z / 2.0)) / 2.0
    return s * (1.0 + z * (1.0 - s))


def first_order_h_tol(g, u, Sg, Su):
    """1e-3 (|SiLU'(g)| |u| Sg + |SiLU(g)| Su) + 2^-11 |h| + 2^-24."""
    h = np_silu(g) * u
    return 1e-3 * (np.abs(np_silu_prime(g)) * np.abs(u) * Sg + np.abs(np_silu(g)) * Su) + \
        2.0 ** -11 * np.abs(h) + 2.0 ** -24


def silu_prime_root():
    """The zero of SiLU' on the negative axis, by bisection on central differences
    of SiLU (no use of the oracle)."""
    def d(z, e=1e-6):
        return (np_silu(z + e) - np_silu(z - e)) / (2 * e)
    a, b = -2.0, -1.0          # d(-2) < 0 < d(-1)
    for _ in range(80):
        m = 0.5 * (a + b)
        if d(m) < 0:
            a = m
        else:
            b = m
    return 0.5 * (a + b)


def test_silu_prime_closed_forms(oracle_lib):
    assert oracle_lib.silu_prime(0.0) == 0.5
    assert abs(oracle_lib.silu_prime(40.0) - 1.0) < 1e-15
    assert abs(oracle_lib.silu_prime(-40.0)) < 1e-15
    # central differences of SiLU
    for z in (-6.0, -2.4, -1.0, 0.3, 1.7, 5.0):
        e = 1e-5
        num = (np_silu(z + e) - np_silu(z - e)) / (2 * e)
        assert abs(oracle_lib.silu_prime(z) - num) < 1e-9
    z0 = silu_prime_root()
    assert -1.29 < z0 < -1.27
    assert abs(oracle_lib.silu_prime(z0)) < 1e-9
    # one sign change of SiLU' on a fine grid (the bound relies on a single
    # critical point)
    z = np.linspace(-30, 40, 700001)
    pos = np_silu_prime(z) > 0
    assert np.count_nonzero(pos[1:] != pos[:-1]) == 1


# g near the zero of SiLU' (-1.2785), at its minimum (-2.3994), and elsewhere
H_POINTS = [(g, u, Sg, Su)
            for g in (-1.2785, -2.3994, -6.0, -0.4, 0.5, 2.0, 8.0)
            for u in (-2.0, 0.3, 1.5)
            for Sg, Su in ((1.0, 1.0), (10.0, 40.0), (100.0, 20.0), (400.0, 400.0))]


def test_h_bound_covers_every_perturbation(oracle_lib):
    """From below: |SiLU(g + dg) (u + du) - SiLU(g) u| <= bound for dg, du on a
    grid over their tolerance intervals (corners included), plus the f16
    rounding of the exact value."""
    for g, u, Sg, Su in H_POINTS:
        eg, eu = 1e-3 * Sg + 1e-6, 1e-3 * Su + 1e-6
        dg = np.linspace(-eg, eg, 41)[:, None]
        du = np.linspace(-eu, eu, 41)[None, :]
        h = np_silu(g) * u
        worst = np.max(np.abs(np_silu(g + dg) * (u + du) - h))
        b = oracle_lib.h_bound(g, u, Sg, Su)
        assert worst <= b, (g, u, Sg, Su, worst, b)
        h16 = float(np.float16(h))
        assert abs(h16 - h) <= b


# Gate and up read the same x through matrices of the same distribution, so
# Sg ~ Su; at the FFN config Sg is about 33 (5120 terms of |w||x| ~ 0.0065).
H_POINTS_TYPICAL = [(g, u, Sg, Su)
                    for g in (-1.2785, -2.3994, -6.0, -0.4, 0.5, 2.0, 8.0)
                    for u in (-2.0, 0.3, 1.5)
                    for Sg, Su in ((1.0, 1.0), (10.0, 12.0), (40.0, 35.0), (100.0, 90.0))]


def test_h_bound_at_most_first_order_formula(oracle_lib):
    """From above: within 1.5x of the first-order formula at typical points (so
    a bound 10x looser, or one using max |SiLU'| instead of SiLU'(g), fails).
    With a much larger error on g than on u the curvature of SiLU matters and
    the first-order formula is no bound at all; there only the brute-force check
    above applies."""
    for g, u, Sg, Su in H_POINTS_TYPICAL:
        b = float(oracle_lib.h_bound(g, u, Sg, Su))
        f = float(first_order_h_tol(g, u, Sg, Su))
        assert b <= 1.5 * f, (g, u, Sg, Su, b, f)
        assert b >= f * (1 - 1e-9), (g, u, Sg, Su, b, f)
    # at the zero of SiLU' the gate's error enters at second order only:
    # SiLU(z0 +- e) - SiLU(z0) ~ SiLU''(z0) e^2 / 2, SiLU''(z0) ~ 0.2175
    z0 = silu_prime_root()
    b = float(oracle_lib.h_bound(z0, 1.0, 100.0, 0.0))
    eg = 0.1 + 1e-6
    assert b <= 0.12 * eg * eg + abs(np_silu(z0)) * 1.1e-6 + \
        2.0 ** -11 * (abs(np_silu(z0)) + 0.01) + 2.0 ** -24 + 1e-6


def _dense(qtype, q, s, oracle_lib):
    return oracle_lib.dequant(qtype, q, s)


def first_order_moe_bound(case, oracle_lib, h_in=None):
    """numpy propagation of the product tolerance through one MoE layer:
    sum_j |rw_j| * sum_i |D_ri| (th_i + 1e-3 |h_i|), th the first-order h
    tolerance (0 when the down projection takes given h values)."""
    t, E, ffn, hid = case["qtype"], case["n_expert"], case["ffn"], case["hidden"]
    ncols, topk = case["ncols"], case["topk"]
    out = np.zeros((ncols, hid))
    for c in range(ncols):
        x = case["x"][c].view(np.float16).astype(np.float64)
        for j in range(topk + 1):
            if j < topk:
                e = int(case["ids"][c][j])
                if e < 0 or e >= E:
                    continue
                r = slice(e * ffn, (e + 1) * ffn)
                rd = slice(e * hid, (e + 1) * hid)
                G = _dense(t, case["qg"][r], case["sg"][r], oracle_lib)
                U = _dense(t, case["qu"][r], case["su"][r], oracle_lib)
                D = _dense(t, case["qd"][rd], case["sd"][rd], oracle_lib)
                w = float(case["rw"][c][j])
            else:
                if case.get("shared") is None:
                    continue
                s = case["shared"]
                G = _dense(t, s["qg"], s["sg"], oracle_lib)
                U = _dense(t, s["qu"], s["su"], oracle_lib)
                D = _dense(t, s["qd"], s["sd"], oracle_lib)
                w = 1.0
            if h_in is None:
                g, u = G @ x, U @ x
                Sg, Su = np.abs(G) @ np.abs(x), np.abs(U) @ np.abs(x)
                h = np_silu(g) * u
                th = first_order_h_tol(g, u, Sg, Su)
            else:
                h = h_in[c, j].view(np.float16).astype(np.float64)
                th = 0.0
            out[c] += abs(w) * (np.abs(D) @ (th + 1e-3 * np.abs(h)))
    return out


def _mutations(case):
    """Three wrong routed combines, each with the size of its change of routing
    weight per column: each column's first routed expert dropped (rw[0]), uniform
    weights 1/topk (sum |1/topk - rw|), the first and last weights swapped
    (|rw[0] - rw[-1]|)."""
    rw = case["rw"].astype(np.float64)
    drop = case["ids"].copy()
    drop[:, 0] = -1
    uni = np.full_like(case["rw"], 1.0 / case["topk"])
    sw = case["rw"].copy()
    sw[:, [0, -1]] = sw[:, [-1, 0]]
    return {"dropped first expert": (dict(case, ids=drop), rw[:, 0]),
            "uniform weights": (dict(case, rw=uni), np.abs(1.0 / case["topk"] - rw).sum(1)),
            "first and last weights swapped": (dict(case, rw=sw), np.abs(rw[:, 0] - rw[:, -1]))}


def test_moe_bounds_first_order_small(oracle_lib):
    """End to end and staged, the oracle's MoE bound lies between 0.9x and 1.5x
    of the first-order numpy propagation."""
    case = synth.moe_case(synth.Q4_0, 6, 64, 96, 3, topk=2, shared=True, residual=True, seed=21)
    y, bound, _, _, rc = oracle_lib.moe(case)
    assert rc == 0
    f = first_order_moe_bound(case, oracle_lib) + 1e-6
    assert np.all(bound <= 1.5 * f + 1e-5) and np.all(bound >= 0.9 * f)
    h, _, _ = moe_slot_h(case)
    h16 = h.astype(np.float16).view(np.uint16)
    ys, bs, _, _, _ = oracle_lib.moe(case, h_in=h16)
    fs = first_order_moe_bound(case, oracle_lib, h_in=h16) + 1e-6
    assert np.all(bs <= 1.5 * fs + 1e-5) and np.all(bs >= 0.9 * fs)


def test_bounds_reject_wrong_combines_small(oracle_lib):
    """At a small shape the end-to-end bound already rejects each mutation (on
    a good share of the elements: a dropped expert whose softmax weight is small
    moves some outputs by less than the bound)."""
    case = synth.moe_case(synth.Q8_0, 12, 64, 128, 4, topk=4, shared=True, residual=False, seed=22)
    y, bound, _, _, _ = oracle_lib.moe(case)
    for what, (mut, _) in _mutations(case).items():
        ym, _, _, _, _ = oracle_lib.moe(mut)
        assert out_of_bound_fraction(ym, y, bound) > 0.2, what


@pytest.mark.parametrize("ncols", [1, 8])
def test_staged_bound_rejects_wrong_combines_at_expert_shape(oracle_lib, ncols):
    """The layer's per-expert shape (ffn 512, hidden 2048, top-8 + shared, Q8_0),
    with a 16-expert stack. The staged check (the down projection fed the f16 h
    of every slot, here the oracle's own h rounded to f16 in place of the GPU's)
    rejects each mutation on a large share of the output, and on most elements
    of every column whose routing weights it moves by 0.03 or more (a smaller
    change, e.g. swapping two nearly equal weights, is inside any tolerance).
    The end-to-end bound, which carries the h tolerance through the down
    projection, is looser than |y| at this shape and rejects almost nothing."""
    case = synth.moe_layer(ncols, seed=23, n_expert=16)
    h, _, _ = moe_slot_h(case, nthreads=NTHREADS)
    h16 = h.astype(np.float16).view(np.uint16)
    ys, bs, _, _, _ = oracle_lib.moe(case, h_in=h16, nthreads=NTHREADS)
    assert np.median(bs / np.abs(ys)) < 0.05
    _, be, _, _, _ = oracle_lib.moe(case, nthreads=NTHREADS)
    assert np.median(be / np.abs(ys)) > 0.5
    for what, (mut, change) in _mutations(case).items():
        ym, _, _, _, _ = oracle_lib.moe(mut, h_in=h16, nthreads=NTHREADS)
        assert out_of_bound_fraction(ym, ys, bs) > 0.3, what
        for c in range(ncols):
            if change[c] >= 0.03:
                assert out_of_bound_fraction(ym[c], ys[c], bs[c]) > 0.3, (what, c, change[c])


def test_ffn_bound_rejects_swapped_gate_and_up(oracle_lib):
    """The end-to-end FFN bound (h tolerance carried through |D|) rejects an FFN
    that applies SiLU to the up projection instead of the gate."""
    c = synth.ffn_case(synth.Q4_0, 128, 96, 4, seed=24)
    h, g, u, Sg, Su = oracle_lib.ffn_gate_up_silu(c["qtype"], c["qg"], c["sg"], c["qu"], c["su"],
                                                  c["x"])
    D = oracle_lib.dequant(c["qtype"], c["qd"], c["sd"])
    th = oracle_lib.h_bound(g, u, Sg, Su)
    ref = c["y0"].astype(np.float64) + h @ D.T
    bound = (th + 1e-3 * (np.abs(h) + th)) @ np.abs(D).T + 1e-6
    wrong = c["y0"].astype(np.float64) + (np_silu(u) * g) @ D.T
    assert out_of_bound_fraction(wrong, ref, bound) > 0.5
    assert out_of_bound_fraction(ref + 0.5 * bound, ref, bound) == 0.0
    assert math.isfinite(float(bound.max()))
