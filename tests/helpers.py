"""Shared helpers of the GPU parity tests: device upload, tolerance checks."""
import os

import numpy as np

NTHREADS = max(1, min(32, os.cpu_count() or 1))


def dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_u16_as_f16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.float16)


def dev_u16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def kernel_layout(qtype, q, scl):
    """The library's stored layout of a matrix given as GGUF-order split arrays:
    the oracle's repack of its GGUF blocks. Stacked expert matrices pass as one
    tall matrix. Returns (quants, scales)."""
    import oracle
    import synth
    q = np.ascontiguousarray(q)
    rows, nb = scl.shape[0] if scl.ndim == 2 else scl.shape[0] * scl.shape[1], scl.shape[-1]
    q2 = q.reshape(rows, -1)
    s2 = np.ascontiguousarray(scl).reshape(rows, nb)
    qr, sr = oracle.repack(qtype, synth.to_gguf_blocks(qtype, q2, s2), rows, nb * 32)
    return qr.reshape(q.shape), sr.reshape(scl.shape)


def dev_q(qtype, q, scl):
    """Device copies (quants, scales) of a GGUF-order matrix in the library's layout."""
    qr, sr = kernel_layout(qtype, q, scl)
    return dev(qr), dev_u16(sr)


def host(t):
    return t.detach().cpu().numpy()


def assert_within(got, ref, bound, what=""):
    """|got - ref| <= bound elementwise (all f64), with a readable failure."""
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        i = tuple(int(v) for v in i)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first {i}: "
            f"got {got[i]!r} ref {ref[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}")


def gemv_bound(S):
    """The product tolerance: |y_gpu - y_ref| <= 1e-3 * sum_k |w_k||x_k| + 1e-6."""
    return 1e-3 * S + 1e-6


def moe_slot_h(case, ids=None, nthreads=1):
    """Reference intermediate h of every (column, slot) of a MoE layer, in the
    workspace order the library documents: f64 [ncols][topk + 1][ffn], slot
    topk being the shared expert. Returns (h, bound, valid): bound is the
    oracle's h tolerance per element, valid marks the slots the layer computes
    (ids inside [0, n_expert), and the shared slot when there is a shared
    expert). Each slot is the oracle's fused gate/up of that expert's slices
    of the stacks on that column."""
    import oracle
    t, E, ffn = case["qtype"], case["n_expert"], case["ffn"]
    ncols, topk = case["ncols"], case["topk"]
    ids = case["ids"] if ids is None else ids
    h = np.zeros((ncols, topk + 1, ffn))
    bound = np.zeros_like(h)
    valid = np.zeros((ncols, topk + 1), dtype=bool)

    def slices(e):
        if e == E:
            s = case["shared"]
            return s["qg"], s["sg"], s["qu"], s["su"]
        r = slice(e * ffn, (e + 1) * ffn)
        return case["qg"][r], case["sg"][r], case["qu"][r], case["su"][r]
    for c in range(ncols):
        for j in range(topk + 1):
            if j < topk:
                e = int(ids[c][j])
                if e < 0 or e >= E:
                    continue
            elif case.get("shared") is None:
                continue
            else:
                e = E
            hh, g, u, Sg, Su = oracle.ffn_gate_up_silu(t, *slices(e), case["x"][c:c + 1],
                                                       nthreads=nthreads)
            h[c, j] = hh[0]
            bound[c, j] = oracle.h_bound(g[0], u[0], Sg[0], Su[0])
            valid[c, j] = True
    return h, bound, valid


def out_of_bound_fraction(got, ref, bound):
    """Fraction of elements with |got - ref| > bound."""
    err = np.abs(np.asarray(got, dtype=np.float64) - ref)
    return float(np.mean(~(err <= bound)))


def workspace_h(ws, case):
    """The layer's intermediate h as the header documents it: the workspace
    starts with f16 [ncols][topk + 1][ffn] (slot topk: the shared expert)."""
    n = case["ncols"] * (case["topk"] + 1) * case["ffn"]
    import torch
    return host(ws[:2 * n].view(torch.int16)).view(np.uint16).reshape(
        case["ncols"], case["topk"] + 1, case["ffn"]).copy()


def check_moe_staged(case, y, h_gpu, ids=None, what=""):
    """Stage by stage: (1) the GPU's h of every valid (column, slot) against the
    oracle's fused gate/up of that expert on that column, within the h bound;
    (2) the oracle's down projection and weighted combine fed the GPU's own h,
    at the plain down-projection tolerance 1e-6 + 1e-3 sum_j |rw_j| sum_i
    |D_ri| |h_i| (qref_moe with h_in), which a dropped expert, wrong weights or
    a wrong expert exceed."""
    import oracle
    href, hb, valid = moe_slot_h(case, ids=ids, nthreads=NTHREADS)
    with np.errstate(invalid="ignore"):  # slots of invalid ids hold unwritten bytes
        got_h = h_gpu.view(np.float16).astype(np.float64)
    assert np.isfinite(got_h[valid]).all(), what
    assert_within(got_h[valid], href[valid], hb[valid], what + " h per slot")
    ys, bs, _, _, _ = oracle.moe(case, h_in=h_gpu, ids=ids, nthreads=NTHREADS)
    assert_within(y, ys, bs, what + " (staged on the GPU's h)")
