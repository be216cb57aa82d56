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
