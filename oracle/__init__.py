"""CPU oracle for the Q4_0 / Q8_0 block-quantised products (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It wraps ``qref.c`` (plain C, f64, k-order
loops) through ctypes and shares nothing with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qref.c")
_LIB = os.path.join(_HERE, "libqref.so")

Q4_0 = 2
Q8_0 = 8

_lib = None


def build(force: bool = False) -> str:
    """Compile qref.c with the host C compiler (no CUDA involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC,
                               "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Expert(C.Structure):
    _fields_ = [("qg", C.c_void_p), ("sg", C.c_void_p), ("qu", C.c_void_p),
                ("su", C.c_void_p), ("qd", C.c_void_p), ("sd", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        vp, i32, i64, dp = C.c_void_p, C.c_int, C.c_int64, C.c_void_p
        L.qref_f16_to_f64.argtypes = [C.c_uint16]
        L.qref_f16_to_f64.restype = C.c_double
        L.qref_silu.argtypes = [C.c_double]
        L.qref_silu.restype = C.c_double
        L.qref_silu_prime.argtypes = [C.c_double]
        L.qref_silu_prime.restype = C.c_double
        L.qref_h_bound.argtypes = [C.c_double] * 4
        L.qref_h_bound.restype = C.c_double
        L.qref_dequant_row.argtypes = [i32, vp, vp, i32, dp]
        L.qref_matmul.argtypes = [i32, vp, vp, i32, i32, vp, i32, vp, dp, dp, i32]
        L.qref_matmul_rows.argtypes = [i32, vp, vp, i32, i32, vp, i32, vp, vp, i64,
                                       dp, dp, i32]
        L.qref_ffn_gate_up_silu.argtypes = [i32, vp, vp, vp, vp, i32, i32, vp, i32,
                                            dp, dp, dp, dp, dp, i32]
        L.qref_moe.argtypes = [i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32,
                               C.POINTER(_Expert), vp, i32, vp, vp, dp, dp, vp,
                               C.POINTER(C.c_int), i32]
        L.qref_repack.argtypes = [i32, vp, i32, i32, vp, vp]
        L.qref_argmax.argtypes = [vp, i32, i32, vp, vp]
        L.qref_topk.argtypes = [vp, i32, i32, i32, vp, vp]
        L.qref_router_logits.argtypes = [vp, vp, i32, i32, i32, dp, dp]
        L.qref_softmax.argtypes = [vp, i32, dp]
        for f in ("qref_dequant_row", "qref_matmul", "qref_matmul_rows",
                  "qref_ffn_gate_up_silu", "qref_moe", "qref_repack", "qref_argmax",
                  "qref_topk", "qref_router_logits", "qref_softmax"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def f16_to_f64(bits: int) -> float:
    return lib().qref_f16_to_f64(int(bits))


def silu(z: float) -> float:
    return lib().qref_silu(float(z))


def silu_prime(z: float) -> float:
    return lib().qref_silu_prime(float(z))


def h_bound(g, u, Sg, Su):
    f = np.vectorize(lambda a, b, c, d: lib().qref_h_bound(a, b, c, d))
    return f(g, u, Sg, Su)


def dequant_row(qtype: int, qrow: np.ndarray, srow: np.ndarray) -> np.ndarray:
    qrow = np.ascontiguousarray(qrow).view(np.uint8)
    srow = _c(srow, np.uint16)
    k = srow.size * 32
    w = np.empty(k, dtype=np.float64)
    rc = lib().qref_dequant_row(qtype, _p(qrow), _p(srow), k, _p(w))
    if rc:
        raise ValueError(f"qref_dequant_row rc={rc}")
    return w


def dequant(qtype: int, q: np.ndarray, scl: np.ndarray) -> np.ndarray:
    return np.stack([dequant_row(qtype, q[r], scl[r]) for r in range(q.shape[0])])


def matmul(qtype: int, q: np.ndarray, scl: np.ndarray, x: np.ndarray,
           y0: np.ndarray | None = None, rows_sel=None, nthreads: int = 1):
    """(y, S): y[c][r] = y0 + sum_k w[r][k] x[c][k] in f64; S = sum_k |w||x|.

    ``x`` holds f16 bit patterns [ncols, k]. With ``rows_sel`` only those rows
    are computed (outputs [ncols, len(rows_sel)])."""
    q = np.ascontiguousarray(q)
    scl = _c(scl, np.uint16)
    x = _c(np.atleast_2d(x), np.uint16)
    rows, k = scl.shape[0], scl.shape[1] * 32
    ncols = x.shape[0]
    assert x.shape[1] == k
    y0c = _c(y0, np.float32)
    if rows_sel is None:
        y = np.empty((ncols, rows), dtype=np.float64)
        S = np.empty_like(y)
        rc = lib().qref_matmul(qtype, _p(q), _p(scl), rows, k, _p(x), ncols, _p(y0c),
                               _p(y), _p(S), nthreads)
    else:
        sel = _c(rows_sel, np.int64)
        y = np.empty((ncols, sel.size), dtype=np.float64)
        S = np.empty_like(y)
        rc = lib().qref_matmul_rows(qtype, _p(q), _p(scl), rows, k, _p(x), ncols,
                                    _p(y0c), _p(sel), sel.size, _p(y), _p(S), nthreads)
    if rc:
        raise ValueError(f"qref_matmul rc={rc}")
    return y, S


def ffn_gate_up_silu(qtype, qg, sg, qu, su, x, nthreads: int = 1):
    """(h, g, u, Sg, Su), all f64 [ncols, rows]."""
    qg, qu = np.ascontiguousarray(qg), np.ascontiguousarray(qu)
    sg, su = _c(sg, np.uint16), _c(su, np.uint16)
    x = _c(np.atleast_2d(x), np.uint16)
    rows, k = sg.shape[0], sg.shape[1] * 32
    ncols = x.shape[0]
    outs = [np.empty((ncols, rows), dtype=np.float64) for _ in range(5)]
    rc = lib().qref_ffn_gate_up_silu(qtype, _p(qg), _p(sg), _p(qu), _p(su), rows, k,
                                     _p(x), ncols, *[_p(o) for o in outs], nthreads)
    if rc:
        raise ValueError(f"qref_ffn_gate_up_silu rc={rc}")
    return tuple(outs)


def moe(case: dict, h_in: np.ndarray | None = None, ids=None, nthreads: int = 1):
    """(y, bound, uniq, n_uniq, rc) for a stacked-expert layer (see qref.c)."""
    t = case["qtype"]
    E, ffn, hidden = case["n_expert"], case["ffn"], case["hidden"]
    ncols, topk = case["ncols"], case["topk"]
    ids = _c(case["ids"] if ids is None else ids, np.int32)
    rw = _c(case["rw"], np.float32)
    arrs = [np.ascontiguousarray(case[n]) for n in ("qg", "sg", "qu", "su", "qd", "sd")]
    sh = case.get("shared")
    shp = None
    keep = []
    if sh is not None:
        sarr = [np.ascontiguousarray(sh[n]) for n in ("qg", "sg", "qu", "su", "qd", "sd")]
        keep.append(sarr)
        shp = C.pointer(_Expert(*[a.ctypes.data for a in sarr]))
    x = _c(case["x"], np.uint16)
    y0 = _c(case.get("y0"), np.float32)
    hin = _c(h_in, np.uint16)
    y = np.empty((ncols, hidden), dtype=np.float64)
    bound = np.empty_like(y)
    uniq = np.empty(ncols * topk, dtype=np.int32)
    nu = C.c_int(0)
    rc = lib().qref_moe(t, *[_p(a) for a in arrs], E, ffn, hidden, _p(ids), _p(rw), topk,
                        shp, _p(x), ncols, _p(y0), _p(hin), _p(y), _p(bound), _p(uniq),
                        C.byref(nu), nthreads)
    if rc not in (0, 3):
        raise ValueError(f"qref_moe rc={rc}")
    return y, bound, uniq, nu.value, rc


def repack(qtype: int, gguf: np.ndarray, rows: int, k: int):
    gguf = np.ascontiguousarray(gguf, dtype=np.uint8)
    qb = 16 if qtype == Q4_0 else 32
    q = np.empty((rows, k // 32 * qb), dtype=np.uint8)
    s = np.empty((rows, k // 32), dtype=np.uint16)
    rc = lib().qref_repack(qtype, _p(gguf), rows, k, _p(q), _p(s))
    if rc:
        raise ValueError(f"qref_repack rc={rc}")
    if qtype == Q8_0:
        q = q.view(np.int8)
    return q, s


def argmax(x: np.ndarray):
    """Greedy argmax of each row of f32 x [ncols, n]: (idx int32 [ncols], val f32 [ncols]).
    Order: numbers before NaN, larger first, ties (and NaNs) by lower index."""
    x = _c(np.atleast_2d(x), np.float32)
    ncols, n = x.shape
    idx = np.empty(ncols, dtype=np.int32)
    val = np.empty(ncols, dtype=np.float32)
    rc = lib().qref_argmax(_p(x), n, ncols, _p(idx), _p(val))
    if rc:
        raise ValueError(f"qref_argmax rc={rc}")
    return idx, val


def topk(x: np.ndarray, k: int):
    """Top-k of each row of f32 x [ncols, n] in rank order (the argmax order):
    (idx int32 [ncols, k], val f32 [ncols, k])."""
    x = _c(np.atleast_2d(x), np.float32)
    ncols, n = x.shape
    idx = np.empty((ncols, k), dtype=np.int32)
    val = np.empty((ncols, k), dtype=np.float32)
    rc = lib().qref_topk(_p(x), n, ncols, k, _p(idx), _p(val))
    if rc:
        raise ValueError(f"qref_topk rc={rc}")
    return idx, val


def router_logits(w: np.ndarray, x: np.ndarray):
    """(logits, S) in f64 [ncols, E]: logits = W_router x per column (w f32 [E, hidden],
    x f16 bits [ncols, hidden]); S = sum |w||x| (for the product tolerance)."""
    w = _c(w, np.float32)
    x = _c(np.atleast_2d(x), np.uint16)
    E, hidden = w.shape
    ncols = x.shape[0]
    lg = np.empty((ncols, E), dtype=np.float64)
    S = np.empty_like(lg)
    rc = lib().qref_router_logits(_p(w), _p(x), E, hidden, ncols, _p(lg), _p(S))
    if rc:
        raise ValueError(f"qref_router_logits rc={rc}")
    return lg, S


def softmax(v: np.ndarray) -> np.ndarray:
    """f64 softmax of the f32 values v (1-D)."""
    v = _c(np.ravel(v), np.float32)
    out = np.empty(v.size, dtype=np.float64)
    rc = lib().qref_softmax(_p(v), v.size, _p(out))
    if rc:
        raise ValueError(f"qref_softmax rc={rc}")
    return out
