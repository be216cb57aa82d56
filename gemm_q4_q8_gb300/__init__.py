"""Python binding of libqgemm (the C ABI in include/qgemm.h).

Argument marshalling only: every function takes torch tensors that already live
on the GPU, derives sizes from their shapes, passes raw device pointers and the
current CUDA stream to the C entry point of the same name, and raises
``QGError`` on a non-zero status. All arithmetic happens in the CUDA kernels of
the shared library; there is no other implementation to fall back to, and
loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

Q4_0 = 2
Q8_0 = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemm.so")

EXPORTS = ("qg_status_str", "qgemv_q4_0", "qgemv_q8_0", "qgemm_cols", "qffn_gate_up_silu",
           "qmoe_workspace_bytes", "qmoe_experts", "qmoe_experts_noalloc", "qrepack",
           "qargmax_f32", "qtopk_f32", "qmoe_router", "qg_kernel_launches", "qg_device_error",
           "qg_wait_selftest", "qg_last_cuda_error", "qg_last_cuda_error_string")

QG_MOE_NOALLOC_WS_BYTES = 1 << 20

# qg_status values (include/qgemm.h)
QG_OK, QG_ERR_NULL, QG_ERR_SHAPE, QG_ERR_ALIGN, QG_ERR_TYPE = 0, 1, 2, 3, 4
QG_ERR_WORKSPACE, QG_ERR_CUDA, QG_ERR_ALIAS = 5, 6, 7
STATUS = {QG_OK: "QG_OK", QG_ERR_NULL: "QG_ERR_NULL", QG_ERR_SHAPE: "QG_ERR_SHAPE",
          QG_ERR_ALIGN: "QG_ERR_ALIGN", QG_ERR_TYPE: "QG_ERR_TYPE",
          QG_ERR_WORKSPACE: "QG_ERR_WORKSPACE", QG_ERR_CUDA: "QG_ERR_CUDA",
          QG_ERR_ALIAS: "QG_ERR_ALIAS"}


class QGError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


class QGExpert(C.Structure):
    _fields_ = [("qg", C.c_void_p), ("sg", C.c_void_p), ("qu", C.c_void_p),
                ("su", C.c_void_p), ("qd", C.c_void_p), ("sd", C.c_void_p)]


_lib = None


def load(path: str | None = None):
    """Load libqgemm.so (built by ``gemm_q4_q8_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libqgemm.so not built ({path}); run gemm_q4_q8_gb300.build.build()")
    L = C.CDLL(path)
    vp, i32, sz = C.c_void_p, C.c_int, C.c_size_t
    L.qg_status_str.argtypes = [i32]
    L.qg_status_str.restype = C.c_char_p
    gemv = [vp, vp, i32, i32, vp, i32, vp, vp, vp]
    L.qgemv_q4_0.argtypes = gemv
    L.qgemv_q8_0.argtypes = gemv
    L.qgemm_cols.argtypes = [i32] + gemv
    L.qffn_gate_up_silu.argtypes = [i32, vp, vp, vp, vp, i32, i32, vp, i32, vp, vp]
    L.qmoe_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.qmoe_workspace_bytes.restype = sz
    L.qmoe_experts.argtypes = [i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32,
                               C.POINTER(QGExpert), vp, i32, vp, vp, vp, sz, vp, vp, vp]
    L.qmoe_experts_noalloc.argtypes = [i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, i32,
                                       C.POINTER(QGExpert), vp, i32, vp, vp, vp, vp, vp]
    L.qrepack.argtypes = [i32, vp, i32, i32, vp, vp, vp]
    L.qargmax_f32.argtypes = [vp, i32, i32, vp, vp, vp]
    L.qtopk_f32.argtypes = [vp, i32, i32, i32, vp, vp, vp]
    L.qmoe_router.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp]
    L.qg_kernel_launches.argtypes = []
    L.qg_kernel_launches.restype = C.c_uint64
    L.qg_device_error.argtypes = [C.POINTER(C.c_int32)]
    L.qg_wait_selftest.argtypes = [C.POINTER(C.c_int32), vp]
    L.qg_last_cuda_error.argtypes = []
    L.qg_last_cuda_error_string.argtypes = []
    L.qg_last_cuda_error_string.restype = C.c_char_p
    for f in EXPORTS:
        if f not in ("qg_status_str", "qmoe_workspace_bytes", "qg_kernel_launches",
                     "qg_last_cuda_error_string"):
            getattr(L, f).restype = i32
    _lib = L
    return L


def _check(fn: str, st: int):
    if st != 0:
        msg = load().qg_status_str(st).decode()
        if st == QG_ERR_CUDA:  # name the CUDA error behind it
            msg += ": " + load().qg_last_cuda_error_string().decode()
        raise QGError(fn, st, msg)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def qgemv_q4_0(nib, scl, x, y, y0=None, stream=None):
    """y[c] = y0[c] + W x[c]; nib uint8 [rows, k/2], scl f16-bits [rows, k/32],
    x f16 [ncols, k] (1..8 columns), y / y0 f32 [ncols, rows]."""
    rows, k = scl.shape[0], scl.shape[1] * 32
    _check("qgemv_q4_0", load().qgemv_q4_0(_ptr(nib), _ptr(scl), rows, k, _ptr(x), x.shape[0],
                                           _ptr(y0), _ptr(y), _stream(stream)))


def qgemv_q8_0(qs, scl, x, y, y0=None, stream=None):
    """As qgemv_q4_0 with int8 quants qs [rows, k]."""
    rows, k = scl.shape[0], scl.shape[1] * 32
    _check("qgemv_q8_0", load().qgemv_q8_0(_ptr(qs), _ptr(scl), rows, k, _ptr(x), x.shape[0],
                                           _ptr(y0), _ptr(y), _stream(stream)))


def qgemm_cols(qtype, q, scl, x, y, y0=None, stream=None):
    """y[c] = y0[c] + W x[c] for 1..16 columns."""
    rows, k = scl.shape[0], scl.shape[1] * 32
    _check("qgemm_cols", load().qgemm_cols(int(qtype), _ptr(q), _ptr(scl), rows, k, _ptr(x),
                                           x.shape[0], _ptr(y0), _ptr(y), _stream(stream)))


def qffn_gate_up_silu(qtype, qg, sg, qu, su, x, h, stream=None):
    """h[c] = f16(SiLU(Wg x[c]) * (Wu x[c])), h f16 [ncols, rows], 1..16 columns."""
    rows, k = sg.shape[0], sg.shape[1] * 32
    _check("qffn_gate_up_silu",
           load().qffn_gate_up_silu(int(qtype), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), rows, k,
                                    _ptr(x), x.shape[0], _ptr(h), _stream(stream)))


def qmoe_workspace_bytes(n_expert, ffn, hidden, ncols, topk) -> int:
    return int(load().qmoe_workspace_bytes(n_expert, ffn, hidden, ncols, topk))


def qmoe_experts(qtype, qg, sg, qu, su, qd, sd, n_expert, ffn, hidden, ids, rw, x, y,
                 ws, y0=None, shared=None, err_flag=None, uniq_ids_out=None, stream=None):
    """Stacked-expert MoE layer; ``shared`` is None or a dict with keys
    qg, sg, qu, su, qd, sd (device tensors)."""
    sh = None
    if shared is not None:
        sh = C.pointer(QGExpert(*[_ptr(shared[n]) for n in ("qg", "sg", "qu", "su", "qd", "sd")]))
    ncols, topk = ids.shape
    _check("qmoe_experts",
           load().qmoe_experts(int(qtype), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su), _ptr(qd),
                               _ptr(sd), n_expert, ffn, hidden, _ptr(ids), _ptr(rw), topk, sh,
                               _ptr(x), ncols, _ptr(y0), _ptr(y), _ptr(ws),
                               ws.numel() * ws.element_size(), _ptr(err_flag),
                               _ptr(uniq_ids_out), _stream(stream)))


def qmoe_experts_noalloc(qtype, qg, sg, qu, su, qd, sd, n_expert, ffn, hidden, ids, rw, x, y,
                         y0=None, shared=None, err_flag=None, uniq_ids_out=None, stream=None):
    """qmoe_experts with the library's built-in workspace of QG_MOE_NOALLOC_WS_BYTES
    (no caller allocation): for callers that cannot allocate device memory. Every
    shape qmoe_experts accepts fits; calls that overlap on the GPU race on the
    shared workspace."""
    sh = None
    if shared is not None:
        sh = C.pointer(QGExpert(*[_ptr(shared[n]) for n in ("qg", "sg", "qu", "su", "qd", "sd")]))
    ncols, topk = ids.shape
    _check("qmoe_experts_noalloc",
           load().qmoe_experts_noalloc(int(qtype), _ptr(qg), _ptr(sg), _ptr(qu), _ptr(su),
                                       _ptr(qd), _ptr(sd), n_expert, ffn, hidden, _ptr(ids),
                                       _ptr(rw), topk, sh, _ptr(x), ncols, _ptr(y0), _ptr(y),
                                       _ptr(err_flag), _ptr(uniq_ids_out), _stream(stream)))


def qg_kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(load().qg_kernel_launches())


QG_DEV_ERR_WAIT = 1


def qg_device_error() -> int:
    """The current device's error word, then cleared (0: no error; bit
    QG_DEV_ERR_WAIT: a tensor-core kernel gave up a wait, so some call since
    the last read returned wrong outputs). Synchronises the device."""
    v = C.c_int32(0)
    _check("qg_device_error", load().qg_device_error(C.byref(v)))
    return int(v.value)


def qg_wait_selftest(stream=None) -> tuple[int, int]:
    """Run the bounded-wait self-test (about 4 s): two waits on an mbarrier
    phase that nothing completes, CTA scope then cluster scope. Returns per
    wait 1 if it completed, 0 if it gave up (both 0 when the bounds work);
    each wait that gives up sets QG_DEV_ERR_WAIT in the device error word."""
    v = (C.c_int32 * 2)()
    _check("qg_wait_selftest", load().qg_wait_selftest(v, _stream(stream)))
    return int(v[0]), int(v[1])


def qrepack(qtype, gguf, rows, k, q_out, scl_out, stream=None):
    """GGUF interleaved blocks (device bytes) -> quant and scale arrays."""
    _check("qrepack", load().qrepack(int(qtype), _ptr(gguf), rows, k, _ptr(q_out), _ptr(scl_out),
                                     _stream(stream)))


def qargmax_f32(x, idx_out, val_out=None, stream=None):
    """Greedy argmax of each row of f32 x [ncols, n] (numbers before NaN, larger
    first, ties by lower index): idx_out int32 [ncols], val_out f32 [ncols] or None."""
    ncols, n = x.shape
    _check("qargmax_f32", load().qargmax_f32(_ptr(x), n, ncols, _ptr(idx_out), _ptr(val_out),
                                             _stream(stream)))


def qtopk_f32(x, k, idx_out, val_out=None, stream=None):
    """The k first-ranked elements of each row of f32 x [ncols, n], in rank order
    (the argmax order): idx_out int32 [ncols, k], val_out f32 [ncols, k] or None."""
    ncols, n = x.shape
    _check("qtopk_f32", load().qtopk_f32(_ptr(x), n, ncols, int(k), _ptr(idx_out), _ptr(val_out),
                                         _stream(stream)))


def qmoe_router(w_router, x, topk, ids_out, rw_out, logits_out=None, stream=None):
    """MoE router: w_router f32 [n_expert, hidden], x f16 [ncols, hidden] ->
    ids_out int32 [ncols, topk] (largest logits, lowest id on ties), rw_out f32
    [ncols, topk] (softmax over them), logits_out None or f32 [ncols, n_expert]."""
    n_expert, hidden = w_router.shape
    _check("qmoe_router", load().qmoe_router(_ptr(w_router), _ptr(x), n_expert, hidden, x.shape[0],
                                             int(topk), _ptr(logits_out), _ptr(ids_out),
                                             _ptr(rw_out), _stream(stream)))
