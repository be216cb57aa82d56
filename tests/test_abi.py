"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function declared in include/qgemm.h, and rejects bad arguments with the
documented status codes before launching anything."""
import ctypes as C
import os
import re

import pytest

import gemm_q4_q8_gb300 as qg
from gemm_q4_q8_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qg.load()


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"\b(q[a-z0-9_]+)\s*\(", txt)
    return sorted(set(n for n in names if not n.startswith("qg_expert")))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in qg.EXPORTS:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"


def test_status_strings(lib):
    for code in range(8):
        s = lib.qg_status_str(code).decode()
        assert s and s != "unknown status"
    assert lib.qg_status_str(99).decode() == "unknown status"


ALIGNED = 0x10000  # a fake, 16-byte aligned address; never dereferenced


def gemv(lib, **kw):
    a = dict(q=ALIGNED, scl=ALIGNED, rows=64, k=64, x=ALIGNED, ncols=1, y0=None, y=ALIGNED + 0x100000)
    a.update(kw)
    return lib.qgemv_q4_0(a["q"], a["scl"], a["rows"], a["k"], a["x"], a["ncols"], a["y0"], a["y"], None)


def test_shape_errors(lib):
    assert gemv(lib, k=48) == 2
    assert gemv(lib, k=0) == 2
    assert gemv(lib, k=-32) == 2
    assert gemv(lib, rows=-1) == 2
    assert gemv(lib, ncols=0) == 2
    assert gemv(lib, ncols=9) == 2
    assert lib.qgemm_cols(2, ALIGNED, ALIGNED, 64, 64, ALIGNED, 17, None, ALIGNED, None) == 2
    assert lib.qffn_gate_up_silu(2, ALIGNED, ALIGNED, ALIGNED, ALIGNED, 64, 64, ALIGNED, 17, ALIGNED, None) == 2


def test_type_errors(lib):
    assert lib.qgemm_cols(3, ALIGNED, ALIGNED, 64, 64, ALIGNED, 1, None, ALIGNED, None) == 4
    assert lib.qrepack(7, ALIGNED, 4, 64, ALIGNED, ALIGNED, None) == 4


def test_null_errors(lib):
    assert gemv(lib, q=None) == 1
    assert gemv(lib, scl=None) == 1
    assert gemv(lib, x=None) == 1
    assert gemv(lib, y=None) == 1
    assert lib.qffn_gate_up_silu(2, ALIGNED, ALIGNED, None, ALIGNED, 64, 64, ALIGNED, 2, ALIGNED, None) == 1


def test_align_errors(lib):
    assert gemv(lib, q=ALIGNED + 8) == 3
    assert gemv(lib, scl=ALIGNED + 2) == 3
    assert gemv(lib, x=ALIGNED + 4) == 3
    assert gemv(lib, y=ALIGNED + 0x100002) == 3
    assert gemv(lib, y0=ALIGNED + 0x200001) == 3


def test_alias_error(lib):
    # y0 overlapping y without being equal to it
    assert gemv(lib, y0=ALIGNED + 0x100000 + 16) == 7


def test_empty_problem_is_ok(lib):
    assert gemv(lib, rows=0, q=None, scl=None, x=None, y=None) == 0
    assert lib.qrepack(2, None, 0, 64, None, None, None) == 0


def test_moe_argument_errors(lib):
    w = lib.qmoe_workspace_bytes(256, 512, 2048, 8, 8)
    assert w > 0
    assert lib.qmoe_workspace_bytes(256, 512, 2048, 16, 16) > 0
    assert lib.qmoe_workspace_bytes(256, 512, 2048, 17, 8) == 0
    assert lib.qmoe_workspace_bytes((1 << 22) + 1, 512, 2048, 1, 8) == 0

    def moe(**kw):
        a = dict(t=8, n_expert=4, ffn=64, hidden=64, topk=2, ncols=2, ws=ALIGNED, wsb=1 << 30,
                 ids=ALIGNED, y=ALIGNED)
        a.update(kw)
        return lib.qmoe_experts(a["t"], ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED, ALIGNED,
                                a["n_expert"], a["ffn"], a["hidden"], a["ids"], ALIGNED, a["topk"],
                                None, ALIGNED, a["ncols"], None, a["y"], a["ws"], a["wsb"], None,
                                None, None)
    assert moe(t=5) == 4
    assert moe(ncols=17) == 2
    assert moe(n_expert=(1 << 22) + 1) == 2
    assert moe(topk=0) == 2
    assert moe(topk=17) == 2
    assert moe(n_expert=0) == 2
    assert moe(ffn=48) == 2
    assert moe(ids=None) == 1
    assert moe(wsb=16) == 5
    assert moe(ws=None) == 5
    assert moe(ids=ALIGNED + 2) == 3


def test_valid_call_without_gpu_reports_cuda_error(lib):
    from conftest import gpu_available
    if gpu_available():
        pytest.skip("a GPU is present")
    # valid arguments: the library must fail loudly (no CPU fallback), and it
    # names the CUDA error behind QG_ERR_CUDA on this thread
    assert gemv(lib) == 6
    assert lib.qg_last_cuda_error() != 0
    assert lib.qg_last_cuda_error_string().decode().startswith("cudaError")


def test_wait_selftest_null_output(lib):
    """The self-test checks its output pointer before launching anything."""
    assert lib.qg_wait_selftest(None, None) == qg.QG_ERR_NULL


def test_device_error_word(lib):
    """qg_device_error: a null output is QG_ERR_NULL; without a GPU the read of
    the device word fails loudly (QG_ERR_CUDA)."""
    import ctypes as C
    from conftest import gpu_available
    assert lib.qg_device_error(None) == 1
    if not gpu_available():
        v = C.c_int32(-5)
        assert lib.qg_device_error(C.byref(v)) == 6 and v.value == -5


def test_sampling_argument_errors(lib):
    assert lib.qargmax_f32(ALIGNED, 0, 1, ALIGNED, None, None) == 2
    assert lib.qargmax_f32(ALIGNED, 10, 65, ALIGNED, None, None) == 2
    assert lib.qargmax_f32(None, 10, 1, ALIGNED, None, None) == 1
    assert lib.qargmax_f32(ALIGNED + 2, 10, 1, ALIGNED, None, None) == 3
    assert lib.qtopk_f32(ALIGNED, 10, 1, 11, ALIGNED, None, None) == 2
    assert lib.qtopk_f32(ALIGNED, 1000, 1, 257, ALIGNED, None, None) == 2
    assert lib.qtopk_f32(ALIGNED, 1000, 1, 0, ALIGNED, None, None) == 2
    assert lib.qtopk_f32(ALIGNED, 1000, 1, 5, None, None, None) == 1


def test_router_argument_errors(lib):
    def router(w=ALIGNED, x=ALIGNED, E=256, hidden=2048, ncols=1, topk=8, lg=None, ids=ALIGNED,
               rw=ALIGNED):
        return lib.qmoe_router(w, x, E, hidden, ncols, topk, lg, ids, rw, None)
    assert router(E=0) == 2
    assert router(E=1025) == 2
    assert router(ncols=17) == 2
    assert router(topk=33, E=64) == 2
    assert router(topk=9, E=8) == 2
    assert router(hidden=0) == 2
    assert router(w=None) == 1
    assert router(ids=None) == 1
    assert router(rw=None) == 1
    assert router(w=ALIGNED + 4) == 3
    assert router(x=ALIGNED + 1) == 3
    assert router(lg=ALIGNED + 2) == 3
    from conftest import gpu_available
    if not gpu_available():
        assert router() == 6
