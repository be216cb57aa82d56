"""qmoe_experts_noalloc: the MoE layer for callers that cannot allocate device
memory (a plugin inside a framework that owns every byte of device memory, a
fixed memory budget, a loop that must not call cudaMalloc). Its workspace is an
array inside the library. The GPU test calls it through the C ABI twice in a
row per case, the second call finding the first call's contents in the shared
array, and checks each output bit for bit against qmoe_experts with a
caller-allocated workspace: both run the same kernels on the same shape, and
the reduction order depends only on the shape. The oracle's MoE bound is kept
as a second check. This file is collected last so that a failure here stops a
run only after every other test has run."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_within, dev, dev_q, dev_u16_as_f16, host

torch = pytest.importorskip("torch")

import gemm_q4_q8_gb300 as qg  # noqa: E402


def _moe_args(case):
    t = case["qtype"]
    sh = None
    if case.get("shared") is not None:
        s_ = case["shared"]
        sh = {}
        for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
            sh[a], sh[b] = dev_q(t, s_[a], s_[b])
    y0 = dev(case["y0"]) if case.get("y0") is not None else None
    dqg, dsg = dev_q(t, case["qg"], case["sg"])
    dqu, dsu = dev_q(t, case["qu"], case["su"])
    dqd, dsd = dev_q(t, case["qd"], case["sd"])
    return dict(qg=dqg, sg=dsg, qu=dqu, su=dsu, qd=dqd, sd=dsd,
                ids=dev(np.ascontiguousarray(case["ids"], np.int32)), rw=dev(case["rw"]),
                x=dev_u16_as_f16(case["x"]), y0=y0, shared=sh)


def _run(case, a, noalloc):
    ncols, hidden = case["ncols"], case["hidden"]
    y = torch.full((ncols, hidden), float("nan"), dtype=torch.float32, device="cuda")
    uniq = torch.full((ncols * case["topk"],), -9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    common = (case["qtype"], a["qg"], a["sg"], a["qu"], a["su"], a["qd"], a["sd"],
              case["n_expert"], case["ffn"], hidden, a["ids"], a["rw"], a["x"], y)
    if noalloc:
        qg.qmoe_experts_noalloc(*common, y0=a["y0"], shared=a["shared"], err_flag=err,
                                uniq_ids_out=uniq)
    else:
        nb = qg.qmoe_workspace_bytes(case["n_expert"], case["ffn"], hidden, ncols, case["topk"])
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        qg.qmoe_experts(*common, ws, y0=a["y0"], shared=a["shared"], err_flag=err,
                        uniq_ids_out=uniq)
    torch.cuda.synchronize()
    return host(y), host(uniq), int(host(err)[0])


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q4_q8_gb300 import build
    build.build()
    oracle.build()
    cases = [synth.moe_layer(8, seed=11),
             synth.moe_case(synth.Q4_0, 16, 64, 256, 5, topk=3, shared=True, residual=True,
                            seed=12)]
    # Per case, two noalloc calls back to back on the same library array (the
    # second finds the first's contents in it), and across cases the array
    # moves to a different shape.
    for case in cases:
        a = _moe_args(case)
        y_ws, u_ws, e_ws = _run(case, a, noalloc=False)
        _, bound, _, _, _ = oracle.moe(case)
        for call in (1, 2):
            y_na, u_na, e_na = _run(case, a, noalloc=True)
            assert np.array_equal(y_na.view(np.uint32), y_ws.view(np.uint32)), \
                f"noalloc call {call} differs from the workspace call"
            assert np.array_equal(u_na, u_ws) and e_na == e_ws == 0
            assert_within(y_na, oracle.moe(case)[0], bound, f"noalloc call {call} vs oracle")


@pytest.mark.gpu
def test_noalloc_at_its_largest_accepted_workspace():
    """16 columns x top-15 with ffn 2048 needs exactly the whole library array
    (1 MiB of h). Two calls in a row, each bit for bit equal to the workspace
    call (a 24-expert stack keeps the test small; the workspace does not depend
    on the number of experts)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q4_q8_gb300 import build
    build.build()
    case = synth.moe_case(synth.Q4_0, 24, 2048, 2048, 16, topk=15, shared=True, residual=True,
                          seed=13)
    assert qg.qmoe_workspace_bytes(24, 2048, 2048, 16, 15) == qg.QG_MOE_NOALLOC_WS_BYTES
    a = _moe_args(case)
    y_ws, u_ws, e_ws = _run(case, a, noalloc=False)
    assert np.isfinite(y_ws).all()
    for call in (1, 2):
        y_na, u_na, e_na = _run(case, a, noalloc=True)
        assert np.array_equal(y_na.view(np.uint32), y_ws.view(np.uint32)), call
        assert np.array_equal(u_na, u_ws) and e_na == e_ws == 0


def test_noalloc_workspace_holds_every_accepted_shape():
    """The library's array is as large as the largest workspace any accepted
    shape needs; shapes the MoE layer rejects get the same status from both
    entry points (nothing is launched: the checks run on the host first)."""
    from gemm_q4_q8_gb300 import build
    build.build()
    L = qg.load()
    # largest accepted: 16 columns, (topk + 1) * ffn = 32768 h values per column
    biggest = qg.qmoe_workspace_bytes(256, 2048, 2048, 16, 15)
    assert biggest == qg.QG_MOE_NOALLOC_WS_BYTES
    assert qg.qmoe_workspace_bytes(256, 32768 // 17 // 32 * 32, 2048, 16, 16) <= biggest
    # one step beyond in ffn, columns or top-k: rejected as a shape
    assert qg.qmoe_workspace_bytes(256, 2048 + 32, 2048, 16, 15) == 0
    assert qg.qmoe_workspace_bytes(256, 2048, 2048, 17, 15) == 0
    assert qg.qmoe_workspace_bytes(256, 2048, 2048, 16, 16) == 0
    p = 0x10000  # aligned, never dereferenced: the shape check comes first
    for shape in ((256, 2048 + 32, 2048, 15, 16), (256, 32768, 1024, 16, 8)):
        E, ffn, hidden, topk, ncols = shape
        st_na = L.qmoe_experts_noalloc(qg.Q8_0, p, p, p, p, p, p, E, ffn, hidden, p, p, topk,
                                       None, p, ncols, None, p, None, None, None)
        st_ws = L.qmoe_experts(qg.Q8_0, p, p, p, p, p, p, E, ffn, hidden, p, p, topk, None, p,
                               ncols, None, p, p, 1 << 30, None, None, None)
        assert st_na == st_ws == qg.QG_ERR_SHAPE
        assert L.qg_status_str(st_na).decode().startswith("invalid shape")
    st = L.qmoe_experts_noalloc(3, p, p, p, p, p, p, 256, 512, 2048, p, p, 8, None, p, 1, None, p,
                                None, None, None)
    assert st == qg.QG_ERR_TYPE
