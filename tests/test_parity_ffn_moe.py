"""GPU parity of the fused gate/up, the 16-column prefill FFN, the MoE layer and
the repack against the oracle.

The f16 output h of the fused gate/up is checked against the oracle's f64
SiLU(g) * u with the propagated bound of the GEMV tolerance through SiLU * up
plus one f16 rounding. The down projection is checked twice: staged (the
oracle takes the GPU's own f16 h as input, plain GEMV tolerance) and end to end
(the oracle's f64 h, with the bound carried through). The MoE layer is checked
the same way: the h of every (column, slot) that the layer leaves in its
workspace against the oracle's gate/up of that expert, then the down projection
and weighted combine staged on the GPU's h (the check that sees a wrong routed
combine at the layer's shape), then end to end. MoE routing (the ascending list
of distinct experts) must match bit for bit.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import (NTHREADS, assert_within, check_moe_staged, dev, dev_q,
                     dev_u16_as_f16, gemv_bound, host, workspace_h)

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


def gpu_gate_up(qtype, qg_, sg, qu, su, x):
    rows = sg.shape[0]
    h = torch.full((x.shape[0], rows), float("nan"), dtype=torch.float16, device="cuda")
    qg.qffn_gate_up_silu(qtype, *dev_q(qtype, qg_, sg), *dev_q(qtype, qu, su), dev_u16_as_f16(x), h)
    torch.cuda.synchronize()
    return host(h.view(torch.int16)).view(np.uint16)


def check_gate_up(qtype, qg_, sg, qu, su, x, what):
    hb = gpu_gate_up(qtype, qg_, sg, qu, su, x)
    href, g, u, Sg, Su = oracle.ffn_gate_up_silu(qtype, qg_, sg, qu, su, x, nthreads=NTHREADS)
    bound = oracle.h_bound(g, u, Sg, Su)
    got = hb.view(np.float16).astype(np.float64)
    assert np.isfinite(got).all()
    assert_within(got, href, bound, what)
    return hb, href, g, u, Sg, Su


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k,ncols", [(1, 32, 1), (37, 96, 2), (300, 1024, 5), (1000, 2048, 16),
                                          (515, 768, 9)])
def test_gate_up_shapes(qtype, rows, k, ncols):
    g = synth.rng(rows * 7 + k)
    qg_, sg = synth.draw_matrix(g, qtype, rows, k)
    qu, su = synth.draw_matrix(g, qtype, rows, k)
    x = synth.draw_x(g, ncols, k)
    check_gate_up(qtype, qg_, sg, qu, su, x, f"gate/up {qtype} {rows}x{k} C={ncols}")


def test_prefill_ffn_16_columns():
    """Gate/up 17408x5120 (fused, SiLU * up in f16), then down 5120x17408 with
    y += into the f32 residual, 16 columns."""
    c = synth.prefill_ffn()
    hb, href, g, u, Sg, Su = check_gate_up(c["qtype"], c["qg"], c["sg"], c["qu"], c["su"], c["x"],
                                           "prefill gate/up 17408x5120 C=16")
    y = dev(c["y0"])
    qg.qgemm_cols(c["qtype"], *dev_q(c["qtype"], c["qd"], c["sd"]), dev_u16_as_f16(hb), y, y)
    torch.cuda.synchronize()
    got = host(y)
    # staged: the oracle down-projects the GPU's own h
    yr, S = oracle.matmul(c["qtype"], c["qd"], c["sd"], hb, c["y0"], nthreads=NTHREADS)
    assert_within(got, yr, gemv_bound(S), "prefill down (staged)")
    # end to end: the oracle's f64 h, bound carried through |D| (th + 1e-3 (|h| + th))
    D = np.stack([oracle.dequant_row(c["qtype"], c["qd"][r], c["sd"][r]) for r in range(c["hidden"])])
    th = oracle.h_bound(g, u, Sg, Su)
    ref = c["y0"].astype(np.float64) + href @ D.T
    bound = (th + 1e-3 * (np.abs(href) + th)) @ np.abs(D).T + 1e-6
    assert_within(got, ref, bound, "prefill FFN end to end")


def gpu_moe(case, ids=None, with_y0=True, nshared=True):
    t = case["qtype"]
    E, ffn, hidden, ncols, topk = (case["n_expert"], case["ffn"], case["hidden"], case["ncols"],
                                   case["topk"])
    ids = case["ids"] if ids is None else ids
    ws_bytes = qg.qmoe_workspace_bytes(E, ffn, hidden, ncols, topk)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    y = torch.full((ncols, hidden), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    uniq = torch.full((ncols * topk,), -7, dtype=torch.int32, device="cuda")
    sh = None
    if case.get("shared") is not None and nshared:
        s_ = case["shared"]
        sh = {}
        for a, b in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
            sh[a], sh[b] = dev_q(t, s_[a], s_[b])
    y0 = dev(case["y0"]) if (case.get("y0") is not None and with_y0) else None
    qg.qmoe_experts(t, *dev_q(t, case["qg"], case["sg"]), *dev_q(t, case["qu"], case["su"]),
                    *dev_q(t, case["qd"], case["sd"]), E, ffn, hidden,
                    dev(np.ascontiguousarray(ids, np.int32)), dev(case["rw"]),
                    dev_u16_as_f16(case["x"]), y, ws, y0=y0, shared=sh, err_flag=err,
                    uniq_ids_out=uniq)
    torch.cuda.synchronize()
    return host(y), int(host(err)[0]), host(uniq), workspace_h(ws, case)


def check_moe(case, ids=None, what=""):
    y, err, uniq, h_gpu = gpu_moe(case, ids)
    yr, bound, uref, nu, rc = oracle.moe(case, ids=ids, nthreads=NTHREADS)
    assert np.array_equal(uniq, uref), (what, uniq[:nu + 2], uref[:nu + 2])
    assert err == (1 if rc == 3 else 0)
    assert np.isfinite(y).all()
    check_moe_staged(case, y, h_gpu, ids=ids, what=what)
    assert_within(y, yr, bound, what + " (end to end)")
    return y, nu


@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_moe_layer(ncols):
    case = synth.moe_layer(ncols)
    y, nu = check_moe(case, what=f"MoE 256x top-8 + shared, C={ncols}")
    assert nu == len(np.unique(case["ids"]))


def test_moe_residual_and_no_shared():
    case = synth.moe_case(synth.Q4_0, 16, 64, 128, 5, topk=3, shared=False, residual=True, seed=3)
    check_moe(case, what="MoE Q4_0 no shared + y0")


def test_moe_duplicate_and_invalid_ids():
    case = synth.moe_case(synth.Q8_0, 12, 96, 160, 4, topk=4, shared=True, residual=True, seed=4)
    ids = case["ids"].copy()
    ids[0, 1] = ids[0, 0]          # duplicate inside a column: both slots count
    ids[1, 2] = 12                 # out of range
    ids[2, 0] = -1                 # negative
    ids[3, :] = ids[2, :]
    check_moe(case, ids=ids, what="MoE duplicates + invalid ids")


def test_moe_16_columns_top16():
    """The largest id list: 16 columns x top-16 = 256 slots, many shared experts."""
    case = synth.moe_case(synth.Q4_0, 40, 96, 256, 16, topk=16, shared=True, residual=True, seed=6)
    y, nu = check_moe(case, what="MoE 16 columns x top-16")
    assert nu == len(np.unique(case["ids"]))


def test_moe_two_columns_no_shared():
    """Two columns (the down projection stages its row slices in shared memory
    by bulk copies), Q4_0, no shared expert, a residual, a duplicate and an
    out-of-range id."""
    case = synth.moe_case(synth.Q4_0, 24, 256, 384, 2, topk=6, shared=False, residual=True,
                          seed=12)
    ids = case["ids"].copy()
    ids[0, 3] = ids[0, 1]
    ids[1, 5] = 24
    check_moe(case, ids=ids, what="MoE Q4_0, 2 columns, no shared expert")


@pytest.mark.parametrize("ncols", [1, 3])
def test_moe_wide_ffn(ncols):
    """ffn 1024 with top-8 and a shared expert: the down projection's row slices
    of all nine experts do not fit in shared memory beside h, so the down and
    combine run on the kernel that streams them through registers (at ffn 512
    they are staged in shared memory by bulk copies)."""
    case = synth.moe_case(synth.Q8_0, 12, 1024, 256, ncols, topk=8, shared=True, residual=True,
                          seed=7 + ncols)
    check_moe(case, what=f"MoE ffn 1024, top-8 + shared, C={ncols}")


def test_moe_topk_one_and_all_experts_shared():
    case = synth.moe_case(synth.Q8_0, 3, 64, 64, 8, topk=1, shared=True, residual=False, seed=5)
    check_moe(case, what="MoE topk=1, 3 experts, 8 columns")


@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_repack_bit_exact(qtype):
    rows, k = 333, 1056
    g = synth.rng(40)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    blocks = synth.to_gguf_blocks(qtype, q, s)
    qref, sref = oracle.repack(qtype, blocks, rows, k)
    qb = 16 if qtype == synth.Q4_0 else 32
    dq = torch.empty((rows, k // 32 * qb), dtype=torch.uint8, device="cuda")
    ds = torch.empty((rows, k // 32), dtype=torch.int16, device="cuda")
    qg.qrepack(qtype, dev(blocks), rows, k, dq, ds)
    torch.cuda.synchronize()
    assert np.array_equal(host(dq), qref.view(np.uint8))
    assert np.array_equal(host(ds).view(np.uint16), sref)
