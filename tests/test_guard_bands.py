"""Memory safety of every entry point without a device sanitizer: guard bands.

Each output buffer is carved out of a larger device allocation whose bytes
before and after it (GUARD each side) hold a fixed pattern. After the call the
bands must be untouched (no write outside the output), every output element
must have been written (outputs start as all-ones bytes: NaN for f16 and f32,
-1 for int32, values no call produces on these inputs), and every input must
be unchanged (no write into a read-only argument). The shapes cover each
kernel family and plan: CUDA-core and tensor-core GEMV with ragged row tails,
K-split clusters, 1/5/8/16 columns, the in-place residual, the fused gate/up,
the MoE layer on both down kernels and with the library's own workspace,
repack, argmax, top-k and the router."""
import numpy as np
import pytest

import synth
from helpers import dev, dev_q, dev_u16_as_f16


torch = pytest.importorskip("torch")

GUARD = 1 << 14   # bytes of guard band on each side of an output
BAND = 0xA5       # guard-band byte
UNSET = 0xFF      # initial byte of every output element


@pytest.fixture(scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gemm_q4_q8_gb300 import build
    build.build()
    import oracle
    oracle.build()  # the stored layout of the test matrices comes from the oracle's repack


import gemm_q4_q8_gb300 as qg  # noqa: E402


class Guarded:
    """A device tensor of `shape` and `dtype` inside a guard-banded allocation
    (the tensor starts GUARD bytes in, so a 256-byte aligned base stays
    aligned)."""

    def __init__(self, shape, dtype, device="cuda"):
        self.nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + self.nbytes,), BAND, dtype=torch.uint8, device=device)
        self.raw[GUARD:GUARD + self.nbytes] = UNSET
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def check(self, what, written=True):
        raw = self.raw.cpu().numpy()
        lo, hi = raw[:GUARD], raw[GUARD + self.nbytes:]
        assert (lo == BAND).all(), f"{what}: {int((lo != BAND).sum())} bytes written before the output"
        assert (hi == BAND).all(), f"{what}: {int((hi != BAND).sum())} bytes written after the output"
        if written:
            body = raw[GUARD:GUARD + self.nbytes]
            esz = self.t.element_size()
            unset = (body.reshape(-1, esz) == UNSET).all(axis=1)
            assert not unset.any(), f"{what}: {int(unset.sum())} output elements never written"


def snapshot(*ts):
    return [None if t is None else t.clone() for t in ts]


def unchanged(before, after, what):
    """Bitwise equality of every input with its copy taken before the call."""
    for i, (b, a) in enumerate(zip(before, after)):
        if b is not None:
            assert torch.equal(b.view(torch.uint8), a.view(torch.uint8)), f"{what}: input {i} changed"


GEMV_SHAPES = [
    (333, 1056),    # CUDA cores, K not a multiple of 256, ragged rows
    (200, 4128),    # CUDA cores, x staged in chunks for 5-8 columns
    (1000, 5120),   # tensor cores, 15 full 64-row tiles and a 40-row tail
    (130, 8192),    # tensor cores, K split over a cluster, 2-row tail
]


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k", GEMV_SHAPES)
@pytest.mark.parametrize("ncols", [1, 5, 8, 16])
@pytest.mark.parametrize("residual", ["none", "y0", "inplace"])
def test_gemv_guard_bands(qtype, rows, k, ncols, residual):
    g = synth.rng(rows * 7 + k + ncols)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    dq, ds = dev_q(qtype, q, s)
    x = dev_u16_as_f16(synth.draw_x(g, ncols, k))
    y = Guarded((ncols, rows), torch.float32)
    y0 = None
    if residual == "y0":
        y0 = dev(synth.draw_y0(g, ncols, rows))
    elif residual == "inplace":
        y.t.copy_(dev(synth.draw_y0(g, ncols, rows)))
        y0 = y.t
    before = snapshot(dq, ds, x, None if residual == "inplace" else y0)
    if ncols <= 8:
        fn = qg.qgemv_q4_0 if qtype == synth.Q4_0 else qg.qgemv_q8_0
        fn(dq, ds, x, y.t, y0)
    else:
        qg.qgemm_cols(qtype, dq, ds, x, y.t, y0)
    torch.cuda.synchronize()
    what = f"gemv {rows}x{k} c{ncols} {residual}"
    y.check(what)
    unchanged(before, [dq, ds, x, y0], what)
    assert torch.isfinite(y.t).all(), what


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
@pytest.mark.parametrize("rows,k", [(300, 1056), (1000, 5120)])
@pytest.mark.parametrize("ncols", [1, 8, 16])
def test_gate_up_guard_bands(qtype, rows, k, ncols):
    g = synth.rng(rows * 11 + k + ncols)
    qg_, sg = synth.draw_matrix(g, qtype, rows, k)
    qu, su = synth.draw_matrix(g, qtype, rows, k)
    dg, dsg = dev_q(qtype, qg_, sg)
    du, dsu = dev_q(qtype, qu, su)
    x = dev_u16_as_f16(synth.draw_x(g, ncols, k))
    h = Guarded((ncols, rows), torch.float16)
    before = snapshot(dg, dsg, du, dsu, x)
    qg.qffn_gate_up_silu(qtype, dg, dsg, du, dsu, x, h.t)
    torch.cuda.synchronize()
    what = f"gate/up {rows}x{k} c{ncols}"
    h.check(what)
    unchanged(before, [dg, dsg, du, dsu, x], what)


def _moe_dev(case):
    t = case["qtype"]
    a = {}
    for n, m in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
        a[n], a[m] = dev_q(t, case[n], case[m])
    sh = None
    if case.get("shared") is not None:
        sh = {}
        for n, m in (("qg", "sg"), ("qu", "su"), ("qd", "sd")):
            sh[n], sh[m] = dev_q(t, case["shared"][n], case["shared"][m])
    a["ids"] = dev(np.ascontiguousarray(case["ids"], np.int32))
    a["rw"] = dev(case["rw"])
    a["x"] = dev_u16_as_f16(case["x"])
    return a, sh


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("ncols", [1, 2, 8, 16])
@pytest.mark.parametrize("noalloc", [False, True])
def test_moe_guard_bands(ncols, noalloc):
    """ffn 512 takes the staged down kernel at 1-2 columns and the register one
    above; the workspace gets a guard band after its documented size."""
    case = synth.moe_case(synth.Q8_0, 24, 512, 1024, ncols, topk=8, shared=True, residual=True,
                          seed=50 + ncols)
    E, ffn, hidden, topk = case["n_expert"], case["ffn"], case["hidden"], case["topk"]
    a, sh = _moe_dev(case)
    y0 = dev(case["y0"])
    y = Guarded((ncols, hidden), torch.float32)
    uniq = Guarded((ncols * topk,), torch.int32)
    err = Guarded((1,), torch.int32)
    err.t.zero_()
    ins = [a[n] for n in ("qg", "sg", "qu", "su", "qd", "sd", "ids", "rw", "x")] + [y0] + \
        [sh[n] for n in ("qg", "sg", "qu", "su", "qd", "sd")]
    before = snapshot(*ins)
    common = (synth.Q8_0, a["qg"], a["sg"], a["qu"], a["su"], a["qd"], a["sd"], E, ffn, hidden,
              a["ids"], a["rw"], a["x"], y.t)
    ws = None
    if noalloc:
        qg.qmoe_experts_noalloc(*common, y0=y0, shared=sh, err_flag=err.t, uniq_ids_out=uniq.t)
    else:
        ws = Guarded((qg.qmoe_workspace_bytes(E, ffn, hidden, ncols, topk),), torch.uint8)
        qg.qmoe_experts(*common, ws.t, y0=y0, shared=sh, err_flag=err.t, uniq_ids_out=uniq.t)
    torch.cuda.synchronize()
    what = f"moe c{ncols} {'noalloc' if noalloc else 'workspace'}"
    y.check(what + " y")
    uniq.check(what + " uniq ids", written=False)
    err.check(what + " err flag", written=False)
    if ws is not None:
        ws.check(what + " workspace", written=False)
    unchanged(before, ins, what)
    assert int(err.t.item()) == 0
    u = uniq.t.cpu().numpy()
    ref = np.unique(case["ids"])
    assert np.array_equal(u[:ref.size], ref) and (u[ref.size:] == -1).all(), what
    assert torch.isfinite(y.t).all(), what


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("qtype", [synth.Q4_0, synth.Q8_0])
def test_repack_guard_bands(qtype):
    rows, k = 333, 1056
    g = synth.rng(60 + qtype)
    q, s = synth.draw_matrix(g, qtype, rows, k)
    blocks = dev(synth.to_gguf_blocks(qtype, q, s))
    qb = 16 if qtype == synth.Q4_0 else 32
    dq = Guarded((rows, k // 32 * qb), torch.uint8)
    ds = Guarded((rows, k // 32), torch.int16)
    before = snapshot(blocks)
    qg.qrepack(qtype, blocks, rows, k, dq.t, ds.t)
    torch.cuda.synchronize()
    # a stored byte may legitimately be 0xFF, so only the bands are checked here;
    # the repack parity test checks every byte
    dq.check("repack quants", written=False)
    ds.check("repack scales", written=False)
    unchanged(before, [blocks], "repack")


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("n,ncols", [(248320, 1), (248320, 8), (1001, 3), (5, 2)])
def test_sampling_guard_bands(n, ncols):
    g = np.random.Generator(np.random.PCG64(n + ncols))
    x = dev(g.standard_normal((ncols, n)).astype(np.float32))
    before = snapshot(x)
    idx = Guarded((ncols,), torch.int32)
    val = Guarded((ncols,), torch.float32)
    qg.qargmax_f32(x, idx.t, val.t)
    k = min(40, n)
    ti = Guarded((ncols, k), torch.int32)
    tv = Guarded((ncols, k), torch.float32)
    qg.qtopk_f32(x, k, ti.t, tv.t)
    torch.cuda.synchronize()
    for b, w in ((idx, "argmax idx"), (val, "argmax val"), (ti, "top-k idx"), (tv, "top-k val")):
        b.check(f"{w} n={n} c{ncols}")
    unchanged(before, [x], "sampling")
    assert ((ti.t >= 0) & (ti.t < n)).all()


@pytest.mark.gpu
@pytest.mark.usefixtures("_lib")
@pytest.mark.parametrize("E,hidden,ncols,k", [(256, 2048, 1, 8), (256, 2048, 16, 8), (60, 96, 3, 5),
                                              (7, 33, 2, 7)])
def test_router_guard_bands(E, hidden, ncols, k):
    g = np.random.Generator(np.random.PCG64(E + hidden + ncols))
    w = dev((g.standard_normal((E, hidden)) * 0.02).astype(np.float32))
    x = dev(g.standard_normal((ncols, hidden)).astype(np.float16))
    before = snapshot(w, x)
    lg = Guarded((ncols, E), torch.float32)
    ids = Guarded((ncols, k), torch.int32)
    rw = Guarded((ncols, k), torch.float32)
    qg.qmoe_router(w, x, k, ids.t, rw.t, logits_out=lg.t)
    torch.cuda.synchronize()
    for b, n in ((lg, "logits"), (ids, "ids"), (rw, "weights")):
        b.check(f"router {n} E={E} c{ncols}")
    unchanged(before, [w, x], "router")
    assert ((ids.t >= 0) & (ids.t < E)).all()


def test_guard_checker_catches_stray_and_missing_writes():
    """The checker itself, on host memory: a write one element before or after
    the output, or an output element left unwritten, each fails the check; a
    fully written output with intact bands passes."""
    for where in ("before", "after", "unwritten", "clean"):
        b = Guarded((3, 5), torch.float32, device="cpu")
        b.t.fill_(1.5)
        if where == "before":
            b.raw[GUARD - 4:GUARD] = 0
        elif where == "after":
            b.raw[GUARD + b.nbytes] = 0
        elif where == "unwritten":
            b.t.view(torch.int32)[2, 4] = -1
        if where == "clean":
            b.check(where)
        else:
            with pytest.raises(AssertionError):
                b.check(where)
    b = Guarded((4,), torch.int32, device="cpu")
    b.t.copy_(torch.tensor([0, -1, 7, 3], dtype=torch.int32))
    with pytest.raises(AssertionError):
        b.check("int -1 counts as unwritten")
    b.check("int -1 allowed when not checked for writes", written=False)
    x = torch.arange(6, dtype=torch.float16)
    before = snapshot(x)
    unchanged(before, [x], "same")
    x[3] = -x[3]
    with pytest.raises(AssertionError):
        unchanged(before, [x], "changed")
