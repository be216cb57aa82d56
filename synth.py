"""Seeded synthetic inputs for the Q4_0 / Q8_0 block-quantized products.

This module only draws random numbers and lays them out in the storage formats
the kernels and the oracle read. It performs none of the method's arithmetic
(no dequantisation, no dot products, no SiLU, no combine), so it can feed both
the CUDA path and the CPU oracle without linking them.

Storage formats (the block format of "Engine and kernels", pooled.run, section
"What it runs": 32 weights plus one f16 scale per block):

* Q4_0, split: ``nib`` uint8 ``[rows, k/2]`` (16 bytes per 32-weight block, in
  GGUF in-block order: byte j of a block holds element j in its low nibble and
  element j+16 in its high nibble) and ``scl`` uint16 ``[rows, k/32]`` (f16 bit
  patterns).
* Q8_0, split: ``qs`` int8 ``[rows, k]`` (GGUF order) and ``scl`` uint16
  ``[rows, k/32]``.
* GGUF interleaved blocks (the input of the load-time repack of
  "Architecture", section "Memory and caching"): per block the f16 scale ``d``
  (2 bytes, little endian) followed by the 16 (Q4_0) or 32 (Q8_0) quant bytes;
  blocks of a row are consecutive, rows are consecutive.

The oracle reads the split arrays. The library reads its own stored layout,
which the repack (the library's ``qrepack`` or the oracle's ``repack``) makes
from the GGUF blocks; this module never produces it.

Draw order inside one workload, from one ``numpy.random.Generator(PCG64(seed))``:
weights q, then scales, then X, then y0, then expert ids, then routing logits.
Nibbles uniform on 0..15 are drawn as uniform bytes (two independent uniform
nibbles per byte); Q8_0 quants are uniform on -127..127; scales are
f16(|N(0, 0.02)| / 8) for Q4_0 and f16(|N(0, 0.02)| / 127) for Q8_0; activations
are f16(N(0, 1)); residuals are f32(N(0, 1)); routing weights are a softmax of
eight f64 N(0, 1) logits per column, stored as f32.
"""
from __future__ import annotations

import numpy as np

Q4_0 = 2  # GGUF type id
Q8_0 = 8  # GGUF type id
QK = 32   # weights per block

BLOCK_QBYTES = {Q4_0: 16, Q8_0: 32}
SCALE_DIV = {Q4_0: 8.0, Q8_0: 127.0}


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def qbytes_per_row(qtype: int, k: int) -> int:
    return k // QK * BLOCK_QBYTES[qtype]


def weight_bytes(qtype: int, rows: int, k: int) -> int:
    """Bytes of one quantised matrix (quants + f16 scales)."""
    return rows * (qbytes_per_row(qtype, k) + (k // QK) * 2)


def draw_quants(g: np.random.Generator, qtype: int, rows: int, k: int) -> np.ndarray:
    if k % QK:
        raise ValueError("k must be a multiple of 32")
    if qtype == Q4_0:
        return g.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    if qtype == Q8_0:
        return g.integers(-127, 128, size=(rows, k), dtype=np.int8)
    raise ValueError(f"unknown quant type {qtype}")


def draw_scales(g: np.random.Generator, qtype: int, rows: int, k: int,
                sigma: float = 0.02) -> np.ndarray:
    d = np.abs(g.standard_normal((rows, k // QK))) * sigma / SCALE_DIV[qtype]
    return d.astype(np.float16).view(np.uint16)


def draw_matrix(g: np.random.Generator, qtype: int, rows: int, k: int):
    """(quants, scales) for one matrix, quants first (the fixed draw order)."""
    q = draw_quants(g, qtype, rows, k)
    s = draw_scales(g, qtype, rows, k)
    return q, s


def draw_x(g: np.random.Generator, ncols: int, k: int) -> np.ndarray:
    return g.standard_normal((ncols, k)).astype(np.float16).view(np.uint16)


def draw_y0(g: np.random.Generator, ncols: int, rows: int) -> np.ndarray:
    return g.standard_normal((ncols, rows)).astype(np.float32)


def draw_routing(g: np.random.Generator, ncols: int, n_expert: int, topk: int):
    """Expert ids drawn without replacement per column, then softmax weights."""
    ids = np.stack([g.choice(n_expert, size=topk, replace=False)
                    for _ in range(ncols)]).astype(np.int32)
    logits = g.standard_normal((ncols, topk))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    rw = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, rw


def to_gguf_blocks(qtype: int, q: np.ndarray, scl: np.ndarray) -> np.ndarray:
    """Interleave split arrays into GGUF blocks: per block d then the quants."""
    rows = q.shape[0]
    nb = scl.shape[1]
    qb = BLOCK_QBYTES[qtype]
    out = np.empty((rows, nb, 2 + qb), dtype=np.uint8)
    out[:, :, 0:2] = scl.astype("<u2").view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = q.view(np.uint8).reshape(rows, nb, qb)
    return out.reshape(rows, nb * (2 + qb))


# --------------------------------------------------------------------------
# Workloads shaped like the pages' models: 2,048- and 5,120-wide hidden
# states, a 17,408-wide FFN, a 248,320-row LM head, a 256-expert top-8 MoE.
# --------------------------------------------------------------------------

def gemv_case(qtype: int, rows: int, k: int, ncols: int, residual: bool,
              seed: int = 0) -> dict:
    g = rng(seed)
    q, s = draw_matrix(g, qtype, rows, k)
    x = draw_x(g, ncols, k)
    y0 = draw_y0(g, ncols, rows) if residual else None
    return dict(qtype=qtype, rows=rows, k=k, ncols=ncols, q=q, scl=s, x=x, y0=y0)


def ffn_case(qtype: int, ffn: int, hidden: int, ncols: int, seed: int = 0) -> dict:
    """Gate and up [ffn, hidden], down [hidden, ffn], X [ncols, hidden], y0."""
    g = rng(seed)
    qg, sg = draw_matrix(g, qtype, ffn, hidden)
    qu, su = draw_matrix(g, qtype, ffn, hidden)
    qd, sd = draw_matrix(g, qtype, hidden, ffn)
    x = draw_x(g, ncols, hidden)
    y0 = draw_y0(g, ncols, hidden)
    return dict(qtype=qtype, ffn=ffn, hidden=hidden, ncols=ncols,
                qg=qg, sg=sg, qu=qu, su=su, qd=qd, sd=sd, x=x, y0=y0)


def moe_case(qtype: int, n_expert: int, ffn: int, hidden: int, ncols: int,
             topk: int = 8, shared: bool = True, residual: bool = True,
             seed: int = 0) -> dict:
    """Stacked experts: gate/up [E, ffn, hidden], down [E, hidden, ffn]."""
    g = rng(seed)
    qg, sg = draw_matrix(g, qtype, n_expert * ffn, hidden)
    qu, su = draw_matrix(g, qtype, n_expert * ffn, hidden)
    qd, sd = draw_matrix(g, qtype, n_expert * hidden, ffn)
    sh = None
    if shared:
        sqg, ssg = draw_matrix(g, qtype, ffn, hidden)
        squ, ssu = draw_matrix(g, qtype, ffn, hidden)
        sqd, ssd = draw_matrix(g, qtype, hidden, ffn)
        sh = dict(qg=sqg, sg=ssg, qu=squ, su=ssu, qd=sqd, sd=ssd)
    x = draw_x(g, ncols, hidden)
    y0 = draw_y0(g, ncols, hidden) if residual else None
    ids, rw = draw_routing(g, ncols, n_expert, topk)
    return dict(qtype=qtype, n_expert=n_expert, ffn=ffn, hidden=hidden,
                ncols=ncols, topk=topk, qg=qg, sg=sg, qu=qu, su=su, qd=qd,
                sd=sd, shared=sh, x=x, y0=y0, ids=ids, rw=rw)


# The five workloads at full size.
def small_q8_gemv(seed: int = 0) -> dict:
    """Q8_0 GEMV, 1 column, W 2048x2048."""
    return gemv_case(Q8_0, 2048, 2048, 1, residual=False, seed=seed)


def q4_gemv_residual(seed: int = 0) -> dict:
    """Q4_0 GEMV with residual accumulate, 1 column, W 5120x5120."""
    return gemv_case(Q4_0, 5120, 5120, 1, residual=True, seed=seed)


def lm_head(seed: int = 0, rows: int = 248320) -> dict:
    """Q8_0 LM-head GEMV, 248,320 x 5,120, 1 column."""
    return gemv_case(Q8_0, rows, 5120, 1, residual=False, seed=seed)


def twins(rows: int, ncols: int, seed: int = 0) -> dict:
    """Q4_0 batched GEMV (verify twins), W rows x 5120, X [ncols, 5120]."""
    return gemv_case(Q4_0, rows, 5120, ncols, residual=False, seed=seed)


def prefill_ffn(seed: int = 0, ffn: int = 17408, hidden: int = 5120) -> dict:
    """Q4_0 16-column prefill FFN: gate/up 17408x5120, down 5120x17408."""
    return ffn_case(Q4_0, ffn, hidden, 16, seed=seed)


def moe_layer(ncols: int, seed: int = 0, n_expert: int = 256) -> dict:
    """Q8_0 stacked-expert MoE: 256 experts, ffn 512, hidden 2048, top-8 + shared."""
    return moe_case(Q8_0, n_expert, 512, 2048, ncols, topk=8, shared=True,
                    residual=False, seed=seed)
