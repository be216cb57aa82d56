// qg_moe.cu -- stacked-expert MoE layer.
//
// "Engine and kernels" (pooled.run), sections "What it runs" and "Kernel
// families": each FFN is 256 experts with 8 active per token plus a shared
// expert; router, top-k, expert gate/up and down and the weighted combine all
// stay on the GPU, so routing needs no readback. "A 235B model in a browser
// window", section "A mixture of experts is a different animal": the gate, up
// and down matrices of all experts are stacked by role, and the chosen experts
// run as one batched multiply over the stack.
//
// GB300 design: two kernels, both reading the device id list directly (no
// host round trip, no compaction pass of its own).
//   K1  gate/up : work items (routed pair, 2-row group). A pair is a valid
//                 (column, k) position of the id list, or a column of the
//                 shared expert. Pairs run in ascending expert id, so the
//                 columns that chose the same expert read its slice back to
//                 back (the second read hits L2). Each warp item is a 1-column
//                 dual GEMV of two rows over the whole hidden size:
//                 h[c][j] = f16(SiLU(G_e x_c) * (U_e x_c)).
//   K2  down+combine : CTA (column c, part); its warps own groups of output
//                 rows and sweep the column's routed experts (k order, the
//                 shared expert last): each lane accumulates
//                 rw[c][j] * d * dot(block) over its blocks and experts, a
//                 fixed butterfly sums the lanes of a row, and
//                 y = y0 + total is written once. The summation order depends
//                 only on the shape, so results are identical run to run.
//                 Two kernels compute it with the same arithmetic: for one or
//                 two columns a CTA owns 8 rows, and their slices of all its
//                 down matrices are staged in shared memory by bulk copies
//                 issued before the kernel waits on K1; otherwise the warps
//                 loop over row groups and each lane streams its blocks
//                 through registers.
// An id outside [0, E) contributes nothing and sets a bit in the caller's error
// word; no trap is raised and no CTA waits on another.
#include <cuda_runtime.h>

#include "qg_async.cuh"
#include "qg_cc_core.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int MOE_WARPS = 8;
constexpr int MOE_THREADS = MOE_WARPS * 32;
constexpr int MOE_RW1 = 2;                 // gate/up rows per warp item
constexpr int MOE_MAXN = 256;              // ncols * topk (16 columns x top-16)
constexpr int MOE_MAXC = 16;               // columns
constexpr int MOE_MAXJ = 17;               // topk + shared
constexpr int MOE_XSMEM_FLOATS = 32768;    // staged activations per CTA (128 KB)
static_assert(MOE_MAXN <= MOE_THREADS, "one id-list slot per thread");

__device__ int32_t g_moe_error = 0;  // QG_DEV_ERR_WAIT: a wait timed out

struct MoeDev {
  const uint8_t *qg, *qu, *qd;
  const uint16_t *sg, *su, *sd;
  int n_expert, ffn, hidden;
  const int32_t* ids;
  const float* rw;
  int topk, ncols;
  int has_shared;
  const uint8_t *sqg, *squ, *sqd;
  const uint16_t *ssg, *ssu, *ssd;
  const __half* x;
  const float* y0;
  float* y;
  __half* hws;   // [ncols][topk + 1][ffn]: h of position (c, j); j = topk is the shared expert
  int32_t* err_flag;
  int32_t* uniq_out;
};

// Stage the selected columns of x (column stride `colstride` halves, k wide)
// as f32 in the consumption order of qt, one 32-element block per thread.
// Two blocks per thread per pass, both loads issued before either is written.
__device__ __forceinline__ void stage_x_cols(int qt, float* xs, int xstride, const __half* x,
                                             size_t colstride, int ncols, int k) {
  const int nbk = k / QK;
  const int total = ncols * nbk;
  for (int it = threadIdx.x; it < total; it += 2 * blockDim.x) {
    const int it2 = it + blockDim.x;
    const int c = it / nbk, b = it % nbk;
    const XBlk a = load_xblk(x + (size_t)c * colstride + (size_t)b * QK);
    XBlk a2;
    const int c2 = it2 / nbk, b2 = it2 % nbk;
    if (it2 < total) a2 = load_xblk(x + (size_t)c2 * colstride + (size_t)b2 * QK);
    stage_xblk(qt, xs + c * xstride, xstride / QK, b, a);
    if (it2 < total) stage_xblk(qt, xs + c2 * xstride, xstride / QK, b2, a2);
  }
}

// ------------------------------------------------------------ K1: gate/up
// The MOE_RW1 rows of one work item: pair pp (expert slice or shared expert,
// column c, k slot j), rows r0 .. r0 + MOE_RW1 - 1 (clamped reads past ffn).
template <int QT>
struct MoeK1Rows {
  const uint8_t *qa, *qb;
  const uint16_t *sa, *sb;
  int c, j, r0;
  int row[MOE_RW1];
};

template <int QT>
__device__ __forceinline__ MoeK1Rows<QT> moe_k1_rows(const MoeDev& p, const int16_t* s_order,
                                                     const int* s_ids, const int8_t* s_pc,
                                                     const int8_t* s_pj, int n, int pp, int g,
                                                     size_t mat_q, size_t mat_s) {
  MoeK1Rows<QT> w;
  const int code = s_order[pp];
  w.c = s_pc[pp];
  w.j = s_pj[pp];
  if (code < n) {
    const size_t e = (size_t)s_ids[code];
    w.qa = p.qg + e * mat_q; w.sa = p.sg + e * mat_s;
    w.qb = p.qu + e * mat_q; w.sb = p.su + e * mat_s;
  } else {
    w.qa = p.sqg; w.sa = p.ssg; w.qb = p.squ; w.sb = p.ssu;
  }
  w.r0 = g * MOE_RW1;
#pragma unroll
  for (int r = 0; r < MOE_RW1; ++r) w.row[r] = min(w.r0 + r, p.ffn - 1);
  return w;
}

// The pair order of K1, shared by both gate/up kernels: every thread of the
// CTA calls this after the kernel's wait. x is staged (f32, consumption order
// of QT) into xs while the ids load; the valid (column, k) positions are
// ranked by (expert id, position) into s_order / s_pc / s_pj, followed by the
// shared expert's columns (codes n + c). CTA 0 also writes the distinct ids
// and the bad-id bit. Returns the number of pairs.
struct MoePairSmem {
  int ids[MOE_MAXN];
  __align__(16) int key[MOE_MAXN];     // id * MOE_MAXN + position, or INT_MAX
  int16_t order[MOE_MAXN + MOE_MAXC];  // routed pairs, then the shared expert's
  int8_t pc[MOE_MAXN + MOE_MAXC], pj[MOE_MAXN + MOE_MAXC];  // column, k slot
};

template <int QT>
__device__ __forceinline__ int moe_pair_order(const MoeDev& p, MoePairSmem& sm, float* xs) {
  const int n = p.ncols * p.topk;
  const int t = threadIdx.x;
  const int k = p.hidden;
  // The ids are loaded first; x is staged while they are in flight.
  int id = -1;
  if (t < n) id = p.ids[t];
  stage_x_cols(QT, xs, k, p.x, (size_t)k, p.ncols, k);
  bool valid = false;
  if (t < n) {
    valid = id >= 0 && id < p.n_expert;
    sm.ids[t] = valid ? id : -1;
  }
  if (t < MOE_MAXN) sm.key[t] = valid ? id * MOE_MAXN + t : 0x7fffffff;
  const int nvalid = __syncthreads_count(valid);  // also publishes the staged x
  if (valid) {
    // rank = number of keys below this one (keys are distinct)
    const int key = id * MOE_MAXN + t;
    const int4* k4 = reinterpret_cast<const int4*>(sm.key);
    int rank = 0;
#pragma unroll 4
    for (int s = 0; s < (n + 3) / 4; ++s) {
      const int4 o = k4[s];
      rank += (o.x < key) + (o.y < key) + (o.z < key) + (o.w < key);
    }
    sm.order[rank] = (int16_t)t;
    sm.pc[rank] = (int8_t)(t / p.topk);
    sm.pj[rank] = (int8_t)(t % p.topk);
  }
  if (p.has_shared && t < p.ncols) {
    sm.order[nvalid + t] = (int16_t)(n + t);
    sm.pc[nvalid + t] = (int8_t)t;
    sm.pj[nvalid + t] = (int8_t)p.topk;
  }
  __syncthreads();

  if (blockIdx.x == 0) {
    // distinct valid ids, ascending, padded with -1; error bit for bad ids
    bool start = false;
    int cur = -1;
    if (t < nvalid) {
      cur = sm.ids[sm.order[t]];
      start = t == 0 || sm.ids[sm.order[t - 1]] != cur;
    }
    const int U = __syncthreads_count(start);
    if (p.uniq_out) {
      if (start) {
        int u = 0;
        for (int r = 1; r <= t; ++r) u += sm.ids[sm.order[r]] != sm.ids[sm.order[r - 1]] ? 1 : 0;
        p.uniq_out[u] = cur;
      }
      if (t >= U && t < n) p.uniq_out[t] = -1;
    }
    if (t == 0 && nvalid < n && p.err_flag) atomicOr(p.err_flag, (int32_t)QG_MOE_BAD_ID);
  }
  return nvalid + (p.has_shared ? p.ncols : 0);
}

// WARPS: 8, or 16 when the staged x is too large for two CTAs per SM (one
// CTA of 16 warps then keeps as many rows in flight as two of 8).
template <int QT, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, WARPS == 8 ? 2 : 1) moe_gate_up_kernel(const MoeDev p) {
  __shared__ MoePairSmem sm;
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);
  constexpr int QB = QTraits<QT>::QB;
  const int n = p.ncols * p.topk;
  const int t = threadIdx.x;
  const int k = p.hidden;
  // Dependents may launch only once this kernel has passed its wait: the
  // staged down kernel reads ids and rw before its own wait, and by then the
  // kernel that wrote them has completed.
  pdl_wait();  // ids and x come from earlier kernels on the stream
  pdl_trigger();
  const int P = moe_pair_order<QT>(p, sm, xs);

  const int lane = t & 31, warp = t >> 5;
  const int nb = k / QK;
  const size_t rowbytes = (size_t)nb * QB;
  const size_t mat_q = (size_t)p.ffn * rowbytes;
  const size_t mat_s = (size_t)p.ffn * nb;
  const int ngroups = (p.ffn + MOE_RW1 - 1) / MOE_RW1;
  const int total = P * ngroups;
  const int stride = gridDim.x * WARPS;
  int item = blockIdx.x * WARPS + warp;

  for (; item < total; item += stride) {
    const MoeK1Rows<QT> cur = moe_k1_rows<QT>(p, sm.order, sm.ids, sm.pc, sm.pj, n,
                                              item / ngroups, item % ngroups, mat_q, mat_s);
    float ta[MOE_RW1], tb[MOE_RW1];
#pragma unroll
    for (int r = 0; r < MOE_RW1; ++r) { ta[r] = 0.f; tb[r] = 0.f; }
    cc_rowdot_1col<QT, MOE_RW1, true>(cur.qa, cur.sa, cur.qb, cur.sb, rowbytes, nb, cur.row,
                                      xs + cur.c * k, nb, 0, nb, lane, ta, tb);
    int idx, idx2;
    const float gs = warp_transpose_reduce<MOE_RW1>(ta, lane, idx);
    const float us = warp_transpose_reduce<MOE_RW1>(tb, lane, idx2);
    if ((lane & (32 / MOE_RW1 - 1)) == 0) {
      const int row = cur.r0 + idx;
      if (row < p.ffn)
        p.hws[((size_t)cur.c * (p.topk + 1) + cur.j) * p.ffn + row] =
            __float2half_rn(silu_f32(gs) * us);
    }
  }
}

// ------------------------------------------------------ K2: down + combine
// RW2 rows per lane per item; JB experts' blocks are loaded before any is used.
template <int QT, int RW2, int JB>
__global__ void __launch_bounds__(MOE_THREADS, 2) moe_down_kernel(const MoeDev p) {
  __shared__ int s_e[MOE_MAXJ];     // expert of each live entry (n_expert = shared)
  __shared__ int s_j[MOE_MAXJ];     // its position j (h index)
  __shared__ float s_w[MOE_MAXJ];   // its routing weight
  __shared__ int s_nj;
  extern __shared__ float4 smem_f4[];
  float* hs = reinterpret_cast<float*>(smem_f4);
  constexpr int QB = QTraits<QT>::QB;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  pdl_trigger();
  pdl_wait();  // ids, rw, y0 and the gate/up results come from earlier kernels
  const int nparts = gridDim.x / p.ncols;
  const int c = blockIdx.x % p.ncols, part = blockIdx.x / p.ncols;
  if (part >= nparts) return;  // uniform over the CTA
  if (warp == 0) {
    // live entries of column c in k order (one load per lane, then a ballot)
    int id = -1;
    float w = 0.f;
    if (lane < p.topk) {
      id = p.ids[c * p.topk + lane];
      w = p.rw[c * p.topk + lane];
    }
    const bool live = lane < p.topk && id >= 0 && id < p.n_expert;
    const unsigned m = __ballot_sync(0xffffffffu, live);
    if (live) {
      const int at = __popc(m & ((1u << lane) - 1u));
      s_e[at] = id; s_j[at] = lane; s_w[at] = w;
    }
    const int nl = __popc(m);
    if (lane == 0) {
      if (p.has_shared) { s_e[nl] = p.n_expert; s_j[nl] = p.topk; s_w[nl] = 1.f; }
      s_nj = nl + (p.has_shared ? 1 : 0);
    }
  }
  __syncthreads();
  const int nj = s_nj;
  const int k = p.ffn, nb = k / QK;
  // h of the live entries, staged as f32 planes (entry m at hs + m * k)
  for (int it = t; it < nj * nb; it += blockDim.x) {
    const int m = it / nb, b = it % nb;
    stage_block(QT, hs + m * k, nb, b,
                p.hws + ((size_t)c * (p.topk + 1) + s_j[m]) * k + (size_t)b * QK);
  }
  __syncthreads();

  const size_t rowbytes = (size_t)nb * QB;
  const size_t mat_q = (size_t)p.hidden * rowbytes;
  const size_t mat_s = (size_t)p.hidden * nb;
  int lpr = 32;  // lanes per row: a power of two, at most the blocks of a row
  while (lpr > nb) lpr >>= 1;
  const int rpw = 32 / lpr;
  const int rs = lane / lpr, bl = lane % lpr;
  const int rows_item = rpw * RW2;
  const int nitems = (p.hidden + rows_item - 1) / rows_item;
  for (int item = part * MOE_WARPS + warp; item < nitems; item += nparts * MOE_WARPS) {
    int rowidx[RW2];
#pragma unroll
    for (int r = 0; r < RW2; ++r) rowidx[r] = min(item * rows_item + r * rpw + rs, p.hidden - 1);
    float acc[RW2];
#pragma unroll
    for (int r = 0; r < RW2; ++r) acc[r] = 0.f;
    for (int b = bl; b < nb; b += lpr) {
      for (int m0 = 0; m0 < nj; m0 += JB) {
        Blk<QT> q[JB][RW2];
        uint16_t sc[JB][RW2];
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          if (m0 + jj < nj) {
            const int e = s_e[m0 + jj];
            const uint8_t* qe = e == p.n_expert ? p.sqd : p.qd + (size_t)e * mat_q;
            const uint16_t* se = e == p.n_expert ? p.ssd : p.sd + (size_t)e * mat_s;
#pragma unroll
            for (int r = 0; r < RW2; ++r) {
              q[jj][r].load(qe + (size_t)rowidx[r] * rowbytes + (size_t)b * QB);
              sc[jj][r] = ld_u16(se + (size_t)rowidx[r] * nb + b);
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          if (m0 + jj < nj) {
            float2 xr[16];
            load_x16(hs + (m0 + jj) * k, nb, b, xr);
            const float w = s_w[m0 + jj];
#pragma unroll
            for (int r = 0; r < RW2; ++r) acc[r] = fmaf(w * h2f(sc[jj][r]), blk_dot(q[jj][r], xr), acc[r]);
          }
        }
      }
    }
    // sum the lanes of each row (fixed butterfly within the lpr-lane group)
#pragma unroll
    for (int r = 0; r < RW2; ++r)
      for (int off = lpr >> 1; off >= 1; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    if (bl == 0) {
#pragma unroll
      for (int r = 0; r < RW2; ++r) {
        const int row = item * rows_item + r * rpw + rs;
        if (row < p.hidden) {
          const size_t o = (size_t)c * p.hidden + row;
          p.y[o] = (p.y0 ? p.y0[o] : 0.f) + acc[r];
        }
      }
    }
  }
}

// ------------------------------------------- K2s: down + combine, staged
// The arithmetic of moe_down_kernel (each lane sums its blocks in ascending
// order, within a block the live experts in k order, then the same fixed
// butterfly per row), so the two kernels give bit-identical outputs. A CTA owns
// one column and R consecutive output rows; one thread brings the R-row slices
// of all the column's down matrices into shared memory with bulk copies issued
// before the kernel waits on its predecessor, so the down weights stream while
// the gate/up kernel finishes. Reading ids and rw before that wait is safe:
// the gate/up kernel lets its dependents launch only after its own wait, by
// which time the kernel that wrote them has completed.
//
// Dynamic shared memory: h of the live entries as f32 planes [nj][ffn], then
// per entry its R rows of quants [R][ffn/32 * QB] and of scales
// [R][ffn/32] (padded to 16 bytes).
template <int QT>
__global__ void __launch_bounds__(MOE_THREADS, 2) moe_down_staged_kernel(const MoeDev p, int R) {
  __shared__ int s_e[MOE_MAXJ];     // expert of each live entry (n_expert = shared)
  __shared__ int s_j[MOE_MAXJ];     // its position j (h index)
  __shared__ float s_w[MOE_MAXJ];   // its routing weight
  __shared__ int s_nj;
  __shared__ __align__(8) uint64_t s_bar;
  extern __shared__ float4 smem_f4[];
  constexpr int QB = QTraits<QT>::QB;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int k = p.ffn, nb = k / QK;
  const int njmax = p.topk + (p.has_shared ? 1 : 0);
  const uint32_t rowbytes = (uint32_t)nb * QB;
  const uint32_t sstride = (uint32_t)((R * nb * 2 + 15) & ~15);
  float* hs = reinterpret_cast<float*>(smem_f4);
  uint8_t* wq = reinterpret_cast<uint8_t*>(hs + (size_t)njmax * k);
  uint8_t* wsc = wq + (size_t)njmax * R * rowbytes;
  pdl_trigger();
  const int c = blockIdx.x % p.ncols, part = blockIdx.x / p.ncols;
  const int r0 = part * R;
  const int nrows = min(R, p.hidden - r0);  // a multiple of 8 (hidden % 32 == 0, R % 8 == 0)
  if (warp == 0) {
    // live entries of column c in k order (one load per lane, then a ballot)
    int id = -1;
    float w = 0.f;
    if (lane < p.topk) {
      id = p.ids[c * p.topk + lane];
      w = p.rw[c * p.topk + lane];
    }
    const bool live = lane < p.topk && id >= 0 && id < p.n_expert;
    const unsigned m = __ballot_sync(0xffffffffu, live);
    if (live) {
      const int at = __popc(m & ((1u << lane) - 1u));
      s_e[at] = id; s_j[at] = lane; s_w[at] = w;
    }
    const int nl = __popc(m);
    if (lane == 0) {
      if (p.has_shared) { s_e[nl] = p.n_expert; s_j[nl] = p.topk; s_w[nl] = 1.f; }
      s_nj = nl + (p.has_shared ? 1 : 0);
      mbar_init(&s_bar, 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  __syncthreads();
  const int nj = s_nj;
  const uint32_t bar = smem_u32(&s_bar);
  if (warp == 0) {
    // lane m issues the two copies of live entry m (one instruction stream per
    // copy pair instead of one thread issuing them all)
    const size_t mat_q = (size_t)p.hidden * rowbytes;
    const size_t mat_s = (size_t)p.hidden * nb;
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)nj * (uint32_t)nrows * (rowbytes + 2u * nb));
    __syncwarp();
    if (lane < nj) {
      const int m = lane;
      const int e = s_e[m];
      const uint8_t* qe = e == p.n_expert ? p.sqd : p.qd + (size_t)e * mat_q;
      const uint16_t* se = e == p.n_expert ? p.ssd : p.sd + (size_t)e * mat_s;
      bulk_g2s(smem_u32(wq + (size_t)m * R * rowbytes), qe + (size_t)r0 * rowbytes,
               (uint32_t)nrows * rowbytes, bar);
      bulk_g2s(smem_u32(wsc + (size_t)m * sstride), se + (size_t)r0 * nb,
               (uint32_t)nrows * nb * 2u, bar);
    }
  }
  pdl_wait();  // the gate/up results, and y0, come from earlier kernels
  for (int it = t; it < nj * nb; it += blockDim.x) {
    const int m = it / nb, b = it % nb;
    stage_block(QT, hs + m * k, nb, b,
                p.hws + ((size_t)c * (p.topk + 1) + s_j[m]) * k + (size_t)b * QK);
  }
  __syncthreads();
  mbar_wait(bar, 0, &g_moe_error);

  int lpr = 32;  // lanes per row: a power of two, at most the blocks of a row
  while (lpr > nb) lpr >>= 1;
  const int rpw = 32 / lpr;
  const int rs = lane / lpr, bl = lane % lpr;
  const int nitems = (R + rpw - 1) / rpw;
  for (int item = warp; item < nitems; item += MOE_WARPS) {
    // rows past the CTA's slice (when R is not a multiple of rpw) are computed
    // on its last row and not stored
    const int row = r0 + item * rpw + rs;
    const int lr = min(row - r0, nrows - 1);
    float acc = 0.f;
    for (int b = bl; b < nb; b += lpr) {
      // three experts' blocks are read before any is used; the sum still
      // takes the experts one at a time, in k order
      for (int m0 = 0; m0 < nj; m0 += 3) {
        Blk<QT> q[3];
        uint16_t sc[3];
#pragma unroll
        for (int jj = 0; jj < 3; ++jj) {
          const int m = min(m0 + jj, nj - 1);
          q[jj].load_shared(wq + ((size_t)m * R + lr) * rowbytes + (size_t)b * QB);
          sc[jj] = *reinterpret_cast<const uint16_t*>(wsc + (size_t)m * sstride +
                                                      ((size_t)lr * nb + b) * 2);
        }
#pragma unroll
        for (int jj = 0; jj < 3; ++jj) {
          if (m0 + jj < nj) {
            float2 xr[16];
            load_x16(hs + (m0 + jj) * k, nb, b, xr);
            acc = fmaf(s_w[m0 + jj] * h2f(sc[jj]), blk_dot(q[jj], xr), acc);
          }
        }
      }
    }
    for (int off = lpr >> 1; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (bl == 0 && row < r0 + nrows) {
      const size_t o = (size_t)c * p.hidden + row;
      p.y[o] = (p.y0 ? p.y0[o] : 0.f) + acc;
    }
  }
}

// Rows per CTA of the staged down kernel for this call, or 0 when the register
// kernel runs instead: for more than two columns (measured at 256 experts,
// ffn 512, hidden 2048, top-8 + shared: 1 column 14.3 -> 12.1 us per layer
// call with the staged kernel, but 8 columns 47.8 -> 56.6 and 16 columns
// 85.1 -> 103.0: its 1,024-2,048 short CTAs each stage h and wait out one
// copy latency), or when its shared memory does not fit two CTAs per SM.
static int moe_staged_rows(int qt, int ffn, int hidden, int ncols, int topk, int has_shared,
                           size_t* smem) {
  constexpr int R = 8;  // rows per CTA: 256 CTAs per column at hidden 2048
  if (ncols > 2 || hidden < R) return 0;
  const int nb = ffn / QK;
  const size_t rowbytes = (size_t)nb * (qt == T_Q4_0 ? 16 : 32);
  const int njmax = topk + (has_shared ? 1 : 0);
  const size_t sstride = ((size_t)R * nb * 2 + 15) & ~(size_t)15;
  const size_t need = (size_t)njmax * ((size_t)ffn * 4 + R * rowbytes + sstride);
  if (need > 100 * 1024) return 0;
  *smem = need;
  return R;
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

size_t moe_ws_bytes(int n_expert, int ffn, int hidden, int ncols, int topk) {
  (void)n_expert;
  (void)hidden;
  return align256((size_t)ncols * (topk + 1) * ffn * sizeof(__half));
}

bool moe_shape_supported(int ffn, int hidden, int ncols, int topk) {
  return ncols >= 1 && ncols <= MOE_MAXC && ncols * topk <= MOE_MAXN &&
         (size_t)ncols * hidden <= MOE_XSMEM_FLOATS &&
         (size_t)(topk + 1) * ffn <= MOE_XSMEM_FLOATS;
}

template <class K>
static cudaError_t launch_moe(K kern, int threads, long grid_max_units, int multiple, size_t smem,
                              const MoeDev& d, cudaStream_t s, LaunchClass cls) {
  int occ = 1;
  cudaError_t e = kernel_occupancy(reinterpret_cast<const void*>(kern), threads, smem, &occ);
  if (e != cudaSuccess) return e;
  long grid = (long)device_sm_count() * occ;
  if (grid > grid_max_units) grid = grid_max_units;
  grid = grid / multiple * multiple;
  if (grid < multiple) grid = multiple;
  return launch_pdl(kern, dim3((unsigned)grid), dim3((unsigned)threads), smem, s, 0, cls, d);
}

template <int QT>
static cudaError_t moe_launch_t(const MoeDev& d, cudaStream_t s) {
  const int ngroups = (d.ffn + MOE_RW1 - 1) / MOE_RW1;
  const long pairs_max = (long)d.ncols * d.topk + (d.has_shared ? d.ncols : 0);
  const size_t smem_gu = (size_t)d.ncols * d.hidden * sizeof(float);
  cudaError_t e;
  if (smem_gu <= 100 * 1024) {
    e = launch_moe(moe_gate_up_kernel<QT, 8>, 256, (pairs_max * ngroups + 7) / 8, 1, smem_gu, d, s,
                   LC_L1);
  } else {
    // One CTA per SM holding more than 100 KB of shared memory: launched as
    // LC_SMEM, so the register down kernel does not start on its SMs (16
    // columns, 256 experts, ffn 512, hidden 2048: 84.9 -> 82.4 us per layer
    // call; as LC_SMEM the 8-warp variant measured slower, 47.8 -> 48.7 us at
    // 8 columns).
    e = launch_moe(moe_gate_up_kernel<QT, 16>, 512, (pairs_max * ngroups + 15) / 16, 1, smem_gu, d, s,
                   LC_SMEM);
  }
  if (e != cudaSuccess) return e;
  size_t smem_ds = 0;
  const int R = moe_staged_rows(QT, d.ffn, d.hidden, d.ncols, d.topk, d.has_shared, &smem_ds);
  if (R > 0) {
    auto kern = moe_down_staged_kernel<QT>;
    if ((e = prepare_kernel(reinterpret_cast<const void*>(kern), smem_ds, false)) != cudaSuccess)
      return e;
    const int parts = (d.hidden + R - 1) / R;
    // Launched as LC_L1, so the next kernel on the stream may still overlap its
    // tail (measured 12.1 us per layer call at 1 column, 12.7 as LC_SMEM).
    return launch_pdl(kern, dim3((unsigned)(parts * d.ncols)), dim3(MOE_THREADS), smem_ds, s, 0,
                      LC_L1, d, R);
  }
  const size_t smem_dn = (size_t)(d.topk + 1) * d.ffn * sizeof(float);
  const long big = 1L << 30;
  // one row per lane per item when few columns share the grid (more items,
  // all of a lane's experts in flight at once); two rows otherwise
  if (d.ncols <= 2)
    return launch_moe(moe_down_kernel<QT, 1, 9>, MOE_THREADS, big, d.ncols, smem_dn, d, s, LC_L1);
  return launch_moe(moe_down_kernel<QT, 2, 3>, MOE_THREADS, big, d.ncols, smem_dn, d, s, LC_L1);
}

cudaError_t moe_device_error(int32_t* bits) {
  const int32_t zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_moe_error, sizeof(*bits));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_moe_error, &zero, sizeof(zero));
  return e;
}

cudaError_t moe_forward(const MoeArgs& a, cudaStream_t s) {
  MoeDev d{};
  d.qg = (const uint8_t*)a.qg; d.qu = (const uint8_t*)a.qu; d.qd = (const uint8_t*)a.qd;
  d.sg = a.sg; d.su = a.su; d.sd = a.sd;
  d.n_expert = a.n_expert; d.ffn = a.ffn; d.hidden = a.hidden;
  d.ids = a.ids; d.rw = a.rw; d.topk = a.topk; d.ncols = a.ncols;
  d.has_shared = a.has_shared ? 1 : 0;
  d.sqg = (const uint8_t*)a.sqg; d.squ = (const uint8_t*)a.squ; d.sqd = (const uint8_t*)a.sqd;
  d.ssg = a.ssg; d.ssu = a.ssu; d.ssd = a.ssd;
  d.x = reinterpret_cast<const __half*>(a.x);
  d.y0 = a.y0; d.y = a.y;
  d.hws = reinterpret_cast<__half*>(a.ws);
  d.err_flag = a.err_flag;
  d.uniq_out = a.uniq_out;
  return a.qt == T_Q4_0 ? moe_launch_t<T_Q4_0>(d, s) : moe_launch_t<T_Q8_0>(d, s);
}

}  // namespace qg
