// qg_cc.cu -- CUDA-core streamed GEMV kernels (the 1-column decode path and the
// CUDA-core twins).
//
// Decode GEMV: "Engine and kernels" (pooled.run), section "Kernel families",
// cooperative GEMV, and section "Reading weights": a row is swept by the lanes
// of a warp with interleaved 32-weight blocks so every read is one contiguous
// stripe, dequantised in registers, with named (never indexed) accumulators.
//
// GB300 layout of the work: a warp owns RW consecutive rows; lane l takes blocks
// l, l+32, ... of those rows, so one warp-wide 16-byte load covers 512
// contiguous bytes of a row. x is staged once per CTA in shared memory as f32,
// pre-scaled to match the exact exponent-OR dequantisation, and reused across
// the RW rows. Each lane folds its blocks into per-row totals (block scale
// applied per block in f32), and a fixed butterfly reduces them across the
// warp. The grid is persistent (a multiple of the SM count); the reduction
// order does not depend on the grid, so results are identical on any device.
#include <cuda_runtime.h>

#include "qg_cc_core.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int CC_WARPS = 8;
constexpr int CC_THREADS = CC_WARPS * 32;
constexpr int CC_XSMEM_FLOATS = 24576;  // 96 KB of staged x per CTA

// Rows per warp: 8 for one column (x reused across 8 rows), fewer for more
// columns (at most 16 accumulators per thread), and fewer again when a matrix
// is too small to give every SM work. The row count never changes a result:
// each row is summed by one warp, blocks in order per lane, then the same
// lane butterfly.
template <int NC, int RW_> struct CCShape {
  static constexpr int RW = RW_;
  static constexpr int V = RW * NC <= 1 ? 1 : (RW * NC <= 2 ? 2 : (RW * NC <= 4 ? 4 : (RW * NC <= 8 ? 8 : (RW * NC <= 16 ? 16 : 32))));
};
template <int NC> struct CCDefaultRW {
  static constexpr int RW = NC >= 8 ? 1 : (NC >= 4 ? 2 : (NC >= 2 ? 4 : 8));
};

struct CCParams {
  const uint8_t* qa;
  const uint16_t* sa;
  const uint8_t* qb;  // second matrix (DUAL) or null
  const uint16_t* sb;
  int rows, k;
  const __half* x;
  int ncols_total;     // columns present in x (for the column map)
  const float* y0;
  float* y;            // EPI_F32 output [ncols][rows]
  __half* h;           // EPI_SILU output [ncols][rows]
  int cb;              // blocks of x staged per chunk
};

enum { EPI_F32 = 0, EPI_SILU = 1 };

template <int QT, int NC, int RW_, bool DUAL, int EPI>
__global__ void __launch_bounds__(CC_THREADS, NC == 1 ? 2 : 1)
qmv_cc_kernel(const CCParams p) {
  using S = CCShape<NC, RW_>;
  constexpr int RW = S::RW;
  constexpr int V = S::V;
  constexpr int QB = QTraits<QT>::QB;
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int k = p.k;
  const int nb = k / QK;
  const size_t rowbytes = (size_t)nb * QB;
  const int cb = p.cb;
  const int nchunk = (nb + cb - 1) / cb;
  const int xstride = cb * QK;
  int cols[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) cols[c] = c;

  const int ngroups = (p.rows + RW - 1) / RW;
  const int gstride = gridDim.x * CC_WARPS;
  const int gfirst = blockIdx.x * CC_WARPS;
  const int iters = gfirst < ngroups ? (ngroups - gfirst + gstride - 1) / gstride : 0;

  pdl_trigger();

  // One block b of the warp's rows, quants and scales already in registers:
  // per row and column, scale * (block dot) into the row's total, in the same
  // order for any column count.
  float ta[RW][NC], tb[RW][NC];
  auto accumulate = [&](const Blk<QT> (&qa)[RW], const uint16_t (&sa)[RW], const Blk<QT> (&qb)[RW],
                        const uint16_t (&sb)[RW], int bx) {
    if (NC == 1) {
      float2 xr[16];
      load_x16(xs, cb, bx, xr);
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        ta[r][0] = fmaf(h2f(sa[r]), blk_dot(qa[r], xr), ta[r][0]);
        if (DUAL) tb[r][0] = fmaf(h2f(sb[r]), blk_dot(qb[r], xr), tb[r][0]);
      }
    } else {
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        float2 wa[16], wb[16];
        blk_dequant(qa[r], wa);
        if (DUAL) blk_dequant(qb[r], wb);
        const float da = h2f(sa[r]);
        const float db = DUAL ? h2f(sb[r]) : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float2 xr[16];
          load_x16(xs + c * xstride, cb, bx, xr);
          ta[r][c] = fmaf(da, wv_dot(wa, xr), ta[r][c]);
          if (DUAL) tb[r][c] = fmaf(db, wv_dot(wb, xr), tb[r][c]);
        }
      }
    }
  };
  // Reduce the row totals across the lanes (fixed butterfly) and write them.
  auto finish = [&](int g) {
    float va[V], vb[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      va[i] = i < RW * NC ? ta[i / NC][i % NC] : 0.f;
      vb[i] = i < RW * NC ? tb[i / NC][i % NC] : 0.f;
    }
    int idx;
    const float sa_tot = warp_transpose_reduce<V>(va, lane, idx);
    float sb_tot = 0.f;
    if (DUAL) {
      int idx2;
      sb_tot = warp_transpose_reduce<V>(vb, lane, idx2);
    }
    // lanes sharing an index hold the same total; the lowest one writes
    const int span = 32 / V;
    if ((lane % span) == 0 && idx < RW * NC) {
      const int r = idx / NC, c = idx % NC;
      const int row = g * RW + r;
      if (row < p.rows) {
        const size_t o = (size_t)c * p.rows + row;
        if (EPI == EPI_F32) {
          float v = sa_tot;
          if (p.y0) v += p.y0[o];
          p.y[o] = v;
        } else {
          p.h[o] = __float2half_rn(silu_f32(sa_tot) * sb_tot);
        }
      }
    }
  };
  auto zero = [&]() {
#pragma unroll
    for (int r = 0; r < RW; ++r)
#pragma unroll
      for (int c = 0; c < NC; ++c) { ta[r][c] = 0.f; tb[r][c] = 0.f; }
  };

  // Rows of at most 64 blocks, one row group per warp (small matrices): the
  // warp's blocks (at most two per lane and row) are loaded into registers
  // before waiting for the previous kernel, which never writes weights, so
  // after the wait only x is fetched. Same blocks, same order as the loop.
  constexpr bool kPreload = !DUAL && RW * (QB / 4) * 2 <= 40;  // registers held across the wait
  if (kPreload && nchunk == 1 && nb <= 64 && iters == 1) {
    const int g = gfirst + warp;
    const bool active = g < ngroups;
    int rowidx[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) rowidx[r] = min(g * RW + r, p.rows - 1);
    Blk<QT> q0[RW], q1[RW];
    uint16_t s0[RW], s1[RW];
    const int b0 = lane, b1 = lane + 32;
    if (active) {
#pragma unroll
      for (int r = 0; r < RW; ++r) {
        if (b0 < nb) {
          q0[r].load(p.qa + (size_t)rowidx[r] * rowbytes + (size_t)b0 * QB);
          s0[r] = ld_u16(p.sa + (size_t)rowidx[r] * nb + b0);
        }
        if (b1 < nb) {
          q1[r].load(p.qa + (size_t)rowidx[r] * rowbytes + (size_t)b1 * QB);
          s1[r] = ld_u16(p.sa + (size_t)rowidx[r] * nb + b1);
        }
      }
    }
    pdl_wait();
    stage_x<QT, NC>(xs, xstride, p.x, k, cols, 0, nb);
    __syncthreads();
    if (!active) return;
    zero();
    if (b0 < nb) accumulate(q0, s0, q0, s0, b0);
    if (b1 < nb) accumulate(q1, s1, q1, s1, b1);
    finish(g);
    return;
  }

  // The first 32 blocks of every row of this CTA's first row groups are pulled
  // into L2 before waiting for the previous kernel (weights are never written
  // by it), so the stream starts while that kernel drains and x is staged.
  if (nchunk == 1 && iters > 0 && threadIdx.x < CC_WARPS * RW) {
    const int row = gfirst * RW + (int)threadIdx.x;
    if (row < p.rows) {
      const int pb = (nb < 32 ? nb : 32) * QB;
      l2_prefetch_bulk(p.qa + (size_t)row * rowbytes, (uint32_t)pb);
      l2_prefetch_line(p.sa + (size_t)row * nb);
      if (DUAL) {
        l2_prefetch_bulk(p.qb + (size_t)row * rowbytes, (uint32_t)pb);
        l2_prefetch_line(p.sb + (size_t)row * nb);
      }
    }
  }
  pdl_wait();

  if (nchunk == 1) {
    stage_x<QT, NC>(xs, xstride, p.x, k, cols, 0, nb);
    __syncthreads();
  }

  for (int it = 0; it < iters; ++it) {
    const int g = gfirst + warp + it * gstride;
    const bool active = g < ngroups;
    int rowidx[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) rowidx[r] = min(g * RW + r, p.rows - 1);
    zero();
    for (int ch = 0; ch < nchunk; ++ch) {
      const int kb0 = ch * cb;
      const int kb1 = min(nb, kb0 + cb);
      if (nchunk > 1) {
        __syncthreads();
        stage_x<QT, NC>(xs, xstride, p.x, k, cols, kb0, kb1);
        __syncthreads();
      }
      if (!active) continue;
      for (int b = kb0 + lane; b < kb1; b += 32) {
        Blk<QT> qa[RW], qb[RW];
        uint16_t sa[RW], sb[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
          qa[r].load(p.qa + (size_t)rowidx[r] * rowbytes + (size_t)b * QB);
          sa[r] = ld_u16(p.sa + (size_t)rowidx[r] * nb + b);
          if (DUAL) {
            qb[r].load(p.qb + (size_t)rowidx[r] * rowbytes + (size_t)b * QB);
            sb[r] = ld_u16(p.sb + (size_t)rowidx[r] * nb + b);
          }
        }
        accumulate(qa, sa, qb, sb, b - kb0);
      }
    }
    if (!active) continue;
    finish(g);
  }
}

// ------------------------------------------------------------- launchers
template <int QT, int NC, int RW, bool DUAL, int EPI>
static cudaError_t launch_cc_t(const CCParams& p0, cudaStream_t s, int* nlaunch) {
  CCParams p = p0;
  const int nb = p.k / QK;
  // x chunks of a multiple of 32 blocks keep lane l on blocks l, l+32, ... in
  // every chunk, as in the 1-column kernel (bit-identical columns)
  int cb = CC_XSMEM_FLOATS / (NC * QK);
  if (cb >= nb) cb = nb;
  else cb &= ~31;
  p.cb = cb;
  const size_t smem = (size_t)NC * cb * QK * sizeof(float);
  auto kern = qmv_cc_kernel<QT, NC, RW, DUAL, EPI>;
  int occ = 1;
  cudaError_t e = kernel_occupancy(reinterpret_cast<const void*>(kern), CC_THREADS, smem, &occ);
  if (e != cudaSuccess) return e;
  const long ngroups = (p.rows + RW - 1) / RW;
  long grid = (ngroups + CC_WARPS - 1) / CC_WARPS;
  const long maxgrid = (long)device_sm_count() * occ;
  if (grid > maxgrid) grid = maxgrid;
  if (grid < 1) grid = 1;
  if (nlaunch) ++*nlaunch;
  return launch_pdl(kern, dim3((unsigned)grid), dim3(CC_THREADS), smem, s, 0, LC_L1, p);
}

template <int QT, bool DUAL, int EPI>
static cudaError_t dispatch_nc(int nc, const CCParams& p, cudaStream_t s, int* nl) {
  switch (nc) {
    case 1: {
      // 8 rows per warp unless that leaves SMs idle (fewer than 2 CTAs per SM)
      const long ctas8 = ((long)p.rows + 8 * CC_WARPS - 1) / (8 * CC_WARPS);
      if (ctas8 >= 2L * device_sm_count()) return launch_cc_t<QT, 1, 8, DUAL, EPI>(p, s, nl);
      return launch_cc_t<QT, 1, 2, DUAL, EPI>(p, s, nl);
    }
    case 2: return launch_cc_t<QT, 2, CCDefaultRW<2>::RW, DUAL, EPI>(p, s, nl);
    case 3: return launch_cc_t<QT, 3, CCDefaultRW<3>::RW, DUAL, EPI>(p, s, nl);
    case 4: return launch_cc_t<QT, 4, CCDefaultRW<4>::RW, DUAL, EPI>(p, s, nl);
    case 5: return launch_cc_t<QT, 5, CCDefaultRW<5>::RW, DUAL, EPI>(p, s, nl);
    case 6: return launch_cc_t<QT, 6, CCDefaultRW<6>::RW, DUAL, EPI>(p, s, nl);
    case 7: return launch_cc_t<QT, 7, CCDefaultRW<7>::RW, DUAL, EPI>(p, s, nl);
    case 8: return launch_cc_t<QT, 8, CCDefaultRW<8>::RW, DUAL, EPI>(p, s, nl);
  }
  return cudaErrorInvalidValue;
}

// Public-to-the-library launchers (column counts 1..8 per launch; larger counts
// are split by the caller into groups of at most 8 columns).
cudaError_t cc_gemv(int qt, const void* q, const uint16_t* scl, int rows, int k,
                    const uint16_t* x, int ncols, const float* y0, float* y, cudaStream_t s) {
  CCParams p{};
  p.qa = static_cast<const uint8_t*>(q);
  p.sa = scl;
  p.rows = rows;
  p.k = k;
  p.x = reinterpret_cast<const __half*>(x);
  p.ncols_total = ncols;
  p.y0 = y0;
  p.y = y;
  if (qt == T_Q4_0) return dispatch_nc<T_Q4_0, false, EPI_F32>(ncols, p, s, nullptr);
  return dispatch_nc<T_Q8_0, false, EPI_F32>(ncols, p, s, nullptr);
}

cudaError_t cc_gate_up_silu(int qt, const void* qg, const uint16_t* sg, const void* qu,
                            const uint16_t* su, int rows, int k, const uint16_t* x,
                            int ncols, uint16_t* h, cudaStream_t s) {
  CCParams p{};
  p.qa = static_cast<const uint8_t*>(qg);
  p.sa = sg;
  p.qb = static_cast<const uint8_t*>(qu);
  p.sb = su;
  p.rows = rows;
  p.k = k;
  p.x = reinterpret_cast<const __half*>(x);
  p.ncols_total = ncols;
  p.h = reinterpret_cast<__half*>(h);
  if (qt == T_Q4_0) return dispatch_nc<T_Q4_0, true, EPI_SILU>(ncols, p, s, nullptr);
  return dispatch_nc<T_Q8_0, true, EPI_SILU>(ncols, p, s, nullptr);
}

}  // namespace qg
