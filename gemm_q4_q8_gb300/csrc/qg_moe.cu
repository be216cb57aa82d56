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
// GB300 design: the device-side id list is compacted inside every CTA into the
// ascending list of distinct valid experts (each routed slice is then read from
// HBM once, for all columns that chose it) plus a per-expert column mask.
//   K1  gate/up : units (expert slot, 64-row tile); h = f16(SiLU(G x) * (U x))
//                 into the workspace, for the columns that route to the expert.
//   K2  down    : units (expert slot, 64-row tile of the hidden size);
//                 o = D h, f32, into the workspace.
//   K3  combine : y = y0 + sum_j rw[c][j] o[slot(c,j)] + o[shared], summed in
//                 slot order j, so the result does not depend on scheduling.
// An id outside [0, E) contributes nothing and sets a bit in the caller's error
// word; no trap is raised and no CTA waits on another.
#include <cuda_runtime.h>

#include "qg_cc_core.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int MOE_WARPS = 8;
constexpr int MOE_THREADS = MOE_WARPS * 32;
constexpr int MOE_RW = 4;                          // rows per warp
constexpr int MOE_TILE = MOE_WARPS * MOE_RW;       // rows per unit
constexpr int MOE_MAXN = 128;                      // ncols * topk
constexpr int MOE_XSMEM_FLOATS = 24576;            // staged activations per CTA

struct MoeRoute {
  int ids[MOE_MAXN];
  int first[MOE_MAXN];
  int slot[MOE_MAXN];      // slot of (c, j), -1 when the id is invalid
  int uniq[MOE_MAXN];
  uint32_t mask[MOE_MAXN + 1];
  int U;
  int bad;
};

struct MoeDev {
  int qt;
  const uint8_t *qg, *qu, *qd;
  const uint16_t *sg, *su, *sd;
  int n_expert, ffn, hidden;
  const int32_t* ids;
  const float* rw;
  int topk, ncols, umax;  // umax = slot index of the shared expert
  int has_shared;
  const uint8_t *sqg, *squ, *sqd;
  const uint16_t *ssg, *ssu, *ssd;
  const __half* x;
  const float* y0;
  float* y;
  __half* hws;   // [umax+1][ncols][ffn]
  float* ows;    // [umax+1][ncols][hidden]
  int32_t* err_flag;
  int32_t* uniq_out;
};

// Compact the id list: distinct valid ids in ascending order, the slot of each
// (column, k) pair and the column mask of each slot.
__device__ void moe_route(const MoeDev& p, MoeRoute& R) {
  const int n = p.ncols * p.topk;
  const int t = threadIdx.x;
  if (t < n) R.ids[t] = p.ids[t];
  for (int i = t; i <= MOE_MAXN; i += blockDim.x) R.mask[i] = 0u;
  if (t == 0) { R.U = 0; R.bad = 0; }
  __syncthreads();
  if (t < n) {
    const int id = R.ids[t];
    const bool valid = id >= 0 && id < p.n_expert;
    int f = valid ? 1 : 0;
    for (int j = 0; j < t && f; ++j)
      if (R.ids[j] == id) f = 0;
    R.first[t] = f;
    if (!valid) atomicOr(&R.bad, 1);
  }
  __syncthreads();
  if (t < n) {
    const int id = R.ids[t];
    const bool valid = id >= 0 && id < p.n_expert;
    if (valid) {
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += (R.first[j] && R.ids[j] < id) ? 1 : 0;
      R.slot[t] = rank;
      if (R.first[t]) {
        R.uniq[rank] = id;
        atomicAdd(&R.U, 1);
      }
      atomicOr(&R.mask[rank], 1u << (t / p.topk));
    } else {
      R.slot[t] = -1;
    }
  }
  __syncthreads();
}

// Stage the selected columns of x (column stride `colstride` halves, k wide)
// as f32 in the consumption order of qt, one 32-element block per thread.
__device__ __forceinline__ void stage_x_rt(int qt, float* xs, int xstride, const __half* x,
                                           size_t colstride, uint32_t cmask, int ncols,
                                           int k) {
  const int nbk = k / QK;
  for (int it = threadIdx.x; it < ncols * nbk; it += blockDim.x) {
    const int c = it / nbk, b = it % nbk;
    if (!((cmask >> c) & 1u)) continue;
    stage_block(qt, xs + c * xstride, xstride / QK, b, x + (size_t)c * colstride + (size_t)b * QK);
  }
}

template <int QT>
__device__ __forceinline__ void expert_ptrs(const MoeDev& p, const MoeRoute& R, int u,
                                            bool gateup, const uint8_t*& qa,
                                            const uint16_t*& sa, const uint8_t*& qb,
                                            const uint16_t*& sb) {
  constexpr int QB = QTraits<QT>::QB;
  if (u == p.umax) {
    qa = gateup ? p.sqg : p.sqd;
    sa = gateup ? p.ssg : p.ssd;
    qb = p.squ;
    sb = p.ssu;
    return;
  }
  const size_t e = (size_t)R.uniq[u];
  const size_t gu_q = (size_t)p.ffn * (p.hidden / QK) * QB;
  const size_t gu_s = (size_t)p.ffn * (p.hidden / QK);
  if (gateup) {
    qa = p.qg + e * gu_q;
    sa = p.sg + e * gu_s;
    qb = p.qu + e * gu_q;
    sb = p.su + e * gu_s;
  } else {
    qa = p.qd + e * gu_q;  // down [hidden][ffn] has the same size as gate/up
    sa = p.sd + e * gu_s;
    qb = nullptr;
    sb = nullptr;
  }
}

template <int QT>
__global__ void __launch_bounds__(MOE_THREADS) moe_gate_up_kernel(const MoeDev p) {
  __shared__ MoeRoute R;
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);
  constexpr int QB = QTraits<QT>::QB;
  moe_route(p, R);
  if (blockIdx.x == 0) {
    const int n = p.ncols * p.topk;
    if (p.uniq_out)
      for (int i = threadIdx.x; i < n; i += blockDim.x) p.uniq_out[i] = i < R.U ? R.uniq[i] : -1;
    if (threadIdx.x == 0 && R.bad && p.err_flag) atomicOr(p.err_flag, (int32_t)QG_MOE_BAD_ID);
  }
  const int k = p.hidden;
  stage_x_rt(QT, xs, k, p.x, (size_t)k, 0xffffffffu, p.ncols, k);
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = k / QK;
  const size_t rowbytes = (size_t)nb * QB;
  const int ntile = (p.ffn + MOE_TILE - 1) / MOE_TILE;
  const int nunits = (p.umax + 1) * ntile;
  const uint32_t allc = p.ncols >= 32 ? 0xffffffffu : ((1u << p.ncols) - 1u);
  for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
    const int u = unit / ntile, tile = unit % ntile;
    if (u == p.umax ? !p.has_shared : u >= R.U) continue;
    const uint32_t cm = u == p.umax ? allc : R.mask[u];
    const uint8_t *qa, *qb;
    const uint16_t *sa, *sb;
    expert_ptrs<QT>(p, R, u, true, qa, sa, qb, sb);
    const int r0 = tile * MOE_TILE + warp * MOE_RW;
    int rowidx[MOE_RW];
#pragma unroll
    for (int r = 0; r < MOE_RW; ++r) rowidx[r] = min(r0 + r, p.ffn - 1);
    for (int c = 0; c < p.ncols; ++c) {
      if (!((cm >> c) & 1u)) continue;
      float ta[MOE_RW], tb[MOE_RW];
#pragma unroll
      for (int r = 0; r < MOE_RW; ++r) { ta[r] = 0.f; tb[r] = 0.f; }
      cc_rowdot_1col<QT, MOE_RW, true>(qa, sa, qb, sb, rowbytes, nb, rowidx, xs + c * k, nb, 0,
                                       nb, lane, ta, tb);
      int idx, idx2;
      const float g = warp_transpose_reduce<MOE_RW>(ta, lane, idx);
      const float uu = warp_transpose_reduce<MOE_RW>(tb, lane, idx2);
      if ((lane & (32 / MOE_RW - 1)) == 0) {
        const int row = r0 + idx;
        if (row < p.ffn)
          p.hws[((size_t)u * p.ncols + c) * p.ffn + row] = __float2half_rn(silu_f32(g) * uu);
      }
    }
  }
}

template <int QT>
__global__ void __launch_bounds__(MOE_THREADS) moe_down_kernel(const MoeDev p) {
  __shared__ MoeRoute R;
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);
  constexpr int QB = QTraits<QT>::QB;
  moe_route(p, R);
  const int k = p.ffn;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nb = k / QK;
  const size_t rowbytes = (size_t)nb * QB;
  const int ntile = (p.hidden + MOE_TILE - 1) / MOE_TILE;
  const int nunits = (p.umax + 1) * ntile;
  const uint32_t allc = p.ncols >= 32 ? 0xffffffffu : ((1u << p.ncols) - 1u);
  for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x) {
    const int u = unit / ntile, tile = unit % ntile;
    if (u == p.umax ? !p.has_shared : u >= R.U) continue;  // uniform over the CTA
    const uint32_t cm = u == p.umax ? allc : R.mask[u];
    __syncthreads();
    stage_x_rt(QT, xs, k, p.hws + (size_t)u * p.ncols * k, (size_t)k, cm, p.ncols, k);
    __syncthreads();
    const uint8_t *qa, *qb;
    const uint16_t *sa, *sb;
    expert_ptrs<QT>(p, R, u, false, qa, sa, qb, sb);
    const int r0 = tile * MOE_TILE + warp * MOE_RW;
    int rowidx[MOE_RW];
#pragma unroll
    for (int r = 0; r < MOE_RW; ++r) rowidx[r] = min(r0 + r, p.hidden - 1);
    for (int c = 0; c < p.ncols; ++c) {
      if (!((cm >> c) & 1u)) continue;
      float ta[MOE_RW], tb[MOE_RW];
#pragma unroll
      for (int r = 0; r < MOE_RW; ++r) { ta[r] = 0.f; tb[r] = 0.f; }
      cc_rowdot_1col<QT, MOE_RW, false>(qa, sa, nullptr, nullptr, rowbytes, nb, rowidx,
                                        xs + c * k, nb, 0, nb, lane, ta, tb);
      int idx;
      const float v = warp_transpose_reduce<MOE_RW>(ta, lane, idx);
      if ((lane & (32 / MOE_RW - 1)) == 0) {
        const int row = r0 + idx;
        if (row < p.hidden) p.ows[((size_t)u * p.ncols + c) * p.hidden + row] = v;
      }
    }
  }
}

__global__ void __launch_bounds__(MOE_THREADS) moe_combine_kernel(const MoeDev p) {
  __shared__ MoeRoute R;
  moe_route(p, R);
  const size_t total = (size_t)p.ncols * p.hidden;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i / p.hidden), r = (int)(i % p.hidden);
    float v = p.y0 ? p.y0[i] : 0.f;
    for (int j = 0; j < p.topk; ++j) {
      const int s = R.slot[c * p.topk + j];
      if (s >= 0) v = fmaf(p.rw[c * p.topk + j], p.ows[((size_t)s * p.ncols + c) * p.hidden + r], v);
    }
    if (p.has_shared) v += p.ows[((size_t)p.umax * p.ncols + c) * p.hidden + r];
    p.y[i] = v;
  }
}

static size_t align256(size_t b) { return (b + 255) & ~(size_t)255; }

static int moe_umax(int n_expert, int ncols, int topk) {
  const int n = ncols * topk;
  return n_expert < n ? n_expert : n;
}

size_t moe_ws_bytes(int n_expert, int ffn, int hidden, int ncols, int topk) {
  const size_t slots = (size_t)moe_umax(n_expert, ncols, topk) + 1;
  return align256(slots * ncols * ffn * sizeof(__half)) + align256(slots * ncols * hidden * sizeof(float));
}

bool moe_shape_supported(int ffn, int hidden, int ncols) {
  return (size_t)ncols * hidden <= MOE_XSMEM_FLOATS && (size_t)ncols * ffn <= MOE_XSMEM_FLOATS;
}

template <class K>
static cudaError_t launch_persistent(K kern, int nunits, size_t smem, const MoeDev& d,
                                     cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int occ = 1;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, MOE_THREADS, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  long grid = nunits;
  const long maxg = (long)device_sm_count() * occ;
  if (grid > maxg) grid = maxg;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, MOE_THREADS, smem, s>>>(d);
  note_launch();
  return cudaGetLastError();
}

cudaError_t moe_forward(const MoeArgs& a, cudaStream_t s) {
  MoeDev d{};
  d.qt = a.qt;
  d.qg = (const uint8_t*)a.qg; d.qu = (const uint8_t*)a.qu; d.qd = (const uint8_t*)a.qd;
  d.sg = a.sg; d.su = a.su; d.sd = a.sd;
  d.n_expert = a.n_expert; d.ffn = a.ffn; d.hidden = a.hidden;
  d.ids = a.ids; d.rw = a.rw; d.topk = a.topk; d.ncols = a.ncols;
  d.umax = moe_umax(a.n_expert, a.ncols, a.topk);
  d.has_shared = a.has_shared ? 1 : 0;
  d.sqg = (const uint8_t*)a.sqg; d.squ = (const uint8_t*)a.squ; d.sqd = (const uint8_t*)a.sqd;
  d.ssg = a.ssg; d.ssu = a.ssu; d.ssd = a.ssd;
  d.x = reinterpret_cast<const __half*>(a.x);
  d.y0 = a.y0; d.y = a.y;
  const size_t slots = (size_t)d.umax + 1;
  d.hws = reinterpret_cast<__half*>(a.ws);
  d.ows = reinterpret_cast<float*>(static_cast<char*>(a.ws) + align256(slots * a.ncols * a.ffn * sizeof(__half)));
  d.err_flag = a.err_flag;
  d.uniq_out = a.uniq_out;

  const int ntile_gu = (a.ffn + MOE_TILE - 1) / MOE_TILE;
  const int ntile_dn = (a.hidden + MOE_TILE - 1) / MOE_TILE;
  const size_t smem_gu = (size_t)a.ncols * a.hidden * sizeof(float);
  const size_t smem_dn = (size_t)a.ncols * a.ffn * sizeof(float);
  cudaError_t e;
  if (a.qt == T_Q4_0) {
    e = launch_persistent(moe_gate_up_kernel<T_Q4_0>, (int)slots * ntile_gu, smem_gu, d, s);
    if (e != cudaSuccess) return e;
    e = launch_persistent(moe_down_kernel<T_Q4_0>, (int)slots * ntile_dn, smem_dn, d, s);
  } else {
    e = launch_persistent(moe_gate_up_kernel<T_Q8_0>, (int)slots * ntile_gu, smem_gu, d, s);
    if (e != cudaSuccess) return e;
    e = launch_persistent(moe_down_kernel<T_Q8_0>, (int)slots * ntile_dn, smem_dn, d, s);
  }
  if (e != cudaSuccess) return e;
  const size_t total = (size_t)a.ncols * a.hidden;
  int grid = (int)((total + MOE_THREADS - 1) / MOE_THREADS);
  if (grid > 4 * device_sm_count()) grid = 4 * device_sm_count();
  moe_combine_kernel<<<grid, MOE_THREADS, 0, s>>>(d);
  note_launch();
  return cudaGetLastError();
}

}  // namespace qg
