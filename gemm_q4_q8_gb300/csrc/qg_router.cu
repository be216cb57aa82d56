// qg_router.cu -- MoE router: logits, top-k experts and routing weights, on
// the GPU, producing the device id list that qmoe_experts reads.
//
// "Engine and kernels" (pooled.run), section "Kernel families": the MoE runs
// router, top-k, expert gate/up and down and the weighted combine all on the
// GPU, so routing needs no readback; section "Fewer passes": lowest-index
// tie-breaking. The router weights are f32 ("Architecture", section "Memory
// and caching": f16/bf16 tensors become f32 on load). Routing weights: a
// softmax over each column's selected logits.
//
// GB300 design: one cluster of 16 CTAs. Each warp owns experts e (one at a
// time) and computes their logits for every column in one sweep of the
// expert's router row: 16 float4 loads per lane in flight at once, x read from
// shared memory (staged as f32 on the float4 sweep, so each column's four
// values are one load with no conversion; f16 on the scalar one), f32
// accumulation in a fixed lane order, then a fixed
// butterfly. The column count is a template parameter (1, 2, 4, 8 or 16) so a
// narrow call issues no instructions for columns it does not have. Lane c of
// the warp stores the logit of column c straight into the shared memory of CTA
// c (distributed shared memory, made visible by the cluster barrier), so CTA c
// then holds every logit of column c. Each expert gets a 64-bit key (the order
// of qargmax_f32: numbers before NaN, larger first, ties to the lower index).
// A threshold T (the k-th largest of 32 segment maxima) leaves only the keys
// that can be in the top k; each of those is ranked by counting the candidates
// that beat it, and since keys are distinct the experts of rank < k land in
// distinct slots. One warp then normalises their exponentials.
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int RT_CLUSTER = 16;
constexpr int RT_THREADS = 512;
constexpr int RT_WARPS = RT_THREADS / 32;
constexpr int RT_MAXE = 1024;                  // experts
constexpr int RT_MAXC = 16;                    // columns (one CTA of the cluster each)
constexpr int RT_MAXK = 32;                    // top-k
constexpr int RT_U = 16;                       // float4 loads in flight per lane
constexpr size_t RT_XS_MAX = 200 * 1024;       // x staged in shared memory up to this size

__device__ __forceinline__ uint64_t rt_key(float v, uint32_t i) {
  const uint32_t b = __float_as_uint(v);
  uint32_t k;
  if (v != v) k = 0u;
  else if ((b & 0x7fffffffu) == 0u) k = 0x80000000u;
  else k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)k << 32) | (uint64_t)(~i);
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Logits of expert row wr for NC columns (lanes hold partial sums; caller
// reduces). VEC: float4 rows (hidden % 4 == 0, 8-byte aligned x rows).
template <int NC, bool VEC, bool XF>
__device__ __forceinline__ void rt_row(const float* __restrict__ wr, const __half* xb,
                                       const float* xf, int hidden, int ncols, int lane,
                                       float (&acc)[NC]) {
#pragma unroll
  for (int c = 0; c < NC; ++c) acc[c] = 0.f;
  if (VEC) {
    // lane owns k = base + 128u + 4 lane .. +3; all RT_U loads issued first
    for (int base = 0; base < hidden; base += 128 * RT_U) {
      float4 wv[RT_U];
#pragma unroll
      for (int u = 0; u < RT_U; ++u) {
        const int k = base + 128 * u + 4 * lane;
        wv[u] = k < hidden ? __ldg(reinterpret_cast<const float4*>(wr + k))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < RT_U; ++u) {
        const int k = base + 128 * u + 4 * lane;
        if (k < hidden) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            if (NC == 1 || c < ncols) {
              float2 a, b;
              if (XF) {
                const float4 xv = *reinterpret_cast<const float4*>(xf + (size_t)c * hidden + k);
                a = make_float2(xv.x, xv.y);
                b = make_float2(xv.z, xv.w);
              } else {
                const uint2 hv = *reinterpret_cast<const uint2*>(xb + (size_t)c * hidden + k);
                a = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
                b = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
              }
              acc[c] = fmaf(wv[u].x, a.x, acc[c]);
              acc[c] = fmaf(wv[u].y, a.y, acc[c]);
              acc[c] = fmaf(wv[u].z, b.x, acc[c]);
              acc[c] = fmaf(wv[u].w, b.y, acc[c]);
            }
        }
      }
    }
  } else {
#pragma unroll 4
    for (int k = lane; k < hidden; k += 32) {
      const float wv = __ldg(wr + k);
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (NC == 1 || c < ncols) acc[c] = fmaf(wv, __half2float(xb[(size_t)c * hidden + k]), acc[c]);
    }
  }
}

template <int NC, bool XS, bool VEC>
__global__ void __launch_bounds__(RT_THREADS) router_kernel(const float* __restrict__ w,
                                                            const __half* __restrict__ x, int E,
                                                            int hidden, int ncols, int topk,
                                                            float* logits_out, int32_t* ids_out,
                                                            float* rw_out) {
  __shared__ float s_lg[RT_MAXE];              // column `rank`: every expert's logit
  __shared__ uint64_t s_key[RT_MAXE];          // candidates (unordered)
  __shared__ uint64_t s_seg[32];
  __shared__ uint64_t s_thr;
  __shared__ int s_nc;
  __shared__ float s_selv[RT_MAXK];
  __shared__ int s_sele[RT_MAXK];
  extern __shared__ __align__(16) unsigned char rt_smem[];  // x staged as f16 [ncols][hidden]
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  pdl_trigger();
  const int per = (E + RT_CLUSTER - 1) / RT_CLUSTER;
  const int e0 = (int)rank * per;
  const int e1 = min(E, e0 + per);
  pdl_wait();  // x comes from an earlier kernel on the stream
  // staged x: f32 (converted once) on the float4 sweep, f16 on the scalar one
  constexpr bool XF = XS && VEC;
  if (XS) {
    const int n = ncols * hidden;
    if (XF) {
      float* sx = reinterpret_cast<float*>(rt_smem);
      for (int i = t; i < n; i += RT_THREADS) sx[i] = __half2float(x[i]);
    } else {
      __half* sx = reinterpret_cast<__half*>(rt_smem);
      for (int i = t; i < n; i += RT_THREADS) sx[i] = x[i];
    }
    __syncthreads();
  }
  const __half* xb = XS ? reinterpret_cast<const __half*>(rt_smem) : x;
  const float* xf = reinterpret_cast<const float*>(rt_smem);
  // lane c stores column c into CTA c's s_lg
  uint32_t dst = 0;
  if (lane < ncols)
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(dst)
                 : "r"((uint32_t)__cvta_generic_to_shared(s_lg)), "r"((uint32_t)lane));
  for (int e = e0 + warp; e < e1; e += RT_WARPS) {
    float acc[NC];
    rt_row<NC, VEC, XF>(w + (size_t)e * hidden, xb, xf, hidden, ncols, lane, acc);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
    }
    float v = acc[0];
#pragma unroll
    for (int c = 1; c < NC; ++c) v = lane == c ? acc[c] : v;
    if (lane < ncols) {
      st_cluster_f32(dst + 4u * (uint32_t)e, v);
      if (logits_out) logits_out[(size_t)lane * E + e] = v;
    }
  }
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  if ((int)rank >= ncols) return;
  const int c = (int)rank;
  // Pruning: T = the k-th largest of 32 segment maxima (16 threads, up to 2
  // keys each, per segment). At least k keys are >= T, so every top-k key is
  // >= T, and a candidate's rank among all keys equals its rank among the
  // candidates (every key that beats it is also >= T).
  uint64_t mk[2];
  uint64_t m = 0;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = t + h * RT_THREADS;
    mk[h] = e < E ? rt_key(s_lg[e], (uint32_t)e) : 0ull;
    m = mk[h] > m ? mk[h] : m;
  }
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, m, off);
    m = o > m ? o : m;
  }
  if ((t & 15) == 0) s_seg[t >> 4] = m;
  if (t == 0) s_nc = 0;
  __syncthreads();
  if (warp == 0) {
    const uint64_t mi = s_seg[lane];
    int r = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) r += s_seg[j] > mi;
    // the k-th largest maximum: the largest one beaten by at least k-1 others
    uint64_t tv = r >= topk - 1 ? mi : 0ull;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, tv, off);
      tv = o > tv ? o : tv;
    }
    if (lane == 0) s_thr = tv;
  }
  __syncthreads();
  const uint64_t thr = s_thr;
#pragma unroll
  for (int h = 0; h < 2; ++h)
    if (mk[h] != 0ull && mk[h] >= thr) s_key[atomicAdd(&s_nc, 1)] = mk[h];
  __syncthreads();
  // rank the candidates among themselves (distinct keys: distinct ranks)
  const int nc = s_nc;
  for (int i = t; i < nc; i += RT_THREADS) {
    const uint64_t me = s_key[i];
    int cnt = 0;
#pragma unroll 4
    for (int j = 0; j < nc; ++j) cnt += s_key[j] > me;
    if (cnt < topk) {
      const int e = (int)(~(uint32_t)me);
      s_selv[cnt] = s_lg[e];
      s_sele[cnt] = e;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float mine = lane < topk ? s_selv[lane] : 0.f;
    const float mx = s_selv[0];
    // exponentials in rank order, summed in rank order by every lane
    const float ex = lane < topk ? expf(mine - mx) : 0.f;
    float sum = 0.f;
    for (int r = 0; r < topk; ++r) sum += __shfl_sync(0xffffffffu, ex, r);
    if (lane < topk) {
      ids_out[(size_t)c * topk + lane] = s_sele[lane];
      rw_out[(size_t)c * topk + lane] = ex / sum;
    }
  }
}

template <int NC, bool XS, bool VEC>
static cudaError_t router_go(size_t smem, const float* w, const __half* x, int E, int hidden,
                             int ncols, int topk, float* logits, int32_t* ids, float* rw,
                             cudaStream_t s) {
  auto kern = router_kernel<NC, XS, VEC>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), smem, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(RT_CLUSTER), dim3(RT_THREADS), smem, s, RT_CLUSTER, LC_L1, w, x, E,
                    hidden, ncols, topk, logits, ids, rw);
}

cudaError_t router_launch(const float* w, const uint16_t* x, int E, int hidden, int ncols,
                          int topk, float* logits, int32_t* ids, float* rw, cudaStream_t s) {
  const __half* xh = reinterpret_cast<const __half*>(x);
  const bool vec = (hidden % 4) == 0 && (reinterpret_cast<uintptr_t>(x) & 7) == 0;
  const size_t s_x = (size_t)ncols * hidden * (vec ? 4 : 2);
  const bool xs = s_x <= RT_XS_MAX;
  // float4 rows need 16-byte row starts (w itself is 16-byte aligned) and
  // 8-byte x row starts. The choice depends on the pointers and hidden only,
  // never on the column count, so a column's logit is the same bit for bit
  // whatever the number of columns (the lane -> k order differs between the
  // float4 and scalar sweeps).
  if (xs && vec) {
    if (ncols == 1) return router_go<1, true, true>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
    if (ncols <= 2) return router_go<2, true, true>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
    if (ncols <= 4) return router_go<4, true, true>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
    if (ncols <= 8) return router_go<8, true, true>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
    return router_go<16, true, true>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
  }
  if (xs) return router_go<RT_MAXC, true, false>(s_x, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
  if (vec) return router_go<RT_MAXC, false, true>(0, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
  return router_go<RT_MAXC, false, false>(0, w, xh, E, hidden, ncols, topk, logits, ids, rw, s);
}

bool router_shape_ok(int E, int hidden, int ncols, int topk) {
  return E >= 1 && E <= RT_MAXE && hidden >= 1 && ncols >= 1 && ncols <= RT_MAXC && topk >= 1 &&
         topk <= RT_MAXK && topk <= E;
}

}  // namespace qg
