// qg_sample.cu -- greedy argmax and top-k over f32 logit columns.
//
// "Engine and kernels" (pooled.run), section "Kernel families": sampling is a
// greedy argmax or a top-k on the GPU, so a token reads back a few bytes
// instead of the logits; section "Fewer passes": lowest-index tie-breaking, as
// the CPU loop does.
//
// Order. Every element gets a 64-bit rank key: the high word maps the f32
// value to an unsigned integer that orders like the value (+0 and -0 map to
// the same word, NaN maps to 0 so it ranks below every number, -inf included),
// the low word is the complement of the index, so of two equal values the
// lower index has the larger key. Keys are distinct, the largest key is the
// first-ranked element, and any reduction order gives the same answer.
//
// GB300 design: a column is read by a cluster of CTAs (16 for argmax, 8 for
// top-k), each over its share with two rounds of 8 independent loads per
// thread in flight.
//  * argmax: warp, CTA and then cluster maximum of the keys (distributed shared
//    memory, read by the rank-0 CTA).
//  * top-k (k <= 256): each CTA keeps a shared-memory candidate buffer; an
//    element enters only if its key beats the CTA's current k-th best. When the
//    buffer fills, a bitonic sort keeps the best k and raises the bar. The
//    rank-0 CTA merges the 8 lists (8k keys) with one more bitonic sort.
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int SMP_CLUSTER = 8;              // CTAs per column for top-k
constexpr int AMX_CLUSTER = 16;             // CTAs per column for argmax (non-portable size)
constexpr int SMP_THREADS = 512;
constexpr int SMP_E = 8;                        // elements per thread per round
constexpr int SMP_ROUND = SMP_THREADS * SMP_E;  // elements per CTA per round
constexpr int SMP_BUF = 2 * SMP_ROUND;          // candidate buffer (keys)

__device__ __forceinline__ uint64_t rank_key(float v, uint32_t i) {
  const uint32_t b = __float_as_uint(v);
  uint32_t k;
  if (v != v) k = 0u;                              // NaN: below every number
  else if ((b & 0x7fffffffu) == 0u) k = 0x80000000u;  // +0 and -0 are equal
  else k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((uint64_t)k << 32) | (uint64_t)(~i);
}
__device__ __forceinline__ uint32_t key_index(uint64_t key) { return ~(uint32_t)key; }

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(const void* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"((uint32_t)__cvta_generic_to_shared(local)), "r"(rank));
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}

// The share of column c that CTA `rank` of `parts` reads: [lo, hi).
__device__ __forceinline__ void chunk_of(int n, uint32_t rank, int parts, int& lo, int& hi) {
  const int per = (n + parts - 1) / parts;
  lo = (int)rank * per;
  hi = min(n, lo + per);
  if (lo > n) lo = n;
}

// ------------------------------------------------------------------ argmax
__global__ void __launch_bounds__(SMP_THREADS) argmax_kernel(const float* __restrict__ x, int n,
                                                             int32_t* idx_out, float* val_out) {
  __shared__ uint64_t s_warp[SMP_THREADS / 32];
  __shared__ uint64_t s_best;
  const int c = blockIdx.x / AMX_CLUSTER;
  const uint32_t rank = cluster_rank();
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  pdl_trigger();
  pdl_wait();  // the logits come from an earlier kernel on the stream
  const float* col = x + (size_t)c * n;
  int lo, hi;
  chunk_of(n, rank, AMX_CLUSTER, lo, hi);
  uint64_t best = 0;
  float v[SMP_E];
#pragma unroll
  for (int e = 0; e < SMP_E; ++e) {
    const int i = lo + e * SMP_THREADS + t;
    v[e] = i < hi ? __ldg(col + i) : 0.f;
  }
  for (int base = lo; base < hi; base += SMP_ROUND) {
    float w[SMP_E];  // the next round's loads are in flight meanwhile
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = base + SMP_ROUND + e * SMP_THREADS + t;
      w[e] = i < hi ? __ldg(col + i) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = base + e * SMP_THREADS + t;
      if (i < hi) best = umax64(best, rank_key(v[e], (uint32_t)i));
    }
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) v[e] = w[e];
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, off));
  if (lane == 0) s_warp[warp] = best;
  __syncthreads();
  if (t == 0) {
    uint64_t b = 0;
    for (int w = 0; w < SMP_THREADS / 32; ++w) b = umax64(b, s_warp[w]);
    s_best = b;
  }
  cluster_sync();
  if (rank == 0 && t == 0) {
    uint64_t b = 0;
    for (uint32_t r = 0; r < AMX_CLUSTER; ++r) b = umax64(b, ld_dsmem_u64(&s_best, r));
    const uint32_t i = key_index(b);
    idx_out[c] = (int32_t)i;
    if (val_out) val_out[c] = col[i];
  }
  cluster_sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ------------------------------------------------------------------- top-k
// Bitonic sort, descending, of buf[0, m) (m a power of two), all threads.
__device__ void bitonic_desc(uint64_t* buf, int m) {
  for (int size = 2; size <= m; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int p = threadIdx.x; p < (m >> 1); p += blockDim.x) {
        const int lo = ((p & ~(stride - 1)) << 1) | (p & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = buf[lo], b = buf[hi];
        if ((a < b) == desc) {
          buf[lo] = b;
          buf[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_at_least(int v) {
  int m = 1;
  while (m < v) m <<= 1;
  return m;
}

// Keep the best k of buf[0, cnt): sort, return the new bar (the k-th key).
__device__ uint64_t compact(uint64_t* buf, int cnt, int k, int* s_cnt) {
  const int m = pow2_at_least(cnt > k ? cnt : k);
  for (int i = cnt + threadIdx.x; i < m; i += blockDim.x) buf[i] = 0;
  __syncthreads();
  bitonic_desc(buf, m);
  if (threadIdx.x == 0) *s_cnt = k < cnt ? k : cnt;
  __syncthreads();
  return cnt >= k ? buf[k - 1] : 0;
}

__global__ void __launch_bounds__(SMP_THREADS) topk_kernel(const float* __restrict__ x, int n, int k,
                                                           int32_t* idx_out, float* val_out) {
  extern __shared__ uint64_t s_buf[];  // SMP_BUF keys
  __shared__ int s_cnt;
  const int c = blockIdx.x / SMP_CLUSTER;
  const uint32_t rank = cluster_rank();
  const int t = threadIdx.x;
  pdl_trigger();
  pdl_wait();  // the logits come from an earlier kernel on the stream
  const float* col = x + (size_t)c * n;
  int lo, hi;
  chunk_of(n, rank, SMP_CLUSTER, lo, hi);
  if (t == 0) s_cnt = 0;
  __syncthreads();
  float v[SMP_E];
#pragma unroll
  for (int e = 0; e < SMP_E; ++e) {
    const int i = lo + e * SMP_THREADS + t;
    v[e] = i < hi ? __ldg(col + i) : 0.f;
  }
  // Starting bar: the k-th largest of the threads' first-round maxima. Those k
  // maxima are k distinct elements of the chunk, so at least k elements reach
  // the bar and no element of the chunk's top k lies below it.
  uint64_t bar;
  {
    uint64_t mx = 0;
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = lo + e * SMP_THREADS + t;
      if (i < hi) mx = umax64(mx, rank_key(v[e], (uint32_t)i));
    }
    s_buf[t] = mx;
    __syncthreads();
    bitonic_desc(s_buf, SMP_THREADS);
    bar = k <= SMP_THREADS ? s_buf[k - 1] : 0;
    if (bar != 0) --bar;  // keys equal to the bar must still enter
    __syncthreads();
  }
  for (int base = lo; base < hi; base += SMP_ROUND) {
    // the next round's loads are in flight while this round is filtered
    float w[SMP_E];
    const int nb = base + SMP_ROUND;
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = nb + e * SMP_THREADS + t;
      w[e] = i < hi ? __ldg(col + i) : 0.f;
    }
    if (s_cnt > SMP_BUF - SMP_ROUND) bar = compact(s_buf, s_cnt, k, &s_cnt);  // uniform
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = base + e * SMP_THREADS + t;
      if (i < hi) {
        const uint64_t key = rank_key(v[e], (uint32_t)i);
        if (key > bar) s_buf[atomicAdd(&s_cnt, 1)] = key;
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) v[e] = w[e];
  }
  compact(s_buf, s_cnt, k, &s_cnt);  // s_buf[0, k) = this CTA's best, padded with 0
  cluster_sync();
  if (rank == 0) {
    // merge: the 8 lists into this CTA's buffer (8k <= SMP_BUF), one sort
    __syncthreads();
    const int m = pow2_at_least(SMP_CLUSTER * k);
    uint64_t* merged = s_buf + k;  // own list stays in [0, k)
    for (int i = t; i < (SMP_CLUSTER - 1) * k; i += SMP_THREADS) {
      const uint32_t r = 1 + i / k;
      merged[i] = ld_dsmem_u64(&s_buf[i % k], r);
    }
    for (int i = SMP_CLUSTER * k + t; i < m; i += SMP_THREADS) s_buf[i] = 0;
    __syncthreads();
    bitonic_desc(s_buf, m);
    for (int r = t; r < k; r += SMP_THREADS) {
      const uint32_t i = key_index(s_buf[r]);
      idx_out[(size_t)c * k + r] = (int32_t)i;
      if (val_out) val_out[(size_t)c * k + r] = col[i];
    }
  }
  cluster_sync();  // keep every CTA's shared memory alive until rank 0 has read it
}

// ----------------------------------------------------------------- launch
cudaError_t argmax_launch(const float* x, int n, int ncols, int32_t* idx, float* val,
                          cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(argmax_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return launch_pdl(argmax_kernel, dim3((unsigned)(ncols * AMX_CLUSTER)), dim3(SMP_THREADS), 0, s,
                    AMX_CLUSTER, LC_L1, x, n, idx, val);
}

cudaError_t topk_launch(const float* x, int n, int ncols, int k, int32_t* idx, float* val,
                        cudaStream_t s) {
  const size_t smem = (size_t)SMP_BUF * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_kernel, dim3((unsigned)(ncols * SMP_CLUSTER)), dim3(SMP_THREADS), smem,
                    s, SMP_CLUSTER, LC_L1, x, n, k, idx, val);
}

}  // namespace qg
