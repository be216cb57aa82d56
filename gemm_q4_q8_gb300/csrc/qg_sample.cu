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
// GB300 design: a column is read by a cluster of 16 CTAs, each over its share
// with 8 independent loads per thread in flight (float4 when the column
// allows, else two rounds of scalar loads).
//  * argmax: warp, CTA and then cluster maximum of the keys (distributed shared
//    memory, read by the rank-0 CTA).
//  * top-k (k <= 256), 16 CTAs per column: each CTA reads its chunk once
//    (kept in shared memory when it fits), takes T = the k-th largest of its
//    512 thread maxima (warp sorts in registers, then ranks by binary search),
//    collects the keys >= T (every key of its top k is one) and ranks them by
//    counting (a bitonic sort when there are many; the old streaming filter
//    when they overflow the buffer). Each CTA stores its sorted list into the
//    rank-0 CTA's shared memory, which ranks every entry by its position plus
//    a binary search in each other list and writes the first k.
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int AMX_CLUSTER = 16;             // CTAs per column for argmax (non-portable size)
constexpr int SMP_THREADS = 512;
constexpr int SMP_E = 8;                        // elements per thread per round
constexpr int SMP_ROUND = SMP_THREADS * SMP_E;  // elements per CTA per round
constexpr int SMP_BUF = 2 * SMP_ROUND;          // fallback candidate buffer (keys)
constexpr int TK_CLUSTER = 16;                  // CTAs per column for top-k (non-portable size)
constexpr int TK_CAND = 4096;                   // candidate keys above the threshold
constexpr int TK_RANKED = 512;                  // ranked by counting up to this many
constexpr int TK_STAGE_MAX = 32768;             // chunk floats kept in shared memory
constexpr int TK_MAXK = 256;

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
// V4: float4 loads (every column starts on a 16-byte boundary and n % 4 == 0;
// the CTAs' shares are then multiples of 4 elements): one round of 8 float4
// per thread covers 16,384 elements per CTA.
template <bool V4>
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
  uint64_t best = 0;
  if (V4) {
    const int per = (((n + AMX_CLUSTER - 1) / AMX_CLUSTER) + 3) & ~3;
    lo = min(n, (int)rank * per);
    hi = min(n, lo + per);
    constexpr int R4 = SMP_THREADS * SMP_E * 4;  // elements per CTA per round
    for (int base = lo; base < hi; base += R4) {
      float4 v[SMP_E];
#pragma unroll
      for (int e = 0; e < SMP_E; ++e) {
        const int i = base + (e * SMP_THREADS + t) * 4;
        v[e] = i < hi ? __ldg(reinterpret_cast<const float4*>(col + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int e = 0; e < SMP_E; ++e) {
        const int i = base + (e * SMP_THREADS + t) * 4;
        if (i < hi) {
          best = umax64(best, rank_key(v[e].x, (uint32_t)i));
          best = umax64(best, rank_key(v[e].y, (uint32_t)i + 1));
          best = umax64(best, rank_key(v[e].z, (uint32_t)i + 2));
          best = umax64(best, rank_key(v[e].w, (uint32_t)i + 3));
        }
      }
    }
  } else {
    chunk_of(n, rank, AMX_CLUSTER, lo, hi);
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

// One CTA's top k of col[lo, hi) by streaming (the fallback when too many keys
// pass the threshold of topk_kernel): candidates above a running bar go to
// buf (SMP_BUF keys); when it fills, a sort keeps the best k and raises the
// bar. Leaves buf[0, k) sorted descending, padded with 0.
__device__ void cta_topk_stream(const float* __restrict__ col, int lo, int hi, int k,
                                uint64_t* buf, int* s_cnt) {
  const int t = threadIdx.x;
  if (t == 0) *s_cnt = 0;
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
    buf[t] = mx;
    __syncthreads();
    bitonic_desc(buf, SMP_THREADS);
    bar = k <= SMP_THREADS ? buf[k - 1] : 0;
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
    if (*s_cnt > SMP_BUF - SMP_ROUND) bar = compact(buf, *s_cnt, k, s_cnt);  // uniform
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = base + e * SMP_THREADS + t;
      if (i < hi) {
        const uint64_t key = rank_key(v[e], (uint32_t)i);
        if (key > bar) buf[atomicAdd(s_cnt, 1)] = key;
      }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) v[e] = w[e];
  }
  compact(buf, *s_cnt, k, s_cnt);
}

// Bitonic sort of one key per lane across a warp, descending (lane 0 largest).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t key, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t other = __shfl_xor_sync(0xffffffffu, key, stride);
      const bool desc = (lane & size) == 0 || size == 32;
      const bool lower = (lane & stride) == 0;
      key = (lower == desc) ? umax64(key, other) : (key < other ? key : other);
    }
  }
  return key;
}


// The high word of rank_key: an unsigned word that orders like the value.
__device__ __forceinline__ uint32_t order_word(float v) { return (uint32_t)(rank_key(v, 0u) >> 32); }

// Largest key of a thread's elements, seen in increasing index order: the
// largest word, and on equal words the first (lowest) index.
struct ThreadMax {
  uint32_t w = 0, i = 0;
  bool any = false;
  __device__ __forceinline__ void add(uint32_t word, uint32_t idx) {
    if (!any || word > w) { w = word; i = idx; any = true; }
  }
  __device__ __forceinline__ uint64_t key() const {
    return any ? (((uint64_t)w << 32) | (uint64_t)(~i)) : 0ull;
  }
};

// Rank among the union of the first q entries of 16 descending lists of length
// len (a power of two, `stride` keys apart): entries greater than v.
__device__ __forceinline__ int count_above16_prefix(const uint64_t* lists, int stride, int len,
                                                    int q, uint64_t v) {
  int pos[16];
#pragma unroll
  for (int l = 0; l < 16; ++l) pos[l] = 0;
  for (int h = len >> 1; h >= 1; h >>= 1) {
#pragma unroll
    for (int l = 0; l < 16; ++l) pos[l] += lists[l * stride + pos[l] + h - 1] > v ? h : 0;
  }
  int sum = 0;
#pragma unroll
  for (int l = 0; l < 16; ++l) sum += min(q, pos[l] + (lists[l * stride + pos[l]] > v ? 1 : 0));
  return sum;
}

// Threshold over 16 sorted lists: the k-th largest key among the first
// q = ceil(k/16) entries of every list (16q >= k keys). At least k keys reach
// it, so every key of the top k of the lists' union does. Called by all
// threads; returns the threshold (0 when fewer than k keys are non-zero).
__device__ __forceinline__ uint64_t threshold16(const uint64_t* lists, int stride, int len, int k,
                                                uint64_t* s_out) {
  const int q = min(len, (k + 15) / 16);
  const int t = threadIdx.x;
  if (t == 0) *s_out = 0;
  __syncthreads();
  if (t < 16 * q) {
    const uint64_t v = lists[(t / q) * stride + t % q];
    if (v != 0 && count_above16_prefix(lists, stride, len, q, v) == k - 1) *s_out = v;
  }
  __syncthreads();
  return *s_out;
}

// Keys >= thr among 16 sorted lists into cand (distinct keys), then the first
// k by rank (candidates that beat each one) into out[0, k). Every key that
// beats a top-k key is itself >= thr, so ranks among the candidates are exact
// for the top k.
__device__ __forceinline__ void select16(const uint64_t* lists, int stride, int len, int k,
                                         uint64_t thr, uint64_t* cand, int* s_n,
                                         int32_t* idx_out, float* val_out, const float* col) {
  const int t = threadIdx.x;
  if (t == 0) *s_n = 0;
  __syncthreads();
  for (int e = t; e < 16 * len; e += SMP_THREADS) {
    const uint64_t v = lists[(e / len) * stride + e % len];
    if (v != 0 && v >= thr) cand[atomicAdd(s_n, 1)] = v;
  }
  __syncthreads();
  const int m = *s_n;
  for (int i = t; i < m; i += SMP_THREADS) {
    const uint64_t v = cand[i];
    int r = 0;
    for (int j = 0; j < m; ++j) r += cand[j] > v;
    if (r < k) {
      const uint32_t ix = key_index(v);
      idx_out[r] = (int32_t)ix;
      if (val_out) val_out[r] = col[ix];
    }
  }
}

// Dynamic shared memory of topk_kernel: [stage_bytes: the chunk's order words
// (u32), or the fallback's SMP_BUF keys] [TK_CAND candidate keys]
// [TK_CLUSTER * kp keys, kp = the power of two >= k: in rank 0, every CTA's
// sorted list, 0-padded]. V4: the column rows and the CTAs' chunks start on
// 16-byte boundaries (float4 loads).
template <bool V4>
__global__ void __launch_bounds__(SMP_THREADS) topk_kernel(const float* __restrict__ x, int n, int k,
                                                           int32_t* idx_out, float* val_out,
                                                           int staged, int stage_bytes) {
  extern __shared__ __align__(16) unsigned char tk_smem[];
  uint32_t* s_w = reinterpret_cast<uint32_t*>(tk_smem);
  uint64_t* s_fb = reinterpret_cast<uint64_t*>(tk_smem);
  uint64_t* s_cand = reinterpret_cast<uint64_t*>(tk_smem + stage_bytes);
  uint64_t* s_merge = s_cand + TK_CAND;
  __shared__ uint64_t s_tm[SMP_THREADS];  // thread maxima, sorted per warp
  __shared__ uint64_t s_list[TK_MAXK];    // this CTA's top k, descending, 0-padded
  __shared__ uint64_t s_thr;
  __shared__ int s_nc;
  const int c = blockIdx.x / TK_CLUSTER;
  const uint32_t rank = cluster_rank();
  const int t = threadIdx.x, lane = t & 31;
  pdl_trigger();
  pdl_wait();  // the logits come from an earlier kernel on the stream
  const float* col = x + (size_t)c * n;
  int lo, hi;
  {
    // chunks of a multiple of 4 elements for float4 loads
    const int per = V4 ? (((n + TK_CLUSTER - 1) / TK_CLUSTER + 3) & ~3) : (n + TK_CLUSTER - 1) / TK_CLUSTER;
    lo = min(n, (int)rank * per);
    hi = min(n, lo + per);
  }
  const int len = hi - lo;

  // Pass 1: every element once, each thread's largest key, and the chunk's
  // order words kept in shared memory when they fit.
  ThreadMax tm;
  if (V4) {
    const float4* c4 = reinterpret_cast<const float4*>(col + lo);
    uint4* w4 = reinterpret_cast<uint4*>(s_w);
    const int nq = len >> 2;  // len is a multiple of 4 (n is)
    constexpr int R = 2 * SMP_THREADS;  // quads per round: two per thread
    float4 v0 = t < nq ? __ldg(c4 + t) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v1 = t + SMP_THREADS < nq ? __ldg(c4 + t + SMP_THREADS) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < nq; base += R) {
      const int q0 = base + R + t, q1 = q0 + SMP_THREADS;
      const float4 n0 = q0 < nq ? __ldg(c4 + q0) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 n1 = q1 < nq ? __ldg(c4 + q1) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int qq = base + t + h * SMP_THREADS;
        if (qq < nq) {
          const float4 v = h ? v1 : v0;
          const uint4 w = make_uint4(order_word(v.x), order_word(v.y), order_word(v.z), order_word(v.w));
          if (staged) w4[qq] = w;
          const uint32_t i0 = (uint32_t)(lo + 4 * qq);
          tm.add(w.x, i0); tm.add(w.y, i0 + 1); tm.add(w.z, i0 + 2); tm.add(w.w, i0 + 3);
        }
      }
      v0 = n0;
      v1 = n1;
    }
  } else {
    float v[SMP_E];
#pragma unroll
    for (int e = 0; e < SMP_E; ++e) {
      const int i = e * SMP_THREADS + t;
      v[e] = i < len ? __ldg(col + lo + i) : 0.f;
    }
    for (int base = 0; base < len; base += SMP_ROUND) {
      float w[SMP_E];
#pragma unroll
      for (int e = 0; e < SMP_E; ++e) {
        const int i = base + SMP_ROUND + e * SMP_THREADS + t;
        w[e] = i < len ? __ldg(col + lo + i) : 0.f;
      }
#pragma unroll
      for (int e = 0; e < SMP_E; ++e) {
        const int i = base + e * SMP_THREADS + t;
        if (i < len) {
          const uint32_t ow = order_word(v[e]);
          if (staged) s_w[i] = ow;
          tm.add(ow, (uint32_t)(lo + i));
        }
      }
#pragma unroll
      for (int e = 0; e < SMP_E; ++e) v[e] = w[e];
    }
  }
  // Threshold T over the 16 warp-sorted lists of thread maxima: the k-th
  // largest among their first ceil(k/16) entries. Those k maxima are distinct
  // elements of the chunk, so every element of the chunk's top k is >= T.
  s_tm[t] = warp_sort_desc(tm.key(), lane);
  const int kp = pow2_at_least(k);  // list length in the merge area
  for (int i = t; i < kp; i += SMP_THREADS) s_list[i] = 0;
  if (t == 0) s_nc = 0;
  const uint64_t thr = threshold16(s_tm, 32, 32, k, &s_thr);
  // Pass 2: the candidates, keys >= T (from the staged words when staged).
  if (staged && V4) {
    const uint4* w4 = reinterpret_cast<const uint4*>(s_w);
    const int nq = len >> 2;
#pragma unroll 2
    for (int qq = t; qq < nq; qq += SMP_THREADS) {
      const uint4 w = w4[qq];
      const uint32_t i0 = (uint32_t)(lo + 4 * qq);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t key = ((uint64_t)ws[j] << 32) | (uint64_t)(~(i0 + j));
        if (key >= thr) {
          const int p = atomicAdd(&s_nc, 1);
          if (p < TK_CAND) s_cand[p] = key;
        }
      }
    }
  } else {
#pragma unroll 4
    for (int i = t; i < len; i += SMP_THREADS) {
      const uint32_t ow = staged ? s_w[i] : order_word(__ldg(col + lo + i));
      const uint64_t key = ((uint64_t)ow << 32) | (uint64_t)(~(uint32_t)(lo + i));
      if (key >= thr) {
        const int p = atomicAdd(&s_nc, 1);
        if (p < TK_CAND) s_cand[p] = key;
      }
    }
  }
  __syncthreads();
  const int nc = s_nc;
  if (nc <= TK_RANKED) {
    // rank each candidate by the candidates that beat it (distinct keys)
    for (int i = t; i < nc; i += SMP_THREADS) {
      const uint64_t key = s_cand[i];
      int r = 0;
      for (int j = 0; j < nc; ++j) r += s_cand[j] > key;
      if (r < k) s_list[r] = key;
    }
  } else if (nc <= TK_CAND) {
    const int m = pow2_at_least(nc);
    for (int i = nc + t; i < m; i += SMP_THREADS) s_cand[i] = 0;
    __syncthreads();
    bitonic_desc(s_cand, m);
    for (int i = t; i < k; i += SMP_THREADS) s_list[i] = s_cand[i];
  } else {
    __shared__ int s_cnt;
    cta_topk_stream(col, lo, hi, k, s_fb, &s_cnt);
    for (int i = t; i < k; i += SMP_THREADS) s_list[i] = s_fb[i];
  }
  __syncthreads();
  // every CTA's list into rank 0's merge area, made visible by the barrier
  {
    uint32_t dst;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;"
                 : "=r"(dst)
                 : "r"((uint32_t)__cvta_generic_to_shared(s_merge)));
    for (int i = t; i < kp; i += SMP_THREADS)
      asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(dst + 8u * (uint32_t)((int)rank * kp + i)),
                   "l"(s_list[i])
                   : "memory");
  }
  cluster_sync();
  if (rank == 0) {
    // the same threshold over the 16 lists, then the survivors ranked
    static_assert(TK_CLUSTER == 16, "the merge searches 16 lists");
    const uint64_t thr2 = threshold16(s_merge, kp, kp, k, &s_thr);
    select16(s_merge, kp, kp, k, thr2, s_cand, &s_nc, idx_out + (size_t)c * k,
             val_out ? val_out + (size_t)c * k : nullptr, col);
  }
}

// ----------------------------------------------------------------- launch
cudaError_t argmax_launch(const float* x, int n, int ncols, int32_t* idx, float* val,
                          cudaStream_t s) {
  const bool v4 = (n % 4) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  auto kern = v4 ? argmax_kernel<true> : argmax_kernel<false>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), 0, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)(ncols * AMX_CLUSTER)), dim3(SMP_THREADS), 0, s,
                    AMX_CLUSTER, LC_L1, x, n, idx, val);
}

cudaError_t topk_launch(const float* x, int n, int ncols, int k, int32_t* idx, float* val,
                        cudaStream_t s) {
  // float4 loads when every column row starts on a 16-byte boundary
  const bool v4 = (n % 4) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const long per = ((long)n + TK_CLUSTER - 1) / TK_CLUSTER;
  const long chunk = v4 ? ((per + 3) & ~3L) : per;
  const int staged = chunk <= TK_STAGE_MAX ? 1 : 0;
  size_t stage_bytes = staged ? (((size_t)chunk * sizeof(uint32_t) + 15) & ~(size_t)15) : 0;
  if (stage_bytes < (size_t)SMP_BUF * sizeof(uint64_t)) stage_bytes = (size_t)SMP_BUF * sizeof(uint64_t);
  int kp = 1;
  while (kp < k) kp <<= 1;
  const size_t smem = stage_bytes + ((size_t)TK_CAND + (size_t)TK_CLUSTER * kp) * sizeof(uint64_t);
  auto kern = v4 ? topk_kernel<true> : topk_kernel<false>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), smem, true);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)(ncols * TK_CLUSTER)), dim3(SMP_THREADS), smem, s,
                    TK_CLUSTER, LC_L1, x, n, k, idx, val, staged, (int)stage_bytes);
}

}  // namespace qg
