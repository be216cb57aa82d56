// qg_tc.cu -- tensor-core skinny GEMM for 2..16 columns (twins, prefill GEMM,
// fused gate/up).
//
// "Engine and kernels" (pooled.run), section "Kernel families": the prefill
// GEMM is row-stationary with the weight tile kept packed in shared memory, and
// section "Batching and prefill": split-K is pinned per shape so every device
// computes identical results. The twins (2..8 columns) read each weight block
// once for all live columns.
//
// GB300 design. A CTA owns 64 rows (4 m-tiles of 16) and a contiguous K range;
// the CTAs that split K for the same rows form a thread-block cluster.
//  * One producer warp streams the packed weights and f16 scales of the CTA's
//    K range with 2-D TMA tiles (128-byte swizzle) into a ring of shared-memory
//    stages guarded by mbarriers; the tiles stay packed in shared memory.
//  * Eight consumer warps (4 m-tiles x 2 k-groups) pull the nibble (or int8)
//    words with ldmatrix straight into the A-fragment layout of
//    mma.sync.m16n8k16, dequantise them exactly to f16 in registers ((q-8) and
//    q are exact in f16), and multiply with the f16 activations (B fragments,
//    pre-permuted once per CTA so the k order matches the dequantised pairs).
//    Each 32-weight block's product is scaled by its f16 scale in f32, so the
//    only roundings are the f32 accumulations.
//  * The two k-groups are summed in a fixed order through shared memory, then
//    the cluster's CTAs are summed in rank order through distributed shared
//    memory by the rank-0 CTA, which runs the epilogue (y = y0 + acc, or
//    h = f16(SiLU(g) * u)). The reduction tree depends only on the shape.
// Every wait is bounded: on timeout the kernel records an error bit in a device
// word and falls through instead of spinning forever.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

constexpr int TC_BM = 64;                 // rows per CTA
constexpr int TC_KT = 256;                // weights per stage (one K unit)
constexpr int TC_CONSUMERS = 8;           // 4 m-tiles x 2 k-groups
constexpr int TC_THREADS = (TC_CONSUMERS + 1) * 32;
constexpr int TC_SMEM_BUDGET = 112 * 1024;  // two CTAs per SM
constexpr long long TC_WAIT_LIMIT = 4000000000LL;  // cycles (~2 s) before giving up

__device__ int32_t g_tc_error = 0;        // bit 1: a wait timed out

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a phase of an mbarrier; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > TC_WAIT_LIMIT) {
      atomicOr(&g_tc_error, 1);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint16_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
// D = A * B (+ C), f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f), "f"(0.f),
        "f"(0.f), "f"(0.f));
}
__device__ __forceinline__ void mma16816_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t hsub2_u(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}

// ------------------------------------------------------ exact f16 dequant
// Q4_0: word w = bytes 4t..4t+3 of one row of a block (byte j holds element j
// low, j+16 high). 0x6400 is f16 1024 (one mantissa step = 1). Results:
//   e0 = (el 4t, 4t+2), e1 = (4t+16, 4t+18), e2 = (4t+1, 4t+3), e3 = (4t+17, 4t+19)
// each equal to (q - 8), exactly.
__device__ __forceinline__ void dq4_f16(uint32_t w, uint32_t& e0, uint32_t& e1, uint32_t& e2,
                                        uint32_t& e3) {
  const uint32_t w8 = w >> 8;
  const uint32_t M = 0x64006400u;
  const uint32_t k1032 = 0x64086408u;  // 1032 = 1024 + 8
  const uint32_t k16th = 0x2C002C00u;  // 1/16
  const uint32_t km72 = 0xD480D480u;   // -72
  e0 = hsub2_u((w & 0x000F000Fu) | M, k1032);
  e2 = hsub2_u((w8 & 0x000F000Fu) | M, k1032);
  e1 = hfma2_u((w & 0x00F000F0u) | M, k16th, km72);   // (1024 + 16 q) / 16 - 72 = q - 8
  e3 = hfma2_u((w8 & 0x00F000F0u) | M, k16th, km72);
}
// Q8_0: word w = int8 elements 4t..4t+3 of a 16-element half block:
//   p0 = (el 4t, 4t+2), p1 = (4t+1, 4t+3), exactly q.
__device__ __forceinline__ void dq8_f16(uint32_t w, uint32_t& p0, uint32_t& p1) {
  const uint32_t u = w ^ 0x80808080u;          // q + 128
  const uint32_t k1152 = 0x64806480u;          // 1024 + 128
  p0 = hsub2_u(__byte_perm(u, 0x64646464u, 0x4240), k1152);
  p1 = hsub2_u(__byte_perm(u, 0x64646464u, 0x4341), k1152);
}

// ------------------------------------------------------------ parameters
struct TcParams {
  int rows, k, ncols;
  int units;   // K / TC_KT
  int ksplit;  // CTAs per cluster along K
  int ns;      // pipeline stages
  int nu_max;  // K units of the largest split
  const __half* x;
  const float* y0;
  float* y;
  __half* h;
};

template <int QT, int NT, bool DUAL>
struct TcShape {
  static constexpr int NMAT = DUAL ? 2 : 1;
  static constexpr int QROW = QT == T_Q4_0 ? 128 : 256;  // quant bytes per row per unit
  static constexpr int A_BYTES = TC_BM * QROW;
  static constexpr int S_BYTES = TC_BM * 16;             // 8 f16 scales per row per unit
  static constexpr int STAGE = NMAT * (A_BYTES + S_BYTES);
  static constexpr int CPAD = 8 * NT;
  static constexpr int XP_UNIT = 8 * CPAD * 64;          // permuted x bytes per unit
  static constexpr int NF = 4 * NT * NMAT;               // accumulator floats per lane
  static constexpr int SLOT = 4 * 32 * NF * 4;           // one CTA's partial tile
};

template <int QT, int NT, bool DUAL>
__global__ void __launch_bounds__(TC_THREADS, 2)
tc_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mS0,
          const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mS1,
          const TcParams p) {
  using S = TcShape<QT, NT, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int ns = p.ns;
  uint8_t* stages = smem;
  uint8_t* xperm = smem + (size_t)ns * S::STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(xperm + (size_t)p.nu_max * S::XP_UNIT);
  uint64_t* empty = full + ns;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = blockIdx.x % p.ksplit;
  const int tile = blockIdx.x / p.ksplit;
  const int m0 = tile * TC_BM;
  const int u0 = (int)((long)rank * p.units / p.ksplit);
  const int u1 = (int)((long)(rank + 1) * p.units / p.ksplit);
  const int nu = u1 - u0;

  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], TC_CONSUMERS);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const bool producer = warp == TC_CONSUMERS;
  uint64_t policy = 0;
  auto issue = [&](int i) {  // stage i of this CTA's K range
    const int s = i % ns;
    uint8_t* st = stages + (size_t)s * S::STAGE;
    mbar_expect_tx(&full[s], (uint32_t)S::STAGE);
    const int u = u0 + i;
#pragma unroll
    for (int m = 0; m < S::NMAT; ++m) {
      const CUtensorMap* mA = m == 0 ? &mA0 : &mA1;
      const CUtensorMap* mS = m == 0 ? &mS0 : &mS1;
      uint8_t* a = st + m * S::A_BYTES;
#pragma unroll
      for (int bx = 0; bx < S::QROW / 128; ++bx)
        tma_load_2d(a + bx * TC_BM * 128, mA, u * S::QROW + bx * 128, m0, &full[s], policy);
      tma_load_2d(st + S::NMAT * S::A_BYTES + m * S::S_BYTES, mS, u * 8, m0, &full[s], policy);
    }
  };
  if (producer && lane == 0) {
    policy = policy_evict_first();
    for (int i = 0; i < nu && i < ns; ++i) issue(i);
  }

  // Permute x for this CTA's K range: for block b, column c, lane slot t, the
  // 16 bytes [x4t, x4t+2, x4t+1, x4t+3, x4t+16, x4t+18, x4t+17, x4t+19].
  // Four items per thread per pass, all sixteen 16-byte loads issued first.
  {
    const int items = nu * 8 * S::CPAD;
    for (int base = tid; base < items; base += 4 * TC_THREADS) {
      uint4 q[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * TC_THREADS;
        const int b = it / S::CPAD, c = it % S::CPAD;
        if (it < items && c < p.ncols) {
          const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)c * p.k +
                                                            (size_t)(u0 * 8 + b) * QK);
#pragma unroll
          for (int v = 0; v < 4; ++v) q[u][v] = src[v];
        } else {
#pragma unroll
          for (int v = 0; v < 4; ++v) q[u][v] = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = base + u * TC_THREADS;
        if (it >= items) continue;
        const int b = it / S::CPAD, c = it % S::CPAD;
        const uint32_t lo[8] = {q[u][0].x, q[u][0].y, q[u][0].z, q[u][0].w,
                                q[u][1].x, q[u][1].y, q[u][1].z, q[u][1].w};
        const uint32_t hi[8] = {q[u][2].x, q[u][2].y, q[u][2].z, q[u][2].w,
                                q[u][3].x, q[u][3].y, q[u][3].z, q[u][3].w};
        uint4* dst = reinterpret_cast<uint4*>(xperm + ((size_t)(b * S::CPAD + c) * 4) * 16);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          dst[t] = make_uint4(__byte_perm(lo[2 * t], lo[2 * t + 1], 0x5410),
                              __byte_perm(lo[2 * t], lo[2 * t + 1], 0x7632),
                              __byte_perm(hi[2 * t], hi[2 * t + 1], 0x5410),
                              __byte_perm(hi[2 * t], hi[2 * t + 1], 0x7632));
      }
    }
  }
  __syncthreads();

  const int mi = warp & 3, kj = (warp >> 2) & 1;
  const int g = lane >> 2, t = lane & 3;
  float acc[S::NMAT][NT][4];
#pragma unroll
  for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.f;

  if (producer) {
    if (lane == 0) {
      for (int i = ns; i < nu; ++i) {
        const int s = i % ns;
        if (!mbar_wait(&empty[s], (uint32_t)(((i / ns) - 1) & 1))) break;
        issue(i);
      }
    }
    __syncwarp();
  } else {
    const uint32_t xp_base = smem_u32(xperm);
    // ldmatrix source row/chunk of this lane: lanes 0-7 rows 0-7 and lanes 8-15
    // rows 8-15 of the m-tile at chunk c; lanes 16-31 the same rows at chunk c+1.
    const int lrow = mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int lchunk = lane >> 4;
    const uint32_t srow_g = (uint32_t)((mi * 16 + g) * 16);
    const uint32_t srow_g8 = (uint32_t)((mi * 16 + g + 8) * 16);
    for (int i = 0; i < nu; ++i) {
      const int s = i % ns;
      if (!mbar_wait(&full[s], (uint32_t)((i / ns) & 1))) break;
      const uint32_t st = smem_u32(stages + (size_t)s * S::STAGE);
      const uint32_t sbase = st + S::NMAT * S::A_BYTES;
      // the 8 f16 scales of rows g and g+8 for this unit, per matrix
      uint4 sg4[S::NMAT], sg84[S::NMAT];
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m) {
        sg4[m] = lds128(sbase + m * S::S_BYTES + srow_g);
        sg84[m] = lds128(sbase + m * S::S_BYTES + srow_g8);
      }
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        // Q4_0: blocks (c0, c0+1), c0 = 2kj + 4pr, from one ldmatrix.x4 per matrix.
        // Q8_0: blocks kj + 4pr and kj + 4pr + 2, one ldmatrix.x4 each.
        uint32_t W[S::NMAT][2][4];  // [matrix][block of the pair][r0..r3]
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m) {
          const uint32_t abase = st + m * S::A_BYTES;
          if (QT == T_Q4_0) {
            const int chunk = 2 * kj + 4 * pr + lchunk;
            uint32_t r0, r1, r2, r3;
            ldsm_x4(abase + (uint32_t)(lrow * 128 + ((chunk ^ (lrow & 7)) << 4)), r0, r1, r2, r3);
            W[m][0][0] = r0; W[m][0][1] = r1; W[m][1][0] = r2; W[m][1][1] = r3;
            W[m][0][2] = W[m][0][3] = W[m][1][2] = W[m][1][3] = 0;
          } else {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const int blk = kj + 4 * pr + 2 * sub;
              const int bx = blk >> 2, chunk = 2 * (blk & 3) + lchunk;
              ldsm_x4(abase + (uint32_t)(bx * TC_BM * 128 + lrow * 128 + ((chunk ^ (lrow & 7)) << 4)),
                      W[m][sub][0], W[m][sub][1], W[m][sub][2], W[m][sub][3]);
            }
          }
        }
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const int blk = QT == T_Q4_0 ? (2 * kj + 4 * pr + sub) : (kj + 4 * pr + 2 * sub);
          uint4 bf[NT];
#pragma unroll
          for (int n = 0; n < NT; ++n)
            bf[n] = lds128(xp_base + (uint32_t)((((i * 8 + blk) * S::CPAD + n * 8 + g) * 4 + t) * 16));
#pragma unroll
          for (int m = 0; m < S::NMAT; ++m) {
            uint32_t A0[4], A1[4];
            if (QT == T_Q4_0) {
              uint32_t e0, e1, e2, e3, f0, f1, f2, f3;
              dq4_f16(W[m][sub][0], e0, e1, e2, e3);
              dq4_f16(W[m][sub][1], f0, f1, f2, f3);
              A0[0] = e0; A0[1] = f0; A0[2] = e2; A0[3] = f2;
              A1[0] = e1; A1[1] = f1; A1[2] = e3; A1[3] = f3;
            } else {
              uint32_t p0, p1, q0, q1;
              dq8_f16(W[m][sub][0], p0, p1);
              dq8_f16(W[m][sub][1], q0, q1);
              A0[0] = p0; A0[1] = q0; A0[2] = p1; A0[3] = q1;
              dq8_f16(W[m][sub][2], p0, p1);
              dq8_f16(W[m][sub][3], q0, q1);
              A1[0] = p0; A1[1] = q0; A1[2] = p1; A1[3] = q1;
            }
            // scale of block blk (word blk/2, half blk%2) without indexed registers:
            // Q4_0: word kj + 2pr, half sub; Q8_0: word 2pr + sub, half kj.
            uint32_t sw, sw8;
            bool hi_half;
            if (QT == T_Q4_0) {
              const uint32_t a0 = pr ? sg4[m].z : sg4[m].x, a1 = pr ? sg4[m].w : sg4[m].y;
              const uint32_t b0 = pr ? sg84[m].z : sg84[m].x, b1 = pr ? sg84[m].w : sg84[m].y;
              sw = kj ? a1 : a0;
              sw8 = kj ? b1 : b0;
              hi_half = sub != 0;
            } else {
              const int wi = 2 * pr + sub;
              sw = wi == 0 ? sg4[m].x : (wi == 1 ? sg4[m].y : (wi == 2 ? sg4[m].z : sg4[m].w));
              sw8 = wi == 0 ? sg84[m].x : (wi == 1 ? sg84[m].y : (wi == 2 ? sg84[m].z : sg84[m].w));
              hi_half = kj != 0;
            }
            const float dg = h2f((uint16_t)(hi_half ? (sw >> 16) : (sw & 0xffffu)));
            const float dg8 = h2f((uint16_t)(hi_half ? (sw8 >> 16) : (sw8 & 0xffffu)));
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              float fr[4];
              mma16816(fr, A0, bf[n].x, bf[n].y);
              mma16816_acc(fr, A1, bf[n].z, bf[n].w);
              float2 lo = fma2(make_float2(dg, dg), make_float2(fr[0], fr[1]),
                               make_float2(acc[m][n][0], acc[m][n][1]));
              float2 hi = fma2(make_float2(dg8, dg8), make_float2(fr[2], fr[3]),
                               make_float2(acc[m][n][2], acc[m][n][3]));
              acc[m][n][0] = lo.x; acc[m][n][1] = lo.y;
              acc[m][n][2] = hi.x; acc[m][n][3] = hi.y;
            }
          }
        }
      }
      // The stage was read through the generic proxy (ldmatrix / ld.shared) and
      // is refilled by TMA through the async proxy: order the reads before the
      // release with a proxy fence, or the refill can overtake them.
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }

  // ---- reduce the two k-groups (fixed order: kj 0 + kj 1) in shared memory
  float* scratch = reinterpret_cast<float*>(stages);
  if (!producer) {
    asm volatile("bar.sync 1, %0;" ::"n"(TC_CONSUMERS * 32) : "memory");
    if (kj == 1) {
      float* dst = scratch + (size_t)(mi * 32 + lane) * S::NF;
      int q = 0;
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[q++] = acc[m][n][e];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(TC_CONSUMERS * 32) : "memory");
    if (kj == 0) {
      const float* srcp = scratch + (size_t)(mi * 32 + lane) * S::NF;
      int q = 0;
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[m][n][e] += srcp[q++];
    }
  }

  // ---- reduce the cluster's K splits in rank order through distributed smem
  if (p.ksplit > 1) {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (!producer && kj == 0 && rank != 0) {
      const uint32_t local = smem_u32(stages) +
                             (uint32_t)(((rank - 1) * 4 * 32 + mi * 32 + lane) * S::NF * 4);
      uint32_t remote;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(0));
      int q = 0;
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote + 4 * q), "f"(acc[m][n][e])
                         : "memory");
            ++q;
          }
    }
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    if (!producer && kj == 0 && rank == 0) {
      for (int r = 1; r < p.ksplit; ++r) {
        const float* srcp = scratch + (size_t)(((r - 1) * 4 * 32) + mi * 32 + lane) * S::NF;
        int q = 0;
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[m][n][e] += srcp[q++];
      }
    }
  }

  // ---- epilogue (rank 0, k-group 0)
  if (producer || kj != 0 || rank != 0) return;
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = m0 + mi * 16 + g + ((e >> 1) << 3);
      const int col = n * 8 + 2 * t + (e & 1);
      if (row >= p.rows || col >= p.ncols) continue;
      const size_t o = (size_t)col * p.rows + row;
      if (DUAL) {
        p.h[o] = __float2half_rn(silu_f32(acc[0][n][e]) * acc[S::NMAT - 1][n][e]);
      } else {
        float v = acc[0][n][e];
        if (p.y0) v += p.y0[o];
        p.y[o] = v;
      }
    }
}

// ----------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D map over a row-major [rows][cols] array of `esize`-byte elements.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)esize};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct TcConfig {
  int ksplit, ns, nu_max;
  size_t smem;
};

// Pinned per shape: depends only on (type, columns, dual, rows, k), never on
// the device, so the reduction order is the same on every GPU.
template <int QT, int NT, bool DUAL>
TcConfig pick_config_budget(int rows, int k, size_t budget) {
  using S = TcShape<QT, NT, DUAL>;
  const int units = k / TC_KT;
  const int ntile = (rows + TC_BM - 1) / TC_BM;
  const int target = 304;  // CTAs that fill two per SM on a 152-SM part
  TcConfig best{0, 0, 0, 0};
  for (int ks = 1; ks <= 8 && ks <= units; ++ks) {
    const int nu_max = (units + ks - 1) / ks;
    for (int ns = 6; ns >= 3; --ns) {
      const size_t reuse = (size_t)ns * S::STAGE + (size_t)nu_max * S::XP_UNIT;
      const size_t smem = 1024 + reuse + 2 * ns * sizeof(uint64_t);
      if (smem > budget) continue;
      if ((size_t)S::SLOT > reuse || (size_t)(ks - 1) * S::SLOT > reuse) continue;
      best = {ks, ns, nu_max, smem};
      break;
    }
    if (best.ksplit == ks && (long)ntile * ks >= target) break;
  }
  return best;
}

// Two CTAs per SM when the shape allows it, else one.
template <int QT, int NT, bool DUAL>
TcConfig pick_config(int rows, int k) {
  TcConfig c = pick_config_budget<QT, NT, DUAL>(rows, k, TC_SMEM_BUDGET);
  if (c.ksplit == 0) c = pick_config_budget<QT, NT, DUAL>(rows, k, 220 * 1024);
  return c;
}

template <int QT, int NT, bool DUAL>
bool config_ok(int rows, int k) { return pick_config<QT, NT, DUAL>(rows, k).ksplit > 0; }

template <int QT, int NT, bool DUAL>
cudaError_t tc_launch(const void* q, const uint16_t* scl, const void* qu, const uint16_t* su,
                      int rows, int k, const uint16_t* x, int ncols, const float* y0, float* y,
                      uint16_t* h, cudaStream_t s) {
  using S = TcShape<QT, NT, DUAL>;
  const TcConfig cfg = pick_config<QT, NT, DUAL>(rows, k);
  if (cfg.ksplit == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap mA0, mS0, mA1, mS1;
  const uint64_t qrow = (uint64_t)k / QK * QTraits<QT>::QB;
  if (!make_map(&mA0, q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qrow, rows, 128, TC_BM,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mS0, scl, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)k / QK, rows, 8, TC_BM,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  if (DUAL) {
    if (!make_map(&mA1, qu, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qrow, rows, 128, TC_BM,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mS1, su, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)k / QK, rows, 8, TC_BM,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  } else {
    mA1 = mA0;
    mS1 = mS0;
  }
  TcParams p{};
  p.rows = rows;
  p.k = k;
  p.ncols = ncols;
  p.units = k / TC_KT;
  p.ksplit = cfg.ksplit;
  p.ns = cfg.ns;
  p.nu_max = cfg.nu_max;
  p.x = reinterpret_cast<const __half*>(x);
  p.y0 = y0;
  p.y = y;
  p.h = reinterpret_cast<__half*>(h);
  auto kern = tc_kernel<QT, NT, DUAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.smem);
  if (e != cudaSuccess) return e;
  const int ntile = (rows + TC_BM - 1) / TC_BM;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3((unsigned)(ntile * cfg.ksplit), 1, 1);
  lc.blockDim = dim3(TC_THREADS, 1, 1);
  lc.dynamicSmemBytes = cfg.smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)cfg.ksplit;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, kern, mA0, mS0, mA1, mS1, p);
  note_launch();
  (void)S::NF;
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool tc_supported(int qt, int ncols, bool dual, int rows, int k) {
  if (k <= 0 || k % TC_KT != 0 || ncols < 2 || ncols > 16 || rows <= 0) return false;
  const bool wide = ncols > 8;
  if (qt == T_Q4_0) {
    if (dual) return wide ? config_ok<T_Q4_0, 2, true>(rows, k) : config_ok<T_Q4_0, 1, true>(rows, k);
    return wide ? config_ok<T_Q4_0, 2, false>(rows, k) : config_ok<T_Q4_0, 1, false>(rows, k);
  }
  if (dual) return wide ? config_ok<T_Q8_0, 2, true>(rows, k) : config_ok<T_Q8_0, 1, true>(rows, k);
  return wide ? config_ok<T_Q8_0, 2, false>(rows, k) : config_ok<T_Q8_0, 1, false>(rows, k);
}

cudaError_t tc_gemm(int qt, const void* q, const uint16_t* scl, const void* qu,
                    const uint16_t* su, int rows, int k, const uint16_t* x, int ncols,
                    const float* y0, float* y, uint16_t* h, cudaStream_t s) {
  const bool dual = qu != nullptr;
  const bool wide = ncols > 8;
  if (qt == T_Q4_0) {
    if (dual) return wide ? tc_launch<T_Q4_0, 2, true>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s)
                          : tc_launch<T_Q4_0, 1, true>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s);
    return wide ? tc_launch<T_Q4_0, 2, false>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s)
                : tc_launch<T_Q4_0, 1, false>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s);
  }
  if (dual) return wide ? tc_launch<T_Q8_0, 2, true>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s)
                        : tc_launch<T_Q8_0, 1, true>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s);
  return wide ? tc_launch<T_Q8_0, 2, false>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s)
              : tc_launch<T_Q8_0, 1, false>(q, scl, qu, su, rows, k, x, ncols, y0, y, h, s);
}

}  // namespace qg
