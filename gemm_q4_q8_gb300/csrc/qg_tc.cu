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
//  * One producer warp streams the packed weights, the f16 scales and the f16
//    activations of the CTA's K range with TMA tiles (128-byte swizzle) into a
//    ring of shared-memory stages guarded by mbarriers; the weight tiles stay
//    packed in shared memory.
//  * Eight consumer warps (4 m-tiles x 2 k-groups) pull the nibble (or int8)
//    words with ldmatrix straight into the A-fragment layout of
//    mma.sync.m16n8k16 and dequantise them exactly to f16 in registers ((q-8)
//    and q are exact in f16). The stored byte order of the blocks (the two
//    8-byte halves of each 16-byte group interleaved) makes the dequantised
//    pairs come out in the natural k order of the fragment, so the B fragments
//    are plain ldmatrix loads of the activation tile. Each 32-weight block's
//    product is scaled by its f16 scale in f32, so the only roundings are the
//    f32 accumulations.
//  * The two k-groups are summed in a fixed order through shared memory, then
//    the cluster's CTAs are summed in rank order by the rank-0 CTA: the other
//    ranks store their partial tiles into its shared memory and arrive on one
//    of its mbarriers (no cluster-wide barrier after the stream), and rank 0
//    runs the epilogue (y = y0 + acc, or h = f16(SiLU(g) * u)). The reduction
//    tree depends only on the shape.
// Every wait is bounded: on timeout the kernel records an error bit in a device
// word and falls through instead of spinning forever.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "qg_async.cuh"
#include "qg_common.cuh"
#include "qg_internal.h"
#include "qg_mma.cuh"

namespace qg {

constexpr int TC_BM = 64;                 // rows per CTA
constexpr int TC_KT = 256;                // weights per stage (one K unit)
constexpr int TC_SMEM_BUDGET = 112 * 1024;  // two CTAs per SM

__device__ int32_t g_tc_error = 0;        // QG_DEV_ERR_WAIT: a wait timed out

// ------------------------------------------------------------- PTX helpers
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  return mbar_wait(bar, parity, &g_tc_error);
}
// ------------------------------------------------------------ parameters
struct TcParams {
  int rows, k, ncols;
  int units;   // K / TC_KT
  int ksplit;  // CTAs per cluster along K
  int ns;      // pipeline stages
  const __half* x;
  const float* y0;
  float* y;
  __half* h;
};

// KG k-groups of consumer warps split a unit's 8 blocks (8 / KG blocks per warp
// and unit); 4 m-tiles x KG k-groups of consumers plus one TMA producer warp.
// Two k-groups, measured against the alternatives: one k-group of four warps,
// each an m-tile across the whole unit, is slower (Q4_0 5120 x 5120 at one
// column 7.3 -> 6.9 us, twins 17408 x 5120 11.8 -> 11.4 us with two); four
// k-groups, 16 consumer warps with half the work each, are slower too (every
// warp pays the per-stage overhead); two units per stage behind one pair of
// barriers are no faster.
template <int QT, int NT, bool DUAL>
struct TcShape {
  static constexpr int KG = 2;
  static constexpr int BPW = 8 / KG;                     // blocks per warp and unit
  static constexpr int CONS = 4 * KG;                    // consumer warps
  static constexpr int THREADS = (CONS + 1) * 32;        // + the producer warp (last)
  static constexpr int NMAT = DUAL ? 2 : 1;
  static constexpr int QROW = QT == T_Q4_0 ? 128 : 256;  // quant bytes per row per unit
  static constexpr int A_BYTES = TC_BM * QROW;
  static constexpr int S_BYTES = TC_BM * 16;             // 8 f16 scales per row per unit
  static constexpr int AS_BYTES = NMAT * (A_BYTES + S_BYTES);  // weights of one unit (TMA)
  static constexpr int CPAD = 8 * NT;
  static constexpr int X_BYTES = CPAD * TC_KT * 2;       // x of one unit (TMA), [4][CPAD][64] f16
  static constexpr int STAGE = AS_BYTES + X_BYTES;
  // Release a stage as soon as its bytes are in registers (before the
  // arithmetic) on the memory-bound plan, the single-matrix Q8_0 one: its
  // refill then overlaps this stage's arithmetic (measured: Q8_0 LM head 192
  // -> 188.6 us). Where the arithmetic is the bound (Q4_0, fused gate/up) the
  // release stays after it: releasing early there only added waits, or spills.
  static constexpr bool EARLY_RELEASE = QT == T_Q8_0 && NT == 1 && !DUAL;
  static constexpr int NF = 4 * NT * NMAT;               // accumulator floats per lane
  static constexpr int SLOT = 4 * 32 * NF * 4;           // one CTA's partial tile
};

template <int QT, int NT, bool DUAL>
__global__ void __launch_bounds__(TcShape<QT, NT, DUAL>::THREADS, 2)
tc_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mS0,
          const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mS1,
          const __grid_constant__ CUtensorMap mX, const TcParams p) {
  using S = TcShape<QT, NT, DUAL>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int ns = p.ns;
  uint8_t* stages = smem;
  // the partial tiles that the other CTAs of the cluster send to rank 0
  float* cscratch = reinterpret_cast<float*>(smem + (size_t)ns * S::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)ns * S::STAGE +
                                               (size_t)(p.ksplit - 1) * S::SLOT);  // A, S, x landed
  uint64_t* empty = full + ns;                                                 // stage free
  uint64_t* sent = empty + ns;  // rank 0: the other ranks' partial tiles have landed
  // Shared-memory addresses as 32-bit values; stage s starts at st0 + s * STAGE,
  // its barriers at full0 + 8 s and empty0 + 8 s.
  const uint32_t st0 = smem_u32(stages);
  const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = blockIdx.x % p.ksplit;
  const int tile = blockIdx.x / p.ksplit;
  const int m0 = tile * TC_BM;
  const int u0 = (int)((long)rank * p.units / p.ksplit);
  const int u1 = (int)((long)(rank + 1) * p.units / p.ksplit);
  const int nu = u1 - u0;

  // Stage layout: [A, S (weights)] [x: 4 boxes of [CPAD][64] f16, 128-byte
  // swizzle]. full[s]: the TMA bytes of the stage; empty[s]: the consumers.
  if (tid == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], S::CONS);
    }
    // one arrival per lane of the k-group-0 consumer warps of every other rank
    if (p.ksplit > 1) mbar_init(sent, (uint32_t)(p.ksplit - 1) * 4 * 32);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // The other ranks touch this CTA's barrier only after the matching cluster
  // wait below, by which time every CTA of the cluster has initialised its own.
  if (p.ksplit > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  const bool producer = warp == S::CONS;
  // Dependents may launch at once: another tensor-core GEMM queues its CTAs
  // behind this grid's and issues its first weight loads as soon as it lands.
  // The host never lets a CUDA-core kernel follow this one programmatically
  // (LC_SMEM -> LC_L1 in launch_pdl): it would inherit this kernel's
  // shared-memory carve-out and stream far slower with that little L1 left.
  pdl_trigger();
  if (producer) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      auto load_weights = [&](uint32_t st, uint32_t fb, int u) {
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m) {
          const CUtensorMap* mA = m == 0 ? &mA0 : &mA1;
          const CUtensorMap* mS = m == 0 ? &mS0 : &mS1;
          const uint32_t a = st + m * S::A_BYTES;
#pragma unroll
          for (int bx = 0; bx < S::QROW / 128; ++bx)
            tma_load_2d(a + bx * TC_BM * 128, mA, u * S::QROW + bx * 128, m0, fb, pol_w);
          tma_load_2d(st + S::NMAT * S::A_BYTES + m * S::S_BYTES, mS, u * 8, m0, fb, pol_w);
        }
      };
      auto load_x = [&](uint32_t st, uint32_t fb, int u) {
        // x[0..CPAD)[u*256 .. u*256+256) as [4][CPAD][64] (3-D map, see tc_launch)
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(st + S::AS_BYTES),
            "l"(&mX), "r"(0), "r"(0), "r"(u * 4), "r"(fb)
            : "memory");
      };
      // The weights of the first ring's worth of stages are requested before
      // waiting for the previous kernel on the stream (it never writes them);
      // their x follows the wait.
      const int npre = nu < ns ? nu : ns;
      for (int i = 0; i < npre; ++i) {
        mbar_expect_tx(full0 + 8 * i, (uint32_t)S::STAGE);
        load_weights(st0 + i * S::STAGE, full0 + 8 * i, u0 + i);
      }
      pdl_wait();
      for (int i = 0; i < npre; ++i) load_x(st0 + i * S::STAGE, full0 + 8 * i, u0 + i);
      // stage s and phase bit ph advance incrementally (no division in the loop)
      for (int i = npre, s = 0, ph = 1; i < nu; ++i, s = s + 1 == ns ? 0 : s + 1, ph ^= s == 0) {
        if (!mbar_wait(empty0 + 8 * s, (uint32_t)(ph ^ 1))) break;
        const uint32_t st = st0 + s * S::STAGE, fb = full0 + 8 * s;
        mbar_expect_tx(fb, (uint32_t)S::STAGE);
        load_x(st, fb, u0 + i);
        load_weights(st, fb, u0 + i);
      }
    }
    __syncwarp();
  }

  const int mi = warp & 3, kj = warp >> 2;  // m-tile, k-group (the producer: kj == KG)
  const int g = lane >> 2, t = lane & 3;
  float y0v[NT][4];  // the epilogue's residual (rank 0, k-group 0; loaded before the loop)
  float acc[S::NMAT][NT][4];
#pragma unroll
  for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[m][n][e] = 0.f;

  if (!producer) {
    // The OR pattern of the Q4_0 dequantisation, held in a register for the
    // whole loop (an opaque move: the compiler neither folds it into an
    // immediate, which would split each extraction in two, nor reloads it).
    uint32_t M;
    asm volatile("mov.b32 %0, 0x64006400;" : "=r"(M));
    // k-group kj owns the BPW contiguous blocks BPW*kj .. BPW*kj + BPW - 1 of
    // every unit (block b of the warp: unit block BPW*kj + b).
    // ldmatrix source of this lane: lanes 0-7 rows 0-7 and lanes 8-15 rows 8-15
    // of the m-tile at chunk c; lanes 16-31 the same rows at chunk c+1. The
    // swizzled byte offsets depend only on the lane and k-group: computed once.
    constexpr int BPW = S::BPW;
    const int lrow = mi * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int lchunk = lane >> 4;
    constexpr int NL = QT == T_Q4_0 ? BPW / 2 : BPW;  // A ldmatrix.x4 per matrix and stage
    uint32_t aoff[NL];  // Q4_0: blocks (2l, 2l+1) of the warp; Q8_0: block l (both halves)
#pragma unroll
    for (int l = 0; l < NL; ++l) {
      int chunk, box;
      if (QT == T_Q4_0) {  // 16 bytes per block and row: one 128-byte box
        chunk = BPW * kj + 2 * l + lchunk;
        box = 0;
      } else {             // 32 bytes per block and row: blocks 4 bx .. 4 bx + 3 in box bx
        const int b = BPW * kj + l;
        chunk = 2 * (b & 3) + lchunk;
        box = b >> 2;
      }
      aoff[l] = (uint32_t)(box * TC_BM * 128 + lrow * 128 + ((chunk ^ (lrow & 7)) << 4));
    }
    const uint32_t soff_g = (uint32_t)(S::NMAT * S::A_BYTES + (mi * 16 + g) * 16 + 2 * BPW * kj);
    // B fragments: ldmatrix.x4 of x rows (columns) n*8 + (lane & 7) at the k
    // offsets 0, 8, 16, 24 of a block (matrix lane >> 3). Unit block b lies in
    // x box b >> 1 at 16-byte chunk 4(b & 1) + (lane >> 3), stored at
    // chunk ^ row (the 128-byte swizzle; rows are 128 bytes).
    const int lm = lane >> 3, lr = lane & 7;
    const uint32_t boff = (uint32_t)(S::AS_BYTES + (BPW * kj >> 1) * S::CPAD * 128 + lr * 128);
    const uint32_t xo0 = boff + (uint32_t)((lm ^ lr) << 4), xo1 = boff + (uint32_t)(((4 + lm) ^ lr) << 4);
    if (!DUAL && p.y0 && kj == 0 && rank == 0 && nu > 0) {
      // The epilogue's residual, fetched before the stream rather than after
      // it (its DRAM round trip then overlaps the stream). It comes from an
      // earlier kernel on the stream: wait for that kernel first. Nothing is
      // lost by waiting here: the first stage's x follows the same wait.
      pdl_wait();
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = m0 + mi * 16 + g + ((e >> 1) << 3);
          const int col = n * 8 + 2 * t + (e & 1);
          y0v[n][e] = (row < p.rows && col < p.ncols) ? p.y0[(size_t)col * p.rows + row] : 0.f;
        }
    }
    uint32_t st = st0, fb = full0, eb = empty0;
    for (int i = 0, s = 0, ph = 0; i < nu; ++i) {
      if (!mbar_wait(fb, (uint32_t)ph)) break;
      // the BPW f16 scales of rows g and g+8 for this k-group's blocks, per matrix
      float dg[S::NMAT][BPW], dg8[S::NMAT][BPW];
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m) {
        uint32_t a[4], b[4];
        if (BPW == 8) {
          lds128(st + soff_g + m * S::S_BYTES, a[0], a[1], a[2], a[3]);
          lds128(st + soff_g + m * S::S_BYTES + 128, b[0], b[1], b[2], b[3]);  // row g + 8
        } else if (BPW == 4) {
          lds64(st + soff_g + m * S::S_BYTES, a[0], a[1]);
          lds64(st + soff_g + m * S::S_BYTES + 128, b[0], b[1]);  // row g + 8
        } else {
          a[0] = lds32(st + soff_g + m * S::S_BYTES);
          b[0] = lds32(st + soff_g + m * S::S_BYTES + 128);
        }
#pragma unroll
        for (int q = 0; q < BPW / 2; ++q) {
          dg[m][2 * q] = lo_f32(a[q]); dg[m][2 * q + 1] = hi_f32(a[q]);
          dg8[m][2 * q] = lo_f32(b[q]); dg8[m][2 * q + 1] = hi_f32(b[q]);
        }
      }
      // All shared-memory reads of the stage are issued first: the raw quant
      // words of rows g and g+8 (Q4_0: one ldmatrix covers blocks j, j+1;
      // Q8_0: one covers both 16-element halves of block j) and the B
      // fragments of the four blocks.
      uint32_t W[S::NMAT][NL][4];
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
        for (int l = 0; l < NL; ++l)
          ldsm_x4(st + m * S::A_BYTES + aoff[l], W[m][l][0], W[m][l][1], W[m][l][2], W[m][l][3]);
      uint4 bf[BPW][NT];
#pragma unroll
      for (int j = 0; j < BPW; ++j)
#pragma unroll
        for (int n = 0; n < NT; ++n)
          ldsm_x4(st + ((j & 1) ? xo1 : xo0) + (uint32_t)((j >> 1) * S::CPAD * 128 + n * 1024),
                  bf[j][n].x, bf[j][n].y, bf[j][n].z, bf[j][n].w);
      // Early release: the whole stage is now in registers. The proxy fence
      // makes the release wait until this thread's shared-memory reads of the
      // stage have completed (the stage is refilled by TMA, the async proxy,
      // once every consumer has arrived).
      auto release = [&]() {
        __syncwarp();
        mbar_arrive_lane0(eb, lane);
        if (++s == ns) {  // next stage (ring of ns; the phase bit flips at the wrap)
          s = 0;
          ph ^= 1;
          st = st0; fb = full0; eb = empty0;
        } else {
          st += S::STAGE; fb += 8; eb += 8;
        }
      };
      if (S::EARLY_RELEASE) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        release();
      }
      // Then the blocks as a software pipeline: the tensor pipe takes a new
      // mma only every few cycles, so block j's two dependent mma are issued
      // around the dequantisation of block j + 1, and block j - 1's scale FMAs
      // follow once its sums are out.
      uint32_t A0[BPW][S::NMAT][4], A1[BPW][S::NMAT][4];
      float fr[BPW][S::NMAT][NT][4];
      auto dequant = [&](int j) {
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m) {
          if (QT == T_Q4_0) {
            const uint32_t wg = W[m][j >> 1][(j & 1) ? 2 : 0];
            const uint32_t wg8 = W[m][j >> 1][(j & 1) ? 3 : 1];
            uint32_t e0, e1, e2, e3, f0, f1, f2, f3;
            dq4_f16(wg, M, e0, e1, e2, e3);
            dq4_f16(wg8, M, f0, f1, f2, f3);
            A0[j][m][0] = e0; A0[j][m][1] = f0; A0[j][m][2] = e2; A0[j][m][3] = f2;
            A1[j][m][0] = e1; A1[j][m][1] = f1; A1[j][m][2] = e3; A1[j][m][3] = f3;
          } else {
            uint32_t p0, p1, q0, q1;
            dq8_f16(W[m][j][0], p0, p1);
            dq8_f16(W[m][j][1], q0, q1);
            A0[j][m][0] = p0; A0[j][m][1] = q0; A0[j][m][2] = p1; A0[j][m][3] = q1;
            dq8_f16(W[m][j][2], p0, p1);
            dq8_f16(W[m][j][3], q0, q1);
            A1[j][m][0] = p0; A1[j][m][1] = q0; A1[j][m][2] = p1; A1[j][m][3] = q1;
          }
        }
      };
      auto mma_lo = [&](int j) {
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n) mma16816(fr[j][m][n], A0[j][m], bf[j][n].x, bf[j][n].y);
      };
      auto mma_hi = [&](int j) {
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n) mma16816_acc(fr[j][m][n], A1[j][m], bf[j][n].z, bf[j][n].w);
      };
      auto scale = [&](int j) {
#pragma unroll
        for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            acc[m][n][0] = fmaf(dg[m][j], fr[j][m][n][0], acc[m][n][0]);
            acc[m][n][1] = fmaf(dg[m][j], fr[j][m][n][1], acc[m][n][1]);
            acc[m][n][2] = fmaf(dg8[m][j], fr[j][m][n][2], acc[m][n][2]);
            acc[m][n][3] = fmaf(dg8[m][j], fr[j][m][n][3], acc[m][n][3]);
          }
      };
      dequant(0);
#pragma unroll
      for (int j = 0; j < BPW; ++j) {
        mma_lo(j);
        if (j + 1 < BPW) dequant(j + 1);
        mma_hi(j);
        if (j > 0) scale(j - 1);
      }
      scale(BPW - 1);
      if (!S::EARLY_RELEASE) {
        // Release after the arithmetic, behind the same proxy fence as the
        // early release: the stage's reads (ldmatrix, ld.shared) are generic-
        // proxy accesses and its refill is a TMA write (async proxy), so only
        // the fence orders the reads before the refill. Data dependences do
        // not: the instruction scheduler may place the arithmetic that
        // consumes the reads after the arrive. (Measured: a build whose block
        // scales used packed FMAs refilled stages under live reads and gave
        // wrong, run-to-run different sums on the 16-column down projection
        // without this fence, and correct ones with it.)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        release();
      }
    }
  }

  // y0, y and h are read or written only after every earlier kernel on the
  // stream has finished
  pdl_wait();
  // ---- reduce the k-groups in shared memory (fixed order: kj 0 + kj 1 + ...)
  float* scratch = reinterpret_cast<float*>(stages);
  if (!producer) {
    asm volatile("bar.sync 1, %0;" ::"n"(S::CONS * 32) : "memory");
    if (kj > 0) {
      float* dst = scratch + (size_t)((kj - 1) * 4 * 32 + mi * 32 + lane) * S::NF;
      int q = 0;
#pragma unroll
      for (int m = 0; m < S::NMAT; ++m)
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[q++] = acc[m][n][e];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(S::CONS * 32) : "memory");
    if (kj == 0) {
#pragma unroll
      for (int r = 1; r < S::KG; ++r) {
        const float* srcp = scratch + (size_t)((r - 1) * 4 * 32 + mi * 32 + lane) * S::NF;
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

  // ---- reduce the cluster's K splits in rank order through distributed smem:
  // each other rank's k-group-0 warps store their partial tile into rank 0's
  // cscratch and arrive (release, cluster scope) on rank 0's `sent` barrier;
  // rank 0 waits for the phase (acquire, cluster scope) and adds the partials
  // in rank order. No rank waits for another except rank 0 for the partials,
  // and no CTA's shared memory is written after that CTA has been waited for.
  if (p.ksplit > 1) {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every `sent` initialised
    if (!producer && kj == 0) {
      if (rank != 0) {
        const uint32_t local = smem_u32(cscratch) +
                               (uint32_t)(((rank - 1) * 4 * 32 + mi * 32 + lane) * S::NF * 4);
        uint32_t remote, rbar;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(0));
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(smem_u32(sent)), "r"(0));
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
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar)
                     : "memory");
      } else {
        mbar_wait_cluster(smem_u32(sent), 0, &g_tc_error);
        for (int r = 1; r < p.ksplit; ++r) {
          const float* srcp = cscratch + (size_t)(((r - 1) * 4 * 32) + mi * 32 + lane) * S::NF;
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
        if (p.y0) v += nu > 0 ? y0v[n][e] : p.y0[o];
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
  int ksplit, ns;
  size_t smem;
};

// Pinned per shape: depends only on (type, columns, dual, rows, k), never on
// the device, so the reduction order is the same on every GPU. The K split is
// the largest (at most 8) whose clusters all fit in one wave of a GB300: the
// tables hold, per cluster size, how many clusters the part keeps resident at
// once (measured with cudaOccupancyMaxActiveClusters for these kernels; two
// CTAs per SM, or one for the large-stage plan). Each CTA then streams as much
// K as possible, which amortises its start-up and reduction. Stages: as many
// as fit, up to the CTA's whole K range.
constexpr int kClusterCap2[9] = {0, 304, 152, 97, 74, 58, 46, 38, 36};  // 2 CTAs / SM
constexpr int kClusterCap1[9] = {0, 152, 76, 46, 36, 28, 23, 15, 15};   // 1 CTA / SM

template <int QT, int NT, bool DUAL>
TcConfig pick_config_budget(int rows, int k, size_t budget, const int (&cap)[9]) {
  using S = TcShape<QT, NT, DUAL>;
  const int units = k / TC_KT;
  const int ntile = (rows + TC_BM - 1) / TC_BM;
  int ks = 8;
  while (ks > 1 && (ks > units || ntile > cap[ks])) --ks;
  for (; ks >= 1; --ks) {
    const int nu_max = (units + ks - 1) / ks;
    // Shared memory: 1 KB of alignment slack, the ring, the partial tiles that
    // the other ranks of the cluster send to rank 0 (the k-group partials
    // reuse the ring), and 2 ns + 1 mbarriers.
    const size_t cscr = (size_t)(ks - 1) * S::SLOT;
    auto need = [&](int n) { return 1024 + (size_t)n * S::STAGE + cscr + (2 * (size_t)n + 1) * 8; };
    int ns = nu_max < 8 ? nu_max : 8;
    while (ns >= 1 && need(ns) > budget) --ns;
    if (ns < 2 && nu_max >= 2) continue;
    if (ns < 1) continue;
    if ((long long)ns * S::STAGE < (long long)(S::KG - 1) * S::SLOT) continue;
    return TcConfig{ks, ns, need(ns)};
  }
  return TcConfig{0, 0, 0};
}

// Two CTAs per SM when the shape allows it, else one.
template <int QT, int NT, bool DUAL>
TcConfig pick_config(int rows, int k) {
  TcConfig c = pick_config_budget<QT, NT, DUAL>(rows, k, TC_SMEM_BUDGET, kClusterCap2);
  if (c.ksplit == 0) c = pick_config_budget<QT, NT, DUAL>(rows, k, 220 * 1024, kClusterCap1);
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
  // x as a 3-D view of the [ncols][k] f16 array: {64 elements, column, k/64},
  // strides 2k and 128 bytes, so one box {64, CPAD, 4} brings a unit's 256 k as
  // four [CPAD][64] tiles (128-byte swizzle); columns past ncols read as zero.
  CUtensorMap mX;
  {
    auto enc = get_encode();
    if (!enc) return cudaErrorInvalidValue;
    cuuint64_t dims[3] = {64, (cuuint64_t)ncols, (cuuint64_t)k / 64};
    cuuint64_t strides[2] = {(cuuint64_t)k * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)S::CPAD, 4};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&mX, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(x), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.rows = rows;
  p.k = k;
  p.ncols = ncols;
  p.units = k / TC_KT;
  p.ksplit = cfg.ksplit;
  p.ns = cfg.ns;
  p.x = reinterpret_cast<const __half*>(x);
  p.y0 = y0;
  p.y = y;
  p.h = reinterpret_cast<__half*>(h);
  auto kern = tc_kernel<QT, NT, DUAL>;
  const cudaError_t e = prepare_kernel(reinterpret_cast<const void*>(kern), cfg.smem, false);
  if (e != cudaSuccess) return e;
  const int ntile = (rows + TC_BM - 1) / TC_BM;
  (void)S::NF;
  return launch_pdl(kern, dim3((unsigned)(ntile * cfg.ksplit)), dim3(S::THREADS), cfg.smem, s,
                    cfg.ksplit, LC_SMEM, mA0, mS0, mA1, mS1, mX, p);
}

}  // namespace

// Shapes the tensor-core plan takes: K a multiple of 256, any column count
// from 1 to 16, except that matrices of at most 2^22 weights with K <= 3072
// keep 1-8 columns on the CUDA cores (their fixed latency is lower there:
// 2048 x 2048 Q8_0 takes 2.7 us on CUDA cores and 6.8 us here at 1 column,
// 7.3 and 6.8 us at 8). For 1-8 columns the choice depends on the matrix only,
// and the plan is the same (one n-tile of 8), so the 1-column GEMV and its
// 2-8-column twins give bit-identical columns: the mma computes each output
// column from that column alone, and the CUDA-core twins repeat the 1-column
// arithmetic column by column.
bool tc_supported(int qt, int ncols, bool dual, int rows, int k) {
  if (k <= 0 || k % TC_KT != 0 || ncols < 1 || ncols > 16 || rows <= 0) return false;
  if (ncols <= 8 && (long long)rows * k <= (1LL << 22) && k <= 3072) return false;
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

// ------------------------------------------ self-test of the bounded waits
// (diagnostic, not part of the method)
__device__ int32_t g_wait_selftest[2];

// One thread waits on phase 0 of a fresh mbarrier that nothing arrives on:
// first with CTA scope (the form of the stage waits), then with cluster-scope
// acquire (the form of the K-split handoff). Each wait gives up after its clock
// bound, sets QG_DEV_ERR_WAIT in the device error word and returns false;
// g_wait_selftest[i] records 1 if wait i completed, 0 if it gave up.
__global__ void wait_selftest_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    g_wait_selftest[0] = mbar_wait(smem_u32(&bar), 0) ? 1 : 0;
    g_wait_selftest[1] = mbar_wait_cluster(smem_u32(&bar), 0, &g_tc_error) ? 1 : 0;
  }
}

}  // namespace qg

extern "C" qg_status qg_wait_selftest(int32_t* completed_out, cudaStream_t stream) {
  if (!completed_out) return QG_ERR_NULL;
  const int32_t unset[2] = {-1, -1};
  cudaError_t e = cudaMemcpyToSymbolAsync(qg::g_wait_selftest, unset, sizeof(unset), 0,
                                          cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) {
    qg::wait_selftest_kernel<<<1, 32, 0, stream>>>();
    e = cudaGetLastError();
    if (e == cudaSuccess) qg::note_launch();
  }
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbolAsync(completed_out, qg::g_wait_selftest, sizeof(unset), 0,
                                  cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    qg::note_cuda_error(e);
    return QG_ERR_CUDA;
  }
  return QG_OK;
}

extern "C" qg_status qg_device_error(int32_t* bits_out) {
  if (!bits_out) return QG_ERR_NULL;
  int32_t v = 0;
  const int32_t zero = 0;
  if (cudaMemcpyFromSymbol(&v, qg::g_tc_error, sizeof(v)) != cudaSuccess) return QG_ERR_CUDA;
  if (cudaMemcpyToSymbol(qg::g_tc_error, &zero, sizeof(zero)) != cudaSuccess) return QG_ERR_CUDA;
  int32_t m = 0;
  if (qg::moe_device_error(&m) != cudaSuccess) return QG_ERR_CUDA;
  *bits_out = v | m;
  return QG_OK;
}
