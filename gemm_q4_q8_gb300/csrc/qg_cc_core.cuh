// qg_cc_core.cuh -- CUDA-core building blocks: per-block loads, exact
// dequantisation dot products and x staging, shared by the GEMV and MoE kernels.
#pragma once
#include "qg_common.cuh"

namespace qg {

// One block's quants for one row. load: from global memory (streamed, read
// once); load_shared: from a copy in shared memory (16-byte aligned).
template <int QT> struct Blk;
template <> struct Blk<T_Q4_0> {
  uint4 a;
  __device__ __forceinline__ void load(const uint8_t* p) { a = ld_stream16(p); }
  __device__ __forceinline__ void load_shared(const uint8_t* p) {
    a = *reinterpret_cast<const uint4*>(p);
  }
};
template <> struct Blk<T_Q8_0> {
  uint4 a, b;
  __device__ __forceinline__ void load(const uint8_t* p) {
    a = ld_stream16(p);
    b = ld_stream16(p + 16);
  }
  __device__ __forceinline__ void load_shared(const uint8_t* p) {
    a = reinterpret_cast<const uint4*>(p)[0];
    b = reinterpret_cast<const uint4*>(p)[1];
  }
};

// Dot of one block of one row with one column's staged x (32 floats in the
// consumption order of the quant type). Returns the unscaled block sum.
__device__ __forceinline__ float blk_dot(const Blk<T_Q4_0>& q, const float2 (&xr)[16]) {
  float2 acc = make_float2(0.f, 0.f);
  const uint32_t w[4] = {q.a.x, q.a.y, q.a.z, q.a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    Q4Word d = dequant_q4_word(w[i]);
    acc = fma2(d.p0, xr[4 * i + 0], acc);
    acc = fma2(d.p1, xr[4 * i + 1], acc);
    acc = fma2(d.p2, xr[4 * i + 2], acc);
    acc = fma2(d.p3, xr[4 * i + 3], acc);
  }
  return acc.x + acc.y;
}
__device__ __forceinline__ float blk_dot(const Blk<T_Q8_0>& q, const float2 (&xr)[16]) {
  float2 acc = make_float2(0.f, 0.f);
  const uint32_t w[8] = {q.a.x, q.a.y, q.a.z, q.a.w, q.b.x, q.b.y, q.b.z, q.b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Q8Word d = dequant_q8_word(w[i]);
    acc = fma2(d.p0, xr[2 * i + 0], acc);
    acc = fma2(d.p1, xr[2 * i + 1], acc);
  }
  return acc.x + acc.y;
}

// Dequantised block (for the multi-column kernel: dequantise once, reuse for
// every column). wv_dot then multiplies and adds in exactly the order of
// blk_dot (one packed accumulator, elements in order), so a column's block sum
// is bit-identical to the 1-column kernel's.
__device__ __forceinline__ void blk_dequant(const Blk<T_Q4_0>& q, float2 (&wv)[16]) {
  const uint32_t w[4] = {q.a.x, q.a.y, q.a.z, q.a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    Q4Word d = dequant_q4_word(w[i]);
    wv[4 * i + 0] = d.p0; wv[4 * i + 1] = d.p1; wv[4 * i + 2] = d.p2; wv[4 * i + 3] = d.p3;
  }
}
__device__ __forceinline__ void blk_dequant(const Blk<T_Q8_0>& q, float2 (&wv)[16]) {
  const uint32_t w[8] = {q.a.x, q.a.y, q.a.z, q.a.w, q.b.x, q.b.y, q.b.z, q.b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Q8Word d = dequant_q8_word(w[i]);
    wv[2 * i + 0] = d.p0; wv[2 * i + 1] = d.p1;
  }
}
__device__ __forceinline__ float wv_dot(const float2 (&wv)[16], const float2 (&xr)[16]) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 16; ++i) acc = fma2(wv[i], xr[i], acc);
  return acc.x + acc.y;
}

// Staged x layout of one column: 8 planes of `plane` float4 each; float4 j of
// block bi (floats 4j..4j+3 of the block's 32) sits at plane j, slot bi. Lanes
// that read consecutive blocks therefore read consecutive 16-byte slots, which
// keeps shared-memory accesses free of bank conflicts.
__device__ __forceinline__ void load_x16(const float* col, int plane, int bi, float2 (&xr)[16]) {
  const float4* p4 = reinterpret_cast<const float4*>(col) + bi;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float4 v = p4[i * plane];
    xr[2 * i] = make_float2(v.x, v.y);
    xr[2 * i + 1] = make_float2(v.z, v.w);
  }
}

// Stage x[c][kb0*32 .. kb1*32) of the selected columns into shared memory as
// f32 in the consumption order of QT. One thread per 32-element block: its four
// 16-byte loads are issued before any use, so a CTA pays about one global-load
// latency per pass instead of one per element.
struct XBlk { uint4 v0, v1, v2, v3; };  // one 32-element f16 block of x

__device__ __forceinline__ XBlk load_xblk(const __half* src) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  return XBlk{s4[0], s4[1], s4[2], s4[3]};
}

// Write a loaded x block into the staged layout (see stage_block).
__device__ __forceinline__ void stage_xblk(int qt, float* col, int plane, int bi, const XBlk& xb) {
  const uint4 v0 = xb.v0, v1 = xb.v1, v2 = xb.v2, v3 = xb.v3;
  __align__(16) __half h[32];
  *reinterpret_cast<uint4*>(&h[0]) = v0;
  *reinterpret_cast<uint4*>(&h[8]) = v1;
  *reinterpret_cast<uint4*>(&h[16]) = v2;
  *reinterpret_cast<uint4*>(&h[24]) = v3;
  float o[32];
#pragma unroll
  for (int s = 0; s < 32; ++s)
    o[s] = qt == T_Q4_0 ? __half2float(h[q4_xorder_elem(s)]) * q4_xorder_scale(s)
                        : __half2float(h[q8_xorder_elem(s)]);
  float4* d4 = reinterpret_cast<float4*>(col) + bi;
#pragma unroll
  for (int i = 0; i < 8; ++i) d4[i * plane] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
}

__device__ __forceinline__ void stage_block(int qt, float* col, int plane, int bi,
                                            const __half* src) {
  stage_xblk(qt, col, plane, bi, load_xblk(src));
}

// Column c occupies xs[c * xstride ...] (xstride = 32 * plane floats).
template <int QT, int NC>
__device__ __forceinline__ void stage_x(float* xs, int xstride, const __half* x, int k,
                                        const int (&cols)[NC], int kb0, int kb1) {
  const int nbk = kb1 - kb0;
  const int plane = xstride / QK;
  for (int it = threadIdx.x; it < NC * nbk; it += blockDim.x) {
    const int c = it / nbk, b = it % nbk;
    stage_block(QT, xs + c * xstride, plane, b, x + (size_t)cols[c] * k + (size_t)(kb0 + b) * QK);
  }
}

// One warp: 1-column dot of RW rows (and of a second matrix when DUAL) over
// the blocks [kb0, kb1) of the staged x chunk; lane l takes blocks kb0+l,
// kb0+l+32, ... Accumulates per-row totals (block scales applied per block).
template <int QT, int RW, bool DUAL>
__device__ __forceinline__ void cc_rowdot_1col(const uint8_t* __restrict__ qa,
                                               const uint16_t* __restrict__ sa,
                                               const uint8_t* __restrict__ qb,
                                               const uint16_t* __restrict__ sb,
                                               size_t rowbytes, int nb, const int (&rowidx)[RW],
                                               const float* xs, int plane, int kb0, int kb1,
                                               int lane, float (&ta)[RW], float (&tb)[RW]) {
  constexpr int QB = QTraits<QT>::QB;
  // two blocks per lane in flight: a 2048-wide row is one round trip, not two
#pragma unroll 2
  for (int b = kb0 + lane; b < kb1; b += 32) {
    Blk<QT> bqa[RW], bqb[RW];
    uint16_t bsa[RW], bsb[RW];
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      bqa[r].load(qa + (size_t)rowidx[r] * rowbytes + (size_t)b * QB);
      bsa[r] = ld_u16(sa + (size_t)rowidx[r] * nb + b);
      if (DUAL) {
        bqb[r].load(qb + (size_t)rowidx[r] * rowbytes + (size_t)b * QB);
        bsb[r] = ld_u16(sb + (size_t)rowidx[r] * nb + b);
      }
    }
    float2 xr[16];
    load_x16(xs, plane, b - kb0, xr);
#pragma unroll
    for (int r = 0; r < RW; ++r) {
      ta[r] = fmaf(h2f(bsa[r]), blk_dot(bqa[r], xr), ta[r]);
      if (DUAL) tb[r] = fmaf(h2f(bsb[r]), blk_dot(bqb[r], xr), tb[r]);
    }
  }
}

}  // namespace qg
