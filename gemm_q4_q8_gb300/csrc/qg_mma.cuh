// qg_mma.cuh -- device helpers of the mma.sync paths (the tensor-core GEMM and
// the tensor-core MoE down projection): TMA tile loads, shared-memory loads,
// m16n8k16 f16 mma with f32 accumulation, and the exact f16 dequantisation of
// the stored Q4_0 / Q8_0 words into A fragments.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "qg_common.cuh"

namespace qg {

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
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
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                       uint32_t& d) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t& a, uint32_t& b) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
}
// Two f16 scales packed in a word, as f32 (the conversion reads each half in
// place, no extraction).
__device__ __forceinline__ float lo_f32(uint32_t w) {
  return __low2float(*reinterpret_cast<const __half2*>(&w));
}
__device__ __forceinline__ float hi_f32(uint32_t w) {
  return __high2float(*reinterpret_cast<const __half2*>(&w));
}
// D = A * B (+ C), f16 inputs, f32 accumulate.
// The mma are pure register operations (not volatile): the compiler may
// interleave them with the dequantisation of the next block.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f), "f"(0.f),
        "f"(0.f), "f"(0.f));
}
__device__ __forceinline__ void mma16816_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm(
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
// Q4_0: word w = stored bytes 4t..4t+3 of one row of a block, i.e. GGUF bytes
// 2t, 2t+8, 2t+1, 2t+9 (GGUF byte j holds element j low, j+16 high). 0x6400 is
// f16 1024 (one mantissa step = 1). Results, each equal to (q - 8) exactly:
//   e0 = (el 2t, 2t+1), e2 = (2t+8, 2t+9), e1 = (2t+16, 2t+17), e3 = (2t+24, 2t+25)
// M: the pattern 0x64006400 (f16 1024 twice), held in a register.
__device__ __forceinline__ void dq4_f16(uint32_t w, uint32_t M, uint32_t& e0, uint32_t& e1,
                                        uint32_t& e2, uint32_t& e3) {
  const uint32_t w8 = w >> 8;
  const uint32_t k1032 = 0x64086408u;  // 1032 = 1024 + 8
  const uint32_t k16th = 0x2C002C00u;  // 1/16
  const uint32_t km72 = 0xD480D480u;   // -72
  e0 = hsub2_u(and_or<0x000F000Fu>(w, M), k1032);
  e2 = hsub2_u(and_or<0x000F000Fu>(w8, M), k1032);
  e1 = hfma2_u(and_or<0x00F000F0u>(w, M), k16th, km72);   // (1024 + 16 q) / 16 - 72 = q - 8
  e3 = hfma2_u(and_or<0x00F000F0u>(w8, M), k16th, km72);
}
// Q8_0: word w = stored bytes 4t..4t+3 of a 16-element half block, i.e. its
// elements 2t, 2t+8, 2t+1, 2t+9:  p0 = (el 2t, 2t+1), p1 = (2t+8, 2t+9), exactly q.
__device__ __forceinline__ void dq8_f16(uint32_t w, uint32_t& p0, uint32_t& p1) {
  const uint32_t u = w ^ 0x80808080u;          // q + 128
  const uint32_t k1152 = 0x64806480u;          // 1024 + 128
  p0 = hsub2_u(__byte_perm(u, 0x64646464u, 0x4240), k1152);
  p1 = hsub2_u(__byte_perm(u, 0x64646464u, 0x4341), k1152);
}

}  // namespace qg
