// qg_common.cuh -- device helpers shared by the libqgemm kernels (sm_103a).
//
// Dequantisation here is exact: every Q4_0 / Q8_0 weight is an integer times
// its block scale, and the integer is formed exactly in f32 with the
// exponent-OR construction (a published bit trick: OR a small integer into the
// mantissa of a float whose exponent makes one mantissa step worth 1, then
// subtract the same float without the integer). No partial sum is held in f16.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace qg {

constexpr int QK = 32;            // weights per block
constexpr int T_Q4_0 = 2;         // GGUF type ids
constexpr int T_Q8_0 = 8;

template <int QT> struct QTraits;
template <> struct QTraits<T_Q4_0> { static constexpr int QB = 16; };  // quant bytes / block
template <> struct QTraits<T_Q8_0> { static constexpr int QB = 32; };

// 2^23 as an f32 bit pattern: one mantissa step of this float is exactly 1.
constexpr uint32_t MAGIC_2P23 = 0x4B000000u;
constexpr float F_2P23 = 8388608.0f;

// The same pattern in constant memory. Read from there, the pattern reaches the
// dequantisers as a register that the compiler cannot fold into an immediate,
// so each (w & mask) | pattern below stays one three-input logic instruction
// (a logic op takes one immediate at most).
static __constant__ uint32_t c_or_f32 = 0x4B000000u;

// (a & MASK) | orv as one lop3 (truth table 0xEA = (A & B) | C).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t orv) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(orv));
  return d;
}

// ---------------------------------------------------------------- loads
// Weights are read once per call: read-only path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint16_t ld_u16(const uint16_t* p) {
  uint16_t v;
  asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// ---------------------------------------------------------- packed f32x2
// sm_100-family packed single-precision ops: two independent f32 lanes per op.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 A, B, C, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\tmov.b64 C, {%6, %7};\n\t"
      "fma.rn.f32x2 D, A, B, C;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 A, B, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "sub.rn.f32x2 D, A, B;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 A, B, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %5};\n\t"
      "mul.rn.f32x2 D, A, B;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// ------------------------------------------------ exact f32 dequantisation
// Q4_0 word (4 bytes of a block = 8 nibbles). With w16 = w >> 16, the nibble at
// bit 4p (p = 0..3) of w or w16 becomes 2^23 + 16^p * q exactly; subtracting
// 2^23 + 16^p * 8 leaves 16^p * (q - 8) exactly. The matching x values are
// pre-scaled by 16^-p (exact in f32), so products are exact before rounding.
//
// Element order of the 8 results (byte b of the word holds elements b (low)
// and b + 16 (high) of its 4-byte group, relative to the word's first byte j0):
//   p0: (j0+0, j0+16)  p1: (j0+1, j0+17)  p2: (j0+2, j0+18)  p3: (j0+3, j0+19)
// each pair being (low nibble * 1, high nibble * 16) for the low byte of a half
// word, (low * 256, high * 4096) for its high byte.
struct Q4Word { float2 p0, p1, p2, p3; };

__device__ __forceinline__ Q4Word dequant_q4_word(uint32_t w) {
  const uint32_t w16 = w >> 16;
  const float2 off_lo = make_float2(F_2P23 + 8.f, F_2P23 + 128.f);
  const float2 off_hi = make_float2(F_2P23 + 2048.f, F_2P23 + 32768.f);
  Q4Word r;
  const uint32_t m = c_or_f32;
  r.p0 = sub2(make_float2(u2f(and_or<0x000Fu>(w, m)), u2f(and_or<0x00F0u>(w, m))), off_lo);
  r.p1 = sub2(make_float2(u2f(and_or<0x0F00u>(w, m)), u2f(and_or<0xF000u>(w, m))), off_hi);
  r.p2 = sub2(make_float2(u2f(and_or<0x000Fu>(w16, m)), u2f(and_or<0x00F0u>(w16, m))), off_lo);
  r.p3 = sub2(make_float2(u2f(and_or<0x0F00u>(w16, m)), u2f(and_or<0xF000u>(w16, m))), off_hi);
  return r;
}

// GGUF byte of a 16-byte group held by stored byte sb of that group: the two
// 8-byte halves are interleaved, stored byte 2m + h = GGUF byte m + 8h.
__host__ __device__ __forceinline__ int gguf_byte_of_stored(int sb) { return (sb >> 1) + 8 * (sb & 1); }

// Pre-scaled x layout for one Q4_0 block (32 floats) in consumption order: for
// word i (stored bytes 4i..4i+3, GGUF bytes g0..g3 = 2i, 2i+8, 2i+1, 2i+9), 8
// floats: x[g0]*1, x[g0+16]/16, x[g1]/256, x[g1+16]/4096, x[g2]*1,
// x[g2+16]/16, x[g3]/256, x[g3+16]/4096 (GGUF byte g holds elements g, g+16).
__host__ __device__ __forceinline__ int q4_xorder_elem(int s) {
  const int i = s >> 3, j = s & 7;
  const int byte = gguf_byte_of_stored(4 * i + (j >> 1));
  return (j & 1) ? byte + 16 : byte;
}
// Q8_0 x order: slot s takes the element of stored byte s (word s/4 gives the
// float pairs (byte 0, byte 1) and (byte 2, byte 3)).
__host__ __device__ __forceinline__ int q8_xorder_elem(int s) {
  return (s & ~15) + gguf_byte_of_stored(s & 15);
}
__device__ __forceinline__ float q4_xorder_scale(int s) {
  // j = s & 7: 0 -> 1, 1 -> 1/16, 2 -> 1/256, 3 -> 1/4096, 4 -> 1, ...
  const int j = s & 3;
  return j == 0 ? 1.0f : (j == 1 ? 0.0625f : (j == 2 ? 0.00390625f : 0.000244140625f));
}

// Q8_0 word (4 int8). Bias to unsigned (q + 128), place each byte as the low
// mantissa byte of 2^23, subtract 2^23 + 128: exact q. x is staged in the
// stored byte order (q8_xorder_elem).
struct Q8Word { float2 p0, p1; };

__device__ __forceinline__ Q8Word dequant_q8_word(uint32_t w) {
  const uint32_t u = w ^ 0x80808080u;
  const float2 off = make_float2(F_2P23 + 128.f, F_2P23 + 128.f);
  Q8Word r;
  r.p0 = sub2(make_float2(u2f(__byte_perm(u, MAGIC_2P23, 0x7440)),
                          u2f(__byte_perm(u, MAGIC_2P23, 0x7441))), off);
  r.p1 = sub2(make_float2(u2f(__byte_perm(u, MAGIC_2P23, 0x7442)),
                          u2f(__byte_perm(u, MAGIC_2P23, 0x7443))), off);
  return r;
}

// ------------------------------------------- programmatic dependent launch
// Kernels of this library are launched with programmatic stream
// serialisation: a kernel may start while the previous kernel on the stream is
// finishing. pdl_trigger() lets the next kernel start early (every kernel
// calls it at its start, except the MoE gate/up kernel, which calls it right
// after its wait; the host keeps a CUDA-core kernel from starting early behind
// the tensor-core kernel, see LaunchClass in qg_internal.h); pdl_wait() blocks
// until every earlier kernel on the stream has completed and its writes are
// visible. Each kernel reads only weights (immutable inputs) before pdl_wait()
// and touches activations, residuals, ids and outputs only after it, with one
// exception: the staged MoE down kernel reads the id list and the routing
// weights before its wait. It is launched behind the gate/up kernel, which lets
// it start only once its own wait has returned, so whatever wrote them has
// completed by then. Launched without the attribute, both instructions are
// no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// L2 prefetch hints: a 16-byte aligned range whose size is a multiple of 16
// (bulk), or the cache line holding one address.
__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void l2_prefetch_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// --------------------------------------------------- warp reductions
// Reduce N values (N a power of two, 1..32) over the 32 lanes of a warp so that
// each value's total ends up in some lane; returns the total held by this lane
// and sets `idx` to the value index it belongs to. The reduction tree is fixed.
template <int N>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane, int& idx) {
  idx = 0;
  int n = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool upper = (lane & off) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < h) {
          float send = upper ? v[i] : v[i + h];
          float keep = upper ? v[i + h] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
      }
      if (upper) idx += h;
      n = h;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
    }
  }
  return v[0];
}

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

}  // namespace qg
