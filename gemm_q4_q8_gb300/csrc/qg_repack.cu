// qg_repack.cu -- load-time repack of GGUF interleaved blocks into the quant
// and scale arrays the kernels stream ("Architecture", pooled.run, section
// "Memory and caching": matrices are repacked on the way into separate nibble
// and scale arrays so the kernels read them in contiguous stripes).
//
// One thread per block: the block (2 + QB bytes, 2-byte aligned) is read as
// 16-bit words; in each 16-byte group of quants the two 8-byte halves are
// interleaved byte by byte (stored byte 2m + h = GGUF byte m + 8h), and the
// group is written as one 16-byte store.
#include <cuda_runtime.h>

#include "qg_common.cuh"
#include "qg_internal.h"

namespace qg {

template <int QT>
__global__ void repack_kernel(const uint16_t* __restrict__ gguf, size_t nblocks,
                              uint4* __restrict__ q_out, uint16_t* __restrict__ scl_out) {
  constexpr int QB = QTraits<QT>::QB;
  constexpr int W = (2 + QB) / 2;  // 16-bit words per block
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
       i += (size_t)gridDim.x * blockDim.x) {
    const uint16_t* src = gguf + i * W;
    scl_out[i] = src[0];
    uint32_t w[QB / 4];
#pragma unroll
    for (int j = 0; j < QB / 4; ++j) w[j] = (uint32_t)src[1 + 2 * j] | ((uint32_t)src[2 + 2 * j] << 16);
#pragma unroll
    for (int j = 0; j < QB / 16; ++j) {
      // GGUF bytes 0-7 of the group are lo = (w0, w1), bytes 8-15 hi = (w2, w3)
      const uint32_t l0 = w[4 * j], l1 = w[4 * j + 1], h0 = w[4 * j + 2], h1 = w[4 * j + 3];
      q_out[i * (QB / 16) + j] =
          make_uint4(__byte_perm(l0, h0, 0x5140), __byte_perm(l0, h0, 0x7362),
                     __byte_perm(l1, h1, 0x5140), __byte_perm(l1, h1, 0x7362));
    }
  }
}

cudaError_t repack_launch(int qt, const void* gguf, int rows, int k, void* q_out,
                          uint16_t* scl_out, cudaStream_t s) {
  const size_t nblocks = (size_t)rows * (k / QK);
  if (nblocks == 0) return cudaSuccess;
  size_t grid = (nblocks + 255) / 256;
  const size_t maxg = (size_t)device_sm_count() * 8;
  if (grid > maxg) grid = maxg;
  if (qt == T_Q4_0)
    repack_kernel<T_Q4_0><<<(unsigned)grid, 256, 0, s>>>((const uint16_t*)gguf, nblocks, (uint4*)q_out, scl_out);
  else
    repack_kernel<T_Q8_0><<<(unsigned)grid, 256, 0, s>>>((const uint16_t*)gguf, nblocks, (uint4*)q_out, scl_out);
  note_launch();
  return cudaGetLastError();
}

}  // namespace qg
