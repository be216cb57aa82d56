// qg_internal.h -- launchers shared between the translation units of libqgemm.
// Host-side only; every launcher enqueues on the given stream and returns the
// CUDA error of the launch (cudaSuccess when nothing went wrong).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "qgemm.h"

namespace qg {

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Raise `kern`'s dynamic shared-memory limit on the current device to at least
// `smem` (never lowers it), and allow cluster sizes above 8 when asked; cached
// per device, safe from several host threads.
cudaError_t prepare_kernel(const void* kern, size_t smem, bool nonportable_cluster);

// prepare_kernel, then how many CTAs of `threads` threads and `smem` bytes of
// dynamic shared memory stay resident per SM (at least 1); cached per device.
cudaError_t kernel_occupancy(const void* kern, int threads, size_t smem, int* occ);

// Remember the CUDA error behind a QG_ERR_CUDA on this host thread
// (qg_last_cuda_error), and read it back.
void note_cuda_error(cudaError_t e);
cudaError_t last_cuda_error();

// Count one kernel launch (see qg_kernel_launches).
void note_launch(int n = 1);

// Launch classes for programmatic dependent launch. LC_SMEM: the tensor-core
// GEMM, whose CTAs hold most of the SM's shared memory and trigger their
// dependents as soon as they start. LC_L1: every other kernel; they stream
// through L1 (in-flight loads are staged there) and lose up to a third of
// their bandwidth if they start on an SM while an LC_SMEM CTA is resident,
// because a CTA inherits the carve-out of the SM it lands on for its whole
// life. So an LC_L1 kernel that directly follows an LC_SMEM kernel on the
// same stream is launched without the programmatic attribute (it starts when
// that grid completes); every other pair overlaps.
enum LaunchClass { LC_L1 = 0, LC_SMEM = 1 };

// Records `cls` as the class of the latest launch on `s` and returns whether
// this launch may use programmatic stream serialisation.
bool pdl_allowed(cudaStream_t s, LaunchClass cls);

// Launch `kern` on `s` (with programmatic stream serialisation when
// pdl_allowed says so: the kernel may begin while the previous kernel on `s`
// finishes; see pdl_wait in qg_common.cuh), plus a cluster of `cluster_x`
// CTAs along x when cluster_x > 0.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, int cluster_x, LaunchClass cls, Args&&... args) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (pdl_allowed(s, cls)) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster_x > 0) {
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = (unsigned)cluster_x;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  }
  lc.attrs = at;
  lc.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&lc, kern, std::forward<Args>(args)...);
  note_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

// CUDA-core GEMV, 1..8 columns per launch: y = y0 + W x.
cudaError_t cc_gemv(int qt, const void* q, const uint16_t* scl, int rows, int k,
                    const uint16_t* x, int ncols, const float* y0, float* y, cudaStream_t s);

// CUDA-core fused gate/up, 1..8 columns per launch: h = f16(SiLU(Wg x) * (Wu x)).
cudaError_t cc_gate_up_silu(int qt, const void* qg, const uint16_t* sg, const void* qu,
                            const uint16_t* su, int rows, int k, const uint16_t* x,
                            int ncols, uint16_t* h, cudaStream_t s);

// Tensor-core (mma.sync) skinny GEMM, 1..16 columns: y = y0 + W x, or, with
// qu != nullptr, h = f16(SiLU(W x) * (Wu x)). Only for shapes where
// tc_supported() holds (k % 256 == 0 and a shared-memory plan exists).
cudaError_t tc_gemm(int qt, const void* q, const uint16_t* scl, const void* qu,
                    const uint16_t* su, int rows, int k, const uint16_t* x, int ncols,
                    const float* y0, float* y, uint16_t* h, cudaStream_t s);
bool tc_supported(int qt, int ncols, bool dual, int rows, int k);

struct MoeArgs {
  int qt;
  const void *qg, *qu, *qd;
  const uint16_t *sg, *su, *sd;
  int n_expert, ffn, hidden;
  const int32_t* ids;
  const float* rw;
  int topk;
  bool has_shared;
  const void *sqg, *squ, *sqd;
  const uint16_t *ssg, *ssu, *ssd;
  const uint16_t* x;
  int ncols;
  const float* y0;
  float* y;
  void* ws;
  int32_t* err_flag;
  int32_t* uniq_out;
};
size_t moe_ws_bytes(int n_expert, int ffn, int hidden, int ncols, int topk);
bool moe_shape_supported(int ffn, int hidden, int ncols, int topk);
// Type and shape checks of the MoE layer: QG_OK, QG_ERR_TYPE or QG_ERR_SHAPE.
qg_status moe_check_shape(int t, int n_expert, int ffn, int hidden, int ncols, int topk);
cudaError_t moe_forward(const MoeArgs& a, cudaStream_t s);
// The MoE kernels' device error word (QG_DEV_ERR_WAIT), read and cleared.
cudaError_t moe_device_error(int32_t* bits);

cudaError_t repack_launch(int qt, const void* gguf, int rows, int k, void* q_out,
                          uint16_t* scl_out, cudaStream_t s);

// Greedy argmax / top-k over f32 columns [ncols][n] (qg_sample.cu).
cudaError_t argmax_launch(const float* x, int n, int ncols, int32_t* idx, float* val,
                          cudaStream_t s);
cudaError_t topk_launch(const float* x, int n, int ncols, int k, int32_t* idx, float* val,
                        cudaStream_t s);

// MoE router: logits, top-k ids and softmax weights (qg_router.cu).
bool router_shape_ok(int E, int hidden, int ncols, int topk);
cudaError_t router_launch(const float* w, const uint16_t* x, int E, int hidden, int ncols,
                          int topk, float* logits, int32_t* ids, float* rw, cudaStream_t s);

}  // namespace qg
