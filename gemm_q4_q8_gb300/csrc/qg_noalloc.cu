// qg_noalloc.cu -- qmoe_experts_noalloc: the MoE layer for callers that cannot
// allocate device memory.
//
// qmoe_experts needs a device workspace that the caller allocates. Some callers
// cannot do that: a plugin hosted by a framework that owns every byte of device
// memory and forbids third-party allocations, code that runs under a fixed
// memory budget that has no room left at the moment of the call, or a
// latency-critical loop where cudaMalloc (which may synchronise the device) is
// not acceptable. For them this entry point uses a workspace that lives in the
// library itself: a file-scope __device__ array of QG_MOE_NOALLOC_WS_BYTES,
// which every GPU that loads this library holds until the process exits. Its
// size is the largest workspace any shape the MoE layer accepts can need, so
// every accepted shape fits; a shape beyond it would get QG_ERR_WORKSPACE.
//
// The array name is only a host-side stand-in in host code, not a device
// address. The first call on each device (with that device current) asks the
// runtime for the array's device address with cudaGetSymbolAddress, checks the
// result, and keeps the address for that device; later calls reuse it. That
// first call should therefore come before any stream capture. The kept address
// belongs to the device's primary context: after cudaDeviceReset (or anything
// else that destroys that context) it is stale, so this entry point must not
// be used across a device reset.
//
// Every call shares the one array and it keeps the previous call's contents.
// Nothing in it needs to start at zero: within a call, every workspace entry
// the MoE kernels read was written earlier in the same call. Calls whose work
// overlaps on the GPU (different streams, or several host threads) race on the
// array; issue them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "qg_internal.h"
#include "qgemm.h"

namespace {

constexpr size_t kNoallocWsBytes = QG_MOE_NOALLOC_WS_BYTES;

static __device__ __align__(256) unsigned char g_moe_noalloc_ws[kNoallocWsBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (set up on first use).
qg_status ws_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    qg::note_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return QG_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ws_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_noalloc_ws);
    if (e != cudaSuccess || p == nullptr) {
      qg::note_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return QG_ERR_CUDA;
    }
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return QG_OK;
}

}  // namespace

extern "C" qg_status qmoe_experts_noalloc(qg_type t, const void* qg, const uint16_t* sg,
                                          const void* qu, const uint16_t* su, const void* qd,
                                          const uint16_t* sd, int n_expert, int ffn, int hidden,
                                          const int32_t* ids, const float* rw, int topk,
                                          const qg_expert* shared, const uint16_t* x, int ncols,
                                          const float* y0, float* y, int32_t* err_flag,
                                          int32_t* uniq_ids_out, cudaStream_t stream) {
  // The same type and shape checks as qmoe_experts, so both return the same status.
  qg_status st = qg::moe_check_shape((int)t, n_expert, ffn, hidden, ncols, topk);
  if (st != QG_OK) return st;
  if (qmoe_workspace_bytes(n_expert, ffn, hidden, ncols, topk) > kNoallocWsBytes)
    return QG_ERR_WORKSPACE;  // beyond the built-in maximum (no accepted shape is)
  void* ws = nullptr;
  if ((st = ws_address(&ws)) != QG_OK) return st;
  return qmoe_experts(t, qg, sg, qu, su, qd, sd, n_expert, ffn, hidden, ids, rw, topk, shared, x,
                      ncols, y0, y, ws, kNoallocWsBytes, err_flag, uniq_ids_out, stream);
}
