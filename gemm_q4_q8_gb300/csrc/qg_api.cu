// qg_api.cu -- the C ABI of libqgemm: argument checks on the host, then
// dispatch to the kernels on the caller's stream. Nothing here allocates.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>
#include <utility>

#include "qg_internal.h"
#include "qgemm.h"

namespace qg {

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

// Kernel preparation, cached per device. The dynamic shared-memory limit of a
// kernel is only ever raised (to the largest size any call has needed), so a
// launch on one host thread never finds the limit lowered by another thread
// between its check and its launch.
namespace {
std::mutex g_kmu;
std::map<std::pair<int, const void*>, size_t> g_smem_limit;          // (device, kernel)
std::map<std::tuple<int, const void*, int, size_t>, int> g_occupancy;  // (device, kernel, threads, smem)
}  // namespace

cudaError_t prepare_kernel(const void* kern, size_t smem, bool nonportable_cluster) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_kmu);
  auto it = g_smem_limit.find({dev, kern});
  if (it == g_smem_limit.end()) {
    if (nonportable_cluster &&
        (e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
      return e;
    it = g_smem_limit.emplace(std::make_pair(dev, kern), (size_t)0).first;
  }
  if (smem > it->second) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    it->second = smem;
  }
  return cudaSuccess;
}

cudaError_t kernel_occupancy(const void* kern, int threads, size_t smem, int* occ) {
  cudaError_t e = prepare_kernel(kern, smem, false);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_kmu);
  const auto key = std::make_tuple(dev, kern, threads, smem);
  auto it = g_occupancy.find(key);
  if (it == g_occupancy.end()) {
    int n = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem)) != cudaSuccess)
      return e;
    it = g_occupancy.emplace(key, n < 1 ? 1 : n).first;
  }
  *occ = it->second;
  return cudaSuccess;
}

// The CUDA error behind the latest QG_ERR_CUDA returned on this host thread.
static thread_local cudaError_t t_last_cuda = cudaSuccess;
void note_cuda_error(cudaError_t e) { t_last_cuda = e; }
cudaError_t last_cuda_error() { return t_last_cuda; }

static std::atomic<uint64_t> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

qg_status moe_check_shape(int t, int n_expert, int ffn, int hidden, int ncols, int topk) {
  if (t != QG_Q4_0 && t != QG_Q8_0) return QG_ERR_TYPE;
  if (n_expert < 1 || n_expert > QG_MOE_MAX_EXPERTS || ffn <= 0 || hidden <= 0 || (ffn % 32) ||
      (hidden % 32) || ncols < 1 || ncols > 16 || topk < 1 || topk > 16 ||
      !moe_shape_supported(ffn, hidden, ncols, topk))
    return QG_ERR_SHAPE;
  return QG_OK;
}

bool pdl_allowed(cudaStream_t s, LaunchClass cls) {
  static std::mutex mu;
  static std::unordered_map<cudaStream_t, int> last;  // class of the latest launch per stream
  std::lock_guard<std::mutex> lk(mu);
  auto it = last.find(s);
  const int prev = it == last.end() ? -1 : it->second;
  if (it == last.end()) {
    if (last.size() > 4096) last.clear();  // streams come and go; forget stale handles
    last.emplace(s, (int)cls);
  } else {
    it->second = (int)cls;
  }
  return !(cls == LC_L1 && prev == LC_SMEM);
}

}  // namespace qg

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_type(int t) { return t == QG_Q4_0 || t == QG_Q8_0; }

// Partial overlap of two byte ranges (identical start is allowed by the caller).
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

qg_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return QG_OK;
  qg::note_cuda_error(e);
  return QG_ERR_CUDA;
}

// Common checks of a (rows x k) matrix product with ncols input columns.
qg_status check_matmul(int t, const void* q, const uint16_t* scl, int rows, int k,
                       const uint16_t* x, int ncols, int max_cols, const float* y0,
                       const void* out, size_t out_elem) {
  if (!valid_type(t)) return QG_ERR_TYPE;
  if (rows < 0 || k <= 0 || (k % 32) != 0 || ncols < 1 || ncols > max_cols) return QG_ERR_SHAPE;
  if (rows == 0) return QG_OK;
  if (!q || !scl || !x || !out) return QG_ERR_NULL;
  if (!aligned(q, 16) || !aligned(scl, 16) || !aligned(x, 16) || !aligned(out, out_elem) ||
      (y0 && !aligned(y0, 4)))
    return QG_ERR_ALIGN;
  if (y0 && y0 != out) {
    const size_t n = (size_t)ncols * rows * sizeof(float);
    if (overlaps(y0, n, out, n)) return QG_ERR_ALIAS;
  }
  return QG_OK;
}

// Device readiness (a device must be present and current).
qg_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return from_cuda(e);
  // A host thread's first runtime calls need not bind the device's primary
  // context, and the tensor-core path calls the driver (tensor-map encoding)
  // before its first launch: on a fresh thread that failed with invalid value.
  // Make the context current once per thread and device.
  static thread_local int bound = -1;
  if (bound != dev) {
    if ((e = cudaSetDevice(dev)) != cudaSuccess) return from_cuda(e);
    bound = dev;
  }
  return qg::device_sm_count() > 0 ? QG_OK : from_cuda(cudaErrorNoDevice);
}

qg_status gemv_any(int t, const void* q, const uint16_t* scl, int rows, int k,
                   const uint16_t* x, int ncols, const float* y0, float* y, cudaStream_t s,
                   int max_cols) {
  qg_status st = check_matmul(t, q, scl, rows, k, x, ncols, max_cols, y0, y, 4);
  if (st != QG_OK || rows == 0) return st;
  if ((st = check_device()) != QG_OK) return st;
  if (qg::tc_supported(t, ncols, false, rows, k))
    return from_cuda(qg::tc_gemm(t, q, scl, nullptr, nullptr, rows, k, x, ncols, y0, y, nullptr, s));
  // CUDA-core path, at most 8 columns per launch
  for (int c0 = 0; c0 < ncols; c0 += 8) {
    const int nc = ncols - c0 < 8 ? ncols - c0 : 8;
    cudaError_t e = qg::cc_gemv(t, q, scl, rows, k, x + (size_t)c0 * k, nc,
                                y0 ? y0 + (size_t)c0 * rows : nullptr, y + (size_t)c0 * rows, s);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return QG_OK;
}

}  // namespace

extern "C" {

int qg_last_cuda_error(void) { return (int)qg::last_cuda_error(); }

const char* qg_last_cuda_error_string(void) {
  static thread_local char buf[256];
  const cudaError_t e = qg::last_cuda_error();
  snprintf(buf, sizeof(buf), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return buf;
}

const char* qg_status_str(qg_status s) {
  switch (s) {
    case QG_OK: return "ok";
    case QG_ERR_NULL: return "a required pointer is NULL";
    case QG_ERR_SHAPE: return "invalid shape (k must be a positive multiple of 32; rows >= 0; ncols/topk/n_expert in range)";
    case QG_ERR_ALIGN: return "misaligned pointer (quants, scales, x: 16 bytes; y, y0: 4 bytes; h: 2 bytes)";
    case QG_ERR_TYPE: return "unknown quant type (expected Q4_0=2 or Q8_0=8)";
    case QG_ERR_WORKSPACE: return "workspace missing or smaller than qmoe_workspace_bytes()";
    case QG_ERR_CUDA: return "CUDA runtime error";
    case QG_ERR_ALIAS: return "y0 partially overlaps y";
  }
  return "unknown status";
}

qg_status qgemv_q4_0(const uint8_t* nib, const uint16_t* scl, int rows, int k,
                     const uint16_t* x, int ncols, const float* y0, float* y,
                     cudaStream_t stream) {
  return gemv_any(QG_Q4_0, nib, scl, rows, k, x, ncols, y0, y, stream, 8);
}

qg_status qgemv_q8_0(const int8_t* qs, const uint16_t* scl, int rows, int k,
                     const uint16_t* x, int ncols, const float* y0, float* y,
                     cudaStream_t stream) {
  return gemv_any(QG_Q8_0, qs, scl, rows, k, x, ncols, y0, y, stream, 8);
}

qg_status qgemm_cols(qg_type t, const void* q, const uint16_t* scl, int rows, int k,
                     const uint16_t* x, int ncols, const float* y0, float* y,
                     cudaStream_t stream) {
  return gemv_any((int)t, q, scl, rows, k, x, ncols, y0, y, stream, 16);
}

qg_status qffn_gate_up_silu(qg_type t, const void* qg, const uint16_t* sg, const void* qu,
                            const uint16_t* su, int rows, int k, const uint16_t* x,
                            int ncols, uint16_t* h, cudaStream_t stream) {
  qg_status st = check_matmul((int)t, qg, sg, rows, k, x, ncols, 16, nullptr, h, 2);
  if (st != QG_OK || rows == 0) return st;
  if (!qu || !su) return QG_ERR_NULL;
  if (!aligned(qu, 16) || !aligned(su, 16)) return QG_ERR_ALIGN;
  if ((st = check_device()) != QG_OK) return st;
  if (qg::tc_supported((int)t, ncols, true, rows, k))
    return from_cuda(qg::tc_gemm((int)t, qg, sg, qu, su, rows, k, x, ncols, nullptr, nullptr, h, stream));
  for (int c0 = 0; c0 < ncols; c0 += 8) {
    const int nc = ncols - c0 < 8 ? ncols - c0 : 8;
    cudaError_t e = qg::cc_gate_up_silu((int)t, qg, sg, qu, su, rows, k, x + (size_t)c0 * k, nc,
                                        h + (size_t)c0 * rows, stream);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return QG_OK;
}

size_t qmoe_workspace_bytes(int n_expert, int ffn, int hidden, int ncols, int topk) {
  if (qg::moe_check_shape(QG_Q8_0, n_expert, ffn, hidden, ncols, topk) != QG_OK) return 0;
  return qg::moe_ws_bytes(n_expert, ffn, hidden, ncols, topk);
}

qg_status qmoe_experts(qg_type t, const void* qg, const uint16_t* sg, const void* qu,
                       const uint16_t* su, const void* qd, const uint16_t* sd,
                       int n_expert, int ffn, int hidden, const int32_t* ids,
                       const float* rw, int topk, const qg_expert* shared,
                       const uint16_t* x, int ncols, const float* y0, float* y,
                       void* ws, size_t ws_bytes, int32_t* err_flag,
                       int32_t* uniq_ids_out, cudaStream_t stream) {
  qg_status st0 = qg::moe_check_shape((int)t, n_expert, ffn, hidden, ncols, topk);
  if (st0 != QG_OK) return st0;
  if (!qg || !sg || !qu || !su || !qd || !sd || !ids || !rw || !x || !y) return QG_ERR_NULL;
  const void* p16[] = {qg, sg, qu, su, qd, sd, x};
  for (const void* p : p16)
    if (!aligned(p, 16)) return QG_ERR_ALIGN;
  if (!aligned(ids, 4) || !aligned(rw, 4) || !aligned(y, 4) || (y0 && !aligned(y0, 4)) ||
      (err_flag && !aligned(err_flag, 4)) || (uniq_ids_out && !aligned(uniq_ids_out, 4)))
    return QG_ERR_ALIGN;
  if (shared) {
    if (!shared->qg || !shared->sg || !shared->qu || !shared->su || !shared->qd || !shared->sd)
      return QG_ERR_NULL;
    const void* s16[] = {shared->qg, shared->sg, shared->qu, shared->su, shared->qd, shared->sd};
    for (const void* p : s16)
      if (!aligned(p, 16)) return QG_ERR_ALIGN;
  }
  if (y0 && y0 != y) {
    const size_t n = (size_t)ncols * hidden * sizeof(float);
    if (overlaps(y0, n, y, n)) return QG_ERR_ALIAS;
  }
  const size_t need = qg::moe_ws_bytes(n_expert, ffn, hidden, ncols, topk);
  if (!ws || ws_bytes < need) return QG_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return QG_ERR_ALIGN;
  qg_status st = check_device();
  if (st != QG_OK) return st;
  qg::MoeArgs a{};
  a.qt = (int)t;
  a.qg = qg; a.qu = qu; a.qd = qd; a.sg = sg; a.su = su; a.sd = sd;
  a.n_expert = n_expert; a.ffn = ffn; a.hidden = hidden;
  a.ids = ids; a.rw = rw; a.topk = topk;
  a.has_shared = shared != nullptr;
  if (shared) {
    a.sqg = shared->qg; a.squ = shared->qu; a.sqd = shared->qd;
    a.ssg = shared->sg; a.ssu = shared->su; a.ssd = shared->sd;
  }
  a.x = x; a.ncols = ncols; a.y0 = y0; a.y = y;
  a.ws = ws; a.err_flag = err_flag; a.uniq_out = uniq_ids_out;
  return from_cuda(qg::moe_forward(a, stream));
}

qg_status qmoe_router(const float* w_router, const uint16_t* x, int n_expert, int hidden,
                      int ncols, int topk, float* logits_out, int32_t* ids_out, float* rw_out,
                      cudaStream_t stream) {
  if (!qg::router_shape_ok(n_expert, hidden, ncols, topk)) return QG_ERR_SHAPE;
  if (!w_router || !x || !ids_out || !rw_out) return QG_ERR_NULL;
  if (!aligned(w_router, 16) || !aligned(x, 2) || !aligned(ids_out, 4) || !aligned(rw_out, 4) ||
      (logits_out && !aligned(logits_out, 4)))
    return QG_ERR_ALIGN;
  qg_status st = check_device();
  if (st != QG_OK) return st;
  return from_cuda(qg::router_launch(w_router, x, n_expert, hidden, ncols, topk, logits_out,
                                     ids_out, rw_out, stream));
}

qg_status qargmax_f32(const float* x, int n, int ncols, int32_t* idx_out, float* val_out,
                      cudaStream_t stream) {
  if (n < 1 || ncols < 1 || ncols > 64) return QG_ERR_SHAPE;
  if (!x || !idx_out) return QG_ERR_NULL;
  if (!aligned(x, 4) || !aligned(idx_out, 4) || (val_out && !aligned(val_out, 4))) return QG_ERR_ALIGN;
  qg_status st = check_device();
  if (st != QG_OK) return st;
  return from_cuda(qg::argmax_launch(x, n, ncols, idx_out, val_out, stream));
}

qg_status qtopk_f32(const float* x, int n, int ncols, int k, int32_t* idx_out, float* val_out,
                    cudaStream_t stream) {
  if (n < 1 || ncols < 1 || ncols > 64 || k < 1 || k > 256 || k > n) return QG_ERR_SHAPE;
  if (!x || !idx_out) return QG_ERR_NULL;
  if (!aligned(x, 4) || !aligned(idx_out, 4) || (val_out && !aligned(val_out, 4))) return QG_ERR_ALIGN;
  qg_status st = check_device();
  if (st != QG_OK) return st;
  return from_cuda(qg::topk_launch(x, n, ncols, k, idx_out, val_out, stream));
}

qg_status qrepack(qg_type t, const void* gguf, int rows, int k, void* q_out,
                  uint16_t* scl_out, cudaStream_t stream) {
  if (!valid_type((int)t)) return QG_ERR_TYPE;
  if (rows < 0 || k <= 0 || (k % 32) != 0) return QG_ERR_SHAPE;
  if (rows == 0) return QG_OK;
  if (!gguf || !q_out || !scl_out) return QG_ERR_NULL;
  if (!aligned(gguf, 2) || !aligned(q_out, 16) || !aligned(scl_out, 16)) return QG_ERR_ALIGN;
  qg_status st = check_device();
  if (st != QG_OK) return st;
  return from_cuda(qg::repack_launch((int)t, gguf, rows, k, q_out, scl_out, stream));
}

uint64_t qg_kernel_launches(void) { return qg::g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
