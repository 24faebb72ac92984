// Pose top-k for callers that cannot allocate device memory.
//
// la_select_context keeps the retrieval kernel's scratch in the cache pool.
// Callers that must not allocate (a host that forbids allocation once it is
// serving, a real-time path where an allocation's implicit synchronisation
// would stall the stream) get this entry point instead: it runs the same
// kernel, with its scratch in one file-scope device array of fixed size.
//
// Scratch layout (one array, 256-byte aligned):
//   [0, 64)            DevError  (error word of the kernel)
//   [64, 256)          DevTopk   (CTA completion counter + ranked results)
//   [256, 256 + 4*N)   per-candidate scores, N = LA_NOALLOC_MAX_ROWS
// The header must start at zero on every call (the completion counter and
// the error word); the ranked ids start at -1, so ranks past the number of
// candidates read -1 rather than a stale or zero id; the scores are written
// before they are read.
#include <cstddef>
#include <mutex>

#include "la_internal.h"

using namespace la;

namespace {

constexpr size_t kErrOff = 0;
constexpr size_t kTopkOff = 64;
constexpr size_t kHeaderBytes = 256;
constexpr size_t kScratchBytes = kHeaderBytes + sizeof(float) * (size_t)LA_NOALLOC_MAX_ROWS;
static_assert(sizeof(DevError) <= kTopkOff - kErrOff, "error word does not fit the header");
static_assert(kTopkOff + sizeof(DevTopk) <= kHeaderBytes, "top-k state does not fit the header");

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) unsigned char g_pose_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
char* g_scratch_addr[kMaxDevices] = {};

// Device address of g_pose_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and kept.
cudaError_t scratch_address(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pose_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<char*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" la_status la_pose_topk_noalloc(float* table, float* inv_norm, int max_rows,
                                          const float* query_kp, int pose_row, int c0, int c1,
                                          int k, int32_t* ids_out, float* scores_out,
                                          int32_t* n_out, int32_t* status_out, void* stream) {
  if (!table || !inv_norm || !query_kp || !ids_out || !scores_out || !n_out || !status_out)
    return LA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(table) & 15) return LA_ERR_INVALID_ARG;
  if (max_rows < 1 || pose_row < -1 || pose_row >= max_rows) return LA_ERR_INVALID_ARG;
  if (c0 < 0 || c1 < c0 || c1 > max_rows) return LA_ERR_INVALID_ARG;
  // The query's row is written by one CTA while every CTA may be scoring the
  // candidates, so it must not be one of them.
  if (pose_row >= c0 && pose_row < c1) return LA_ERR_INVALID_ARG;
  if (c1 > LA_NOALLOC_MAX_ROWS) return LA_ERR_INVALID_ARG;   // beyond the fixed scratch
  if (k < 0 || k > LA_MAX_TOPK) return LA_ERR_INVALID_ARG;
  for (int i = 0; i < 34; ++i)
    if (!(query_kp[i] == query_kp[i]) || query_kp[i] > 3.0e38f || query_kp[i] < -3.0e38f)
      return LA_ERR_INVALID_ARG;

  char* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return LA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(base, 0, kHeaderBytes, s) != cudaSuccess ||
      cudaMemsetAsync(base + kTopkOff + offsetof(DevTopk, ids), 0xFF,
                      sizeof(int32_t) * (LA_MAX_TOPK + 1), s) != cudaSuccess)
    return LA_ERR_CUDA;

  RetrievalArgs a{};
  for (int i = 0; i < 34; ++i) a.kp[i] = query_kp[i];
  a.pose_row = pose_row;
  a.c0 = c0;
  a.c1 = c1;
  a.k = k;
  a.max_history = max_rows;
  a.table = table;
  a.inv_norm = inv_norm;
  a.scores = reinterpret_cast<float*>(base + kHeaderBytes);
  a.topk = reinterpret_cast<DevTopk*>(base + kTopkOff);
  a.err = reinterpret_cast<DevError*>(base + kErrOff);
  if (launch_retrieval(a, s) != cudaSuccess) return LA_ERR_CUDA;

  // Results: device-to-device copies out of the scratch's top-k state.
  const char* topk = base + kTopkOff;
  const size_t n_rank = (size_t)k + 1;
  if (cudaMemcpyAsync(ids_out, topk + offsetof(DevTopk, ids), sizeof(int32_t) * n_rank,
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(scores_out, topk + offsetof(DevTopk, scores), sizeof(float) * n_rank,
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(n_out, topk + offsetof(DevTopk, n), sizeof(int32_t),
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(status_out, base + kErrOff + offsetof(DevError, code), sizeof(int32_t),
                      cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return LA_ERR_CUDA;
  return LA_OK;
}
