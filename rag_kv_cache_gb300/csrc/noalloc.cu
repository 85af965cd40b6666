// HKVD selection without any allocation: cb_hkvd_select_noalloc.
//
// Some callers cannot allocate device memory at the point where they select
// tokens: a serving engine that hands all free HBM to its own KV-cache pool
// at start-up (a cudaMalloc on the request path would fail, or fragment the
// pool), or a latency-critical request path that must not pay the implicit
// device synchronisation of cudaMalloc/cudaFree. They also cannot create a
// cb_plan, which allocates. This entry point runs the same deviation and top-k
// kernels as cb_kv_deviation + cb_hkvd_topk, but keeps the per-candidate
// deviations (the only intermediate) in a fixed array compiled into the
// library instead of a buffer someone has to allocate.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <mutex>

#include "../../include/cacheblend.h"
#include "common.cuh"
#include "kernels.h"

namespace cb {
cb_status set_last_error(cb_status s, const char* msg);  // cb_api.cu: the text cb_last_error_string returns
}

namespace {

// Deviation of each candidate between the two kernels. 65536 floats = 256 KiB,
// held by every GPU that loads the library until the process exits.
static __device__ __align__(256) float g_select_scratch[CB_NOALLOC_MAX_CANDIDATES];

// The array's device address, per device, together with the ID of the CUDA context it was
// looked up in. A context that is torn down and created again (cudaDeviceReset, or a primary
// context released by its last user) reloads the library's module, and the array may then sit
// at another address: a call that finds a different context ID on its device looks it up again.
struct ScratchAddr {
  unsigned long long ctx_id;
  float* ptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mutex;
ScratchAddr g_scratch[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

cb_status noalloc_fail(cb_status s, const char* msg) { return cb::set_last_error(s, msg); }

template <typename Fn>
bool driver_entry(const char* name, int version, Fn* out) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return false;
  *out = reinterpret_cast<Fn>(p);
  return true;
}

// ID of the context current on this thread; 0 if none is current yet.
cudaError_t current_context_id(unsigned long long* id) {
  *id = 0;
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) return cudaSuccess;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array in the current device's current context. The array's name
// in host code is only a host-side stand-in, so the address is asked for with the device current
// (once per device and context) and remembered.
cudaError_t scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_ctx_current == nullptr &&
      !(driver_entry("cuCtxGetCurrent", 4000, &g_ctx_current) && driver_entry("cuCtxGetId", 12000, &g_ctx_id)))
    return cudaErrorNotSupported;
  unsigned long long id = 0;
  e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  if (id == 0 || g_scratch[dev].ptr == nullptr || g_scratch[dev].ctx_id != id) {
    // The lookup also makes the device's primary context current if none was yet.
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_select_scratch);
    if (e != cudaSuccess) return e;
    e = current_context_id(&id);
    if (e != cudaSuccess) return e;
    g_scratch[dev] = ScratchAddr{id, static_cast<float*>(p)};
  }
  *out = g_scratch[dev].ptr;
  return cudaSuccess;
}

cb_status select_noalloc(const void* v_new, const void* v_old, const int32_t* cand, int32_t m, int32_t k,
                         int32_t n_rows, int32_t hkv, int32_t head_dim, int32_t* sel_tok, int32_t* sel_row,
                         void* stream) {
  if (m < 0 || k < 0 || k > m) return noalloc_fail(CB_ERR_INVALID_ARG, "need 0 <= k <= m");
  if (m > CB_NOALLOC_MAX_CANDIDATES)
    return noalloc_fail(CB_ERR_INVALID_ARG,
                        "m exceeds CB_NOALLOC_MAX_CANDIDATES (65536): use cb_kv_deviation + cb_hkvd_topk");
  if (hkv <= 0 || head_dim <= 0 || (hkv * head_dim) % 8 != 0 || hkv * head_dim > 2048)
    return noalloc_fail(CB_ERR_INVALID_ARG, "hkv * head_dim must be a positive multiple of 8, at most 2048");
  if (n_rows < 0 || (cand == nullptr && m > n_rows)) return noalloc_fail(CB_ERR_INVALID_ARG, "m > n_rows without cand");
  if (k == 0) return CB_OK;
  if (v_new == nullptr || v_old == nullptr || sel_tok == nullptr || sel_row == nullptr)
    return noalloc_fail(CB_ERR_INVALID_ARG, "NULL tensor pointer");
  if ((reinterpret_cast<uintptr_t>(v_new) | reinterpret_cast<uintptr_t>(v_old)) & 15u)
    return noalloc_fail(CB_ERR_INVALID_ARG, "v_new / v_old must be 16-byte aligned");
  float* scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (e == cudaSuccess) e = cb::launch_kv_deviation(nullptr, nullptr, v_new, v_old, cand, m, n_rows, hkv, head_dim, 1, 0,
                                                       cb::RopeTable{nullptr, 0}, scratch, nullptr, s);
  if (e == cudaSuccess) e = cb::launch_hkvd_topk(scratch, cand, m, k, sel_tok, sel_row, nullptr, s);
  if (e != cudaSuccess) return noalloc_fail(CB_ERR_CUDA, cudaGetErrorString(e));
  return CB_OK;
}

}  // namespace

extern "C" cb_status cb_hkvd_select_noalloc(const void* v_new, const void* v_old, const int32_t* cand, int32_t m,
                                            int32_t k, int32_t n_rows, int32_t hkv, int32_t head_dim,
                                            int32_t* sel_tok, int32_t* sel_row, void* stream) {
  nvtxRangePushA("cb_hkvd_select_noalloc");  // one NVTX range per entry point, as in cb_api.cu
  const cb_status st = select_noalloc(v_new, v_old, cand, m, k, n_rows, hkv, head_dim, sel_tok, sel_row, stream);
  nvtxRangePop();
  return st;
}
