// cp_attn_partial_kv_noalloc: the partial-KV decomposition with library-owned
// scratch, for callers that must not allocate device memory themselves.
//
// Some callers cannot call cudaMalloc: a serving engine or framework whose
// allocator owns all device memory and forbids allocations outside its plan,
// a deployment with a fixed device-memory budget decided at start-up, or a
// hot path that cannot take the implicit device synchronisation of
// cudaMalloc / cudaFree.  This entry point takes no workspace: the scratch it
// needs is a file-scope __device__ array of CPATTN_NOALLOC_SCRATCH_BYTES that
// every GPU loading this library holds until the process exits.
//
// The host code cannot use the array's name as a device address (in host code
// it is only a stand-in symbol), so the first call in each CUDA context looks
// its address up with cudaGetSymbolAddress while that context's device is
// current, checks the result and caches it together with the context's unique
// id; later calls in the same context reuse the address.  A new context on the
// same device (after cudaDeviceReset, or a caller that switches to a context
// of its own) has a new id, so its first call looks the address up again
// instead of using a stale one.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/cpattn.h"
#include "trace.h"

namespace {

static __device__ __align__(256) unsigned char g_pkv_scratch[CPATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
struct ScratchEntry {
  unsigned long long ctx_id;  // unique id of the context the address belongs to
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Driver entry points for the current context and its id (resolved once
// through the runtime, so the library needs no link against libcuda).
struct CtxApi {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxApi& ctx_api() {
  static CtxApi api;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      api.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      api.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return api;
}

// Unique id of the context current on this thread.  When no context is
// current yet, the device's primary context is made current first, as any
// runtime call would do.
int current_context_id(int dev, unsigned long long* id) {
  const CtxApi& api = ctx_api();
  if (!api.get_current || !api.get_id) return CPATTN_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (api.get_current(&ctx) != CUDA_SUCCESS) return CPATTN_ERR_CUDA;
  if (!ctx) {
    if (cudaSetDevice(dev) != cudaSuccess || api.get_current(&ctx) != CUDA_SUCCESS || !ctx)
      return CPATTN_ERR_CUDA;
  }
  return api.get_id(ctx, id) == CUDA_SUCCESS ? CPATTN_OK : CPATTN_ERR_CUDA;
}

// Device address of g_pkv_scratch in the current context (looked up once per
// context).
int scratch_in_current_context(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CPATTN_ERR_CUDA;
  unsigned long long id = 0;
  const int rc = current_context_id(dev, &id);
  if (rc != CPATTN_OK) return rc;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  ScratchEntry& e = g_scratch[dev];
  if (!e.ptr || e.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || !p) return CPATTN_ERR_CUDA;
    e.ptr = p;
    e.ctx_id = id;
  }
  *out = e.ptr;
  return CPATTN_OK;
}

}  // namespace

extern "C" int cp_attn_partial_kv_noalloc(
    const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev, int num_tiles,
    const void* q, int num_q_rows, const void* k, int64_t k_row_stride, int64_t k_head_stride,
    const void* v, int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv,
    int d, int dv, float scale, int kv_block, int max_blocks, int max_seg_rows,
    const int32_t* dst_rows,
    void* o_out, int o_is_fp32, float* lse_out, int num_out_rows, int64_t workspace_bytes_needed,
    int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_partial_kv_noalloc");
  if (workspace_bytes_needed < 0) return CPATTN_ERR_INVALID_ARG;
  if (workspace_bytes_needed > (int64_t)CPATTN_NOALLOC_SCRATCH_BYTES) return CPATTN_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int rc = scratch_in_current_context(&scratch);
  if (rc != CPATTN_OK) return rc;
  // The same three launches as cp_attn_partial_kv, on the static scratch.
  // Nothing in the scratch must start at zero: the layout kernel rewrites
  // the slot table and every partial the merge reads is written earlier in
  // the same call.  The layout kernel also checks the real need against the
  // array's size on the device, so a caller figure that is too small gives
  // the device-status error of cp_attn_partial_kv rather than a write past
  // the array.
  return cp_attn_partial_kv(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k,
                            k_row_stride, k_head_stride, v, v_row_stride, v_head_stride,
                            num_kv_rows, Hq, Hkv, d, dv, scale, kv_block, max_blocks,
                            max_seg_rows, dst_rows,
                            o_out, o_is_fp32, lse_out, num_out_rows, scratch,
                            (int64_t)CPATTN_NOALLOC_SCRATCH_BYTES, status_dev, stream);
}
