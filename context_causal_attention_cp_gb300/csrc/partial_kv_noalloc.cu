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
// it is only a stand-in symbol), so the first call on each device looks its
// address up with cudaGetSymbolAddress while that device is current, checks
// the result and caches it; later calls on that device reuse the address.
#include <cstdint>
#include <mutex>

#include "../../include/cpattn.h"

namespace {

static __device__ __align__(256) unsigned char g_pkv_scratch[CPATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_pkv_scratch on the current device (set up once).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CPATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_scratch) != cudaSuccess || !p) return CPATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  if (workspace_bytes_needed < 0) return CPATTN_ERR_INVALID_ARG;
  if (workspace_bytes_needed > (int64_t)CPATTN_NOALLOC_SCRATCH_BYTES) return CPATTN_ERR_TOO_LARGE;
  void* scratch = nullptr;
  const int rc = scratch_on_current_device(&scratch);
  if (rc != CPATTN_OK) return rc;
  // The same three launches as cp_attn_partial_kv, on the static scratch.
  // Nothing in the scratch must start at zero: the layout kernel rewrites
  // the slot table and every partial the merge reads is written earlier in
  // the same call.
  return cp_attn_partial_kv(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k,
                            k_row_stride, k_head_stride, v, v_row_stride, v_head_stride,
                            num_kv_rows, Hq, Hkv, d, dv, scale, kv_block, max_blocks,
                            max_seg_rows, dst_rows,
                            o_out, o_is_fp32, lse_out, num_out_rows, scratch,
                            (int64_t)CPATTN_NOALLOC_SCRATCH_BYTES, status_dev, stream);
}
