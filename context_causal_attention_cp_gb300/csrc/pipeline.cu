// Host-to-host full-KV CP prefill: the end-to-end path as one call.
//
// For a sequence of same-shaped batches held in host memory, every batch is
// uploaded, sharded and attended by all CP shards against the gathered KV,
// and its output O and LSE come back to host memory in causal token order
// (SGLang docs, "Prefill Context Parallelism", §Zigzag / §Interleave strategy
// and §Attention backend integration; blog "什么是 Context Parallelism", §2.1,
// the restore after the all-gather).
//
// Per batch, on the caller's three streams:
//   upload:   q, k (and v) host -> device buffer set i % 2
//   compute:  cp_shard_plan; zigzag: cp_attn_prefill (queries read and O / LSE
//             written by token index); interleave: cp_restore of the queries
//             into shard (cat) order and cp_attn_partial_restore (the restore
//             fused into the store)
//   download: O and LSE device -> host
// Two device buffer sets let batch i's attention overlap batch i+1's upload
// and batch i-1's download; events order every reuse of a buffer set.
#include <algorithm>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/cpattn.h"
#include "host_plan.h"
#include "trace.h"

namespace {

inline long long r256(long long x) { return (x + 255) & ~255LL; }

struct PrefillLayout {
  long long rows, segs, tiles, kv_rows;
  // byte offsets in the workspace
  long long lens, segs_off, seg_offs, row_offs, gather, pos, restore, tiles_off;
  long long set_off[2], q, k, v, q_cat, o, lse;  // q..lse: offsets inside a set
  long long set_bytes, total;
};

int prefill_layout(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                   int cp_size, int strategy, int Hq, int Hkv, int d, int dv, int v_is_k_prefix,
                   PrefillLayout* L) {
  if (Hq < 1 || Hkv < 1 || d < 1 || dv < 1 || (v_is_k_prefix && dv > d))
    return CPATTN_ERR_INVALID_ARG;
  std::vector<int32_t> rows(cp_size > 0 ? cp_size : 1), segs(rows.size()), tiles(rows.size());
  const int rc = cp_shard_plan_sizes(new_lens, prefix_lens, num_reqs, cp_size, strategy,
                                     rows.data(), segs.data(), tiles.data());
  if (rc != CPATTN_OK) return rc;
  L->rows = L->segs = L->tiles = L->kv_rows = 0;
  for (int r = 0; r < cp_size; ++r) {
    L->rows += rows[r];
    L->segs += segs[r];
    L->tiles += tiles[r];
  }
  for (int b = 0; b < num_reqs; ++b) L->kv_rows += (long long)new_lens[b] + prefix_lens[b];
  long long off = 0;
  auto take = [&](long long bytes) {
    const long long o = off;
    off += r256(std::max(bytes, 16LL));
    return o;
  };
  L->lens = take(2LL * std::max(num_reqs, 1) * 4);
  L->segs_off = take(std::max(L->segs, 1LL) * (long long)sizeof(cp_segment_t));
  L->seg_offs = take((cp_size + 1LL) * 4);
  L->row_offs = take((cp_size + 1LL) * 4);
  L->gather = take(std::max(L->rows, 1LL) * 4);
  L->pos = take(std::max(L->rows, 1LL) * 4);
  L->restore = take(std::max(L->rows, 1LL) * 4);
  L->tiles_off = take(std::max(L->tiles, 1LL) * 8);
  long long so = 0;
  auto take_set = [&](long long bytes) {
    const long long o = so;
    so += r256(std::max(bytes, 16LL));
    return o;
  };
  L->q = take_set(L->rows * Hq * d * 2);
  L->k = take_set(L->kv_rows * Hkv * d * 2);
  L->v = v_is_k_prefix ? -1 : take_set(L->kv_rows * Hkv * dv * 2);
  L->q_cat = strategy == CP_INTERLEAVE ? take_set(L->rows * Hq * d * 2) : -1;
  L->o = take_set(L->rows * Hq * dv * 2);
  L->lse = take_set(L->rows * Hq * 4);
  L->set_bytes = so;
  L->set_off[0] = off;
  L->set_off[1] = off + so;
  L->total = off + 2 * so;
  return CPATTN_OK;
}

}  // namespace

extern "C" int cp_prefill_host_workspace_size(const int32_t* new_lens, const int32_t* prefix_lens,
                                              int num_reqs, int cp_size, int strategy, int Hq,
                                              int Hkv, int d, int dv, int v_is_k_prefix,
                                              int64_t* bytes) {
  if (!bytes) return CPATTN_ERR_INVALID_ARG;
  PrefillLayout L;
  const int rc = prefill_layout(new_lens, prefix_lens, num_reqs, cp_size, strategy, Hq, Hkv, d, dv,
                                v_is_k_prefix, &L);
  if (rc != CPATTN_OK) return rc;
  *bytes = L.total;
  return CPATTN_OK;
}

extern "C" int cp_prefill_host(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                               int cp_size, int strategy, int Hq, int Hkv, int d, int dv,
                               float scale, int v_is_k_prefix, int num_batches,
                               const void* const* q_host, const void* const* k_host,
                               const void* const* v_host, void* const* o_host,
                               float* const* lse_host, void* workspace, int64_t workspace_bytes,
                               int32_t* status_dev, cudaStream_t compute, cudaStream_t upload,
                               cudaStream_t download) {
  CPATTN_TRACE("cp_prefill_host");
  PrefillLayout L;
  int rc = prefill_layout(new_lens, prefix_lens, num_reqs, cp_size, strategy, Hq, Hkv, d, dv,
                          v_is_k_prefix, &L);
  if (rc != CPATTN_OK) return rc;
  if (num_batches < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_batches == 0 || L.rows == 0) return CPATTN_OK;
  if (!q_host || !k_host || !o_host || !lse_host || (!v_is_k_prefix && !v_host))
    return CPATTN_ERR_INVALID_ARG;
  for (int i = 0; i < num_batches; ++i)
    if (!q_host[i] || !k_host[i] || !o_host[i] || !lse_host[i] || (!v_is_k_prefix && !v_host[i]))
      return CPATTN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < L.total) return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return CPATTN_ERR_ALIGNMENT;
  auto* ws = static_cast<uint8_t*>(workspace);
  auto* lens_dev = reinterpret_cast<int32_t*>(ws + L.lens);
  auto* segs = reinterpret_cast<cp_segment_t*>(ws + L.segs_off);
  auto* seg_offs = reinterpret_cast<int32_t*>(ws + L.seg_offs);
  auto* row_offs = reinterpret_cast<int32_t*>(ws + L.row_offs);
  auto* gather = reinterpret_cast<int32_t*>(ws + L.gather);
  auto* pos = reinterpret_cast<int32_t*>(ws + L.pos);
  auto* restore = reinterpret_cast<int32_t*>(ws + L.restore);
  auto* tiles = reinterpret_cast<int32_t*>(ws + L.tiles_off);

  const size_t q_bytes = (size_t)L.rows * Hq * d * 2, k_bytes = (size_t)L.kv_rows * Hkv * d * 2;
  const size_t v_bytes = (size_t)L.kv_rows * Hkv * dv * 2;
  const size_t o_bytes = (size_t)L.rows * Hq * dv * 2, l_bytes = (size_t)L.rows * Hq * 4;

  // events: upload done, compute done, download done, per buffer set
  cudaEvent_t ev[3][2] = {};
  bool ok = true;
  for (int a = 0; a < 3 && ok; ++a)
    for (int s = 0; s < 2 && ok; ++s)
      ok = cudaEventCreateWithFlags(&ev[a][s], cudaEventDisableTiming) == cudaSuccess;
  auto release = [&]() {
    for (int a = 0; a < 3; ++a)
      for (int s = 0; s < 2; ++s)
        if (ev[a][s]) cudaEventDestroy(ev[a][s]);  // freed once their work completes
  };
  if (!ok) {
    release();
    return CPATTN_ERR_CUDA;
  }
  // request lengths, once (the plan is rebuilt for every batch on the compute
  // stream, as the device step does)
  if (num_reqs > 0 &&
      (cudaMemcpyAsync(lens_dev, new_lens, (size_t)num_reqs * 4, cudaMemcpyHostToDevice,
                       compute) != cudaSuccess ||
       cudaMemcpyAsync(lens_dev + num_reqs, prefix_lens, (size_t)num_reqs * 4,
                       cudaMemcpyHostToDevice, compute) != cudaSuccess)) {
    release();
    return CPATTN_ERR_CUDA;
  }
  rc = CPATTN_OK;
  for (int i = 0; i < num_batches && rc == CPATTN_OK; ++i) {
    const int s = i % 2;
    uint8_t* set = ws + L.set_off[s];
    void* dq = set + L.q;
    void* dk = set + L.k;
    const void* dv_ptr = v_is_k_prefix ? dk : static_cast<const void*>(set + L.v);
    void* dqc = L.q_cat >= 0 ? set + L.q_cat : nullptr;
    void* dout = set + L.o;
    float* dlse = reinterpret_cast<float*>(set + L.lse);
    const bool reuse = i >= 2;
    // upload batch i once batch i-2 has finished reading set s
    if (reuse && cudaStreamWaitEvent(upload, ev[1][s], 0) != cudaSuccess) { rc = CPATTN_ERR_CUDA; break; }
    if (cudaMemcpyAsync(dq, q_host[i], q_bytes, cudaMemcpyHostToDevice, upload) != cudaSuccess ||
        cudaMemcpyAsync(dk, k_host[i], k_bytes, cudaMemcpyHostToDevice, upload) != cudaSuccess ||
        (!v_is_k_prefix && cudaMemcpyAsync(set + L.v, v_host[i], v_bytes, cudaMemcpyHostToDevice,
                                           upload) != cudaSuccess) ||
        cudaEventRecord(ev[0][s], upload) != cudaSuccess) {
      rc = CPATTN_ERR_CUDA;
      break;
    }
    // compute once the upload is in and batch i-2's outputs are downloaded
    if (cudaStreamWaitEvent(compute, ev[0][s], 0) != cudaSuccess ||
        (reuse && cudaStreamWaitEvent(compute, ev[2][s], 0) != cudaSuccess)) {
      rc = CPATTN_ERR_CUDA;
      break;
    }
    rc = cp_shard_plan(lens_dev, lens_dev + num_reqs, num_reqs, cp_size, strategy, (int)L.rows,
                       (int)L.segs, (int)L.tiles, segs, seg_offs, row_offs, gather, pos, restore,
                       tiles, status_dev, compute);
    if (rc != CPATTN_OK) break;
    const int64_t k_row = (int64_t)Hkv * d, v_row = v_is_k_prefix ? k_row : (int64_t)Hkv * dv;
    const int64_t v_head = v_is_k_prefix ? d : dv;
    if (strategy == CP_ZIGZAG) {
      rc = cp_attn_prefill(segs, (int)L.segs, tiles, (int)L.tiles, dq, (int)L.rows, dk, k_row, d,
                           dv_ptr, v_row, v_head, (int)L.kv_rows, Hq, Hkv, d, dv, scale, dout, 0,
                           dlse, status_dev, compute);
    } else {
      rc = cp_restore(dq, (int)L.rows, gather, (int)L.rows, (int64_t)Hq * d * 2, dqc, status_dev,
                      compute);
      if (rc == CPATTN_OK)
        rc = cp_attn_partial_restore(segs, (int)L.segs, tiles, (int)L.tiles, dqc, (int)L.rows, dk,
                                     k_row, d, dv_ptr, v_row, v_head, (int)L.kv_rows, Hq, Hkv, d,
                                     dv, scale, 0, -1, gather, dout, 0, dlse, (int)L.rows,
                                     status_dev, compute);
    }
    if (rc != CPATTN_OK) break;
    if (cudaEventRecord(ev[1][s], compute) != cudaSuccess ||
        cudaStreamWaitEvent(download, ev[1][s], 0) != cudaSuccess ||
        cudaMemcpyAsync(o_host[i], dout, o_bytes, cudaMemcpyDeviceToHost, download) != cudaSuccess ||
        cudaMemcpyAsync(lse_host[i], dlse, l_bytes, cudaMemcpyDeviceToHost, download) !=
            cudaSuccess ||
        cudaEventRecord(ev[2][s], download) != cudaSuccess) {
      rc = CPATTN_ERR_CUDA;
      break;
    }
  }
  // the download stream ends after every batch's compute and download
  if (rc == CPATTN_OK) {
    for (int s = 0; s < 2 && rc == CPATTN_OK; ++s)
      if (cudaStreamWaitEvent(download, ev[1][s], 0) != cudaSuccess) rc = CPATTN_ERR_CUDA;
  }
  release();
  return rc;
}
