// Pass-Q ring: schedule (host) and the whole ring as one call (device).
//
// Blog "什么是 Context Parallelism", §3.3.2 (pass-Q: the KV stays where it is,
// each rank's query block travels round the ring and carries a partial
// accumulator (O_acc, L_acc); every hop merges the local partial into it) and
// §3.5 (the persistent KV cache is split into 2N blocks and rank i keeps the
// first/last pair i and 2N-1-i).
//
// KV residency: each request's key positions 0..p+n-1 are cut into 2C blocks
// like the zigzag query split (the remainder goes to the first blocks) and
// rank r keeps blocks r and 2C-1-r.  At ring hop s the query shard of rank q
// is on rank (q + s) mod C.  Every (hop, resident block) pair is one launch of
// the accumulate kernel: it takes every plan segment whose request's block on
// its host rank is non-empty and starts at or before the segment's last
// position, with that block as the segment's key window.  A launch never
// holds a row twice (a row is on exactly one host rank at a hop), so it
// merges every rank's hop at once: at most 2C launches for any batch.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "attn_common.cuh"
#include "host_plan.h"
#include "trace.h"

namespace cpattn {
namespace {

// Resident block b (0: block r, 1: block 2C-1-r) of rank r for a request
// with kv_total key positions: [lo, hi).
void resident_block(long long kv_total, int C, int r, int b, long long* lo, long long* hi) {
  const long long nb = 2LL * C, base = kv_total / nb, rem = kv_total % nb;
  const long long k = b == 0 ? r : nb - 1 - r;
  *lo = k * base + std::min(k, rem);
  *hi = *lo + base + (k < rem ? 1 : 0);
}

struct RingEntry {
  int hop, block, seg_id;
  cp_segment_t seg;
  int32_t lo, hi;
};

// The schedule's entries in launch order (hop-major, block-minor, then
// segment-table order).
int ring_entries(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs, int cp_size,
                 int strategy, std::vector<RingEntry>& out) {
  std::vector<cp_segment_t> segs;
  std::vector<int> rank_of;
  const int rc = for_each_plan_segment(new_lens, prefix_lens, num_reqs, cp_size, strategy,
                                       [&](int r, const cp_segment_t& s) {
                                         segs.push_back(s);
                                         rank_of.push_back(r);
                                       });
  if (rc != CPATTN_OK) return rc;
  out.clear();
  for (int hop = 0; hop < cp_size; ++hop)
    for (int b = 0; b < 2; ++b)
      for (size_t i = 0; i < segs.size(); ++i) {
        const cp_segment_t& s = segs[i];
        const int host = (rank_of[i] + hop) % cp_size;
        const long long kv_total = (long long)new_lens[s.req] + prefix_lens[s.req];
        long long lo, hi;
        resident_block(kv_total, cp_size, host, b, &lo, &hi);
        if (hi > lo && lo <= segment_last_pos(s))
          out.push_back(RingEntry{hop, b, (int)i, s, (int32_t)lo, (int32_t)hi});
      }
  return CPATTN_OK;
}

// O = 0 and both LSE buffers = -inf: the identity of the LSE merge.
__global__ void ring_init_kernel(float4* __restrict__ o, long long n_o4, float* __restrict__ la,
                                 float* __restrict__ lb, long long n_l) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_o4; i += stride)
    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_l; i += stride) {
    la[i] = -INFINITY;
    lb[i] = -INFINITY;
  }
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" int cp_pass_q_schedule_size(const int32_t* new_lens, const int32_t* prefix_lens,
                                       int num_reqs, int cp_size, int strategy,
                                       int32_t* num_launches, int32_t* num_entries) {
  if (!num_launches || !num_entries) return CPATTN_ERR_INVALID_ARG;
  std::vector<RingEntry> e;
  const int rc = ring_entries(new_lens, prefix_lens, num_reqs, cp_size, strategy, e);
  if (rc != CPATTN_OK) return rc;
  int launches = 0;
  for (size_t i = 0; i < e.size(); ++i)
    if (i == 0 || e[i].hop != e[i - 1].hop || e[i].block != e[i - 1].block) ++launches;
  if (e.size() > 0x7fffffffULL) return CPATTN_ERR_INVALID_ARG;
  *num_launches = launches;
  *num_entries = (int32_t)e.size();
  return CPATTN_OK;
}

extern "C" int cp_pass_q_schedule(const int32_t* new_lens, const int32_t* prefix_lens,
                                  int num_reqs, int cp_size, int strategy, int32_t* launch_first,
                                  int32_t* launch_hop, int32_t* launch_block,
                                  cp_segment_t* entry_segs, int32_t* entry_windows,
                                  int32_t* entry_seg_ids) {
  std::vector<RingEntry> e;
  const int rc = ring_entries(new_lens, prefix_lens, num_reqs, cp_size, strategy, e);
  if (rc != CPATTN_OK) return rc;
  if (!launch_first || (!e.empty() && (!entry_segs || !entry_windows)))
    return CPATTN_ERR_INVALID_ARG;
  int li = 0;
  for (size_t i = 0; i < e.size(); ++i) {
    if (i == 0 || e[i].hop != e[i - 1].hop || e[i].block != e[i - 1].block) {
      launch_first[li] = (int32_t)i;
      if (launch_hop) launch_hop[li] = e[i].hop;
      if (launch_block) launch_block[li] = e[i].block;
      ++li;
    }
    entry_segs[i] = e[i].seg;
    entry_windows[2 * i] = e[i].lo;
    entry_windows[2 * i + 1] = e[i].hi;
    if (entry_seg_ids) entry_seg_ids[i] = e[i].seg_id;
  }
  launch_first[li] = (int32_t)e.size();
  return CPATTN_OK;
}

extern "C" int cp_attn_pass_q(const cp_segment_t* entry_segs_dev, const int32_t* entry_windows_dev,
                              const int32_t* launch_first, int num_launches, const void* q,
                              int num_q_rows, const void* k, int64_t k_row_stride,
                              int64_t k_head_stride, const void* v, int64_t v_row_stride,
                              int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv, int d,
                              int dv, float scale, float* o_acc, float* lse, float* lse_scratch,
                              int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_pass_q");
  if (num_launches < 0 || num_q_rows < 0 || Hq < 1 || dv < 4 || (dv % 4) != 0)
    return CPATTN_ERR_INVALID_ARG;
  if (num_q_rows == 0) return CPATTN_OK;
  if (!o_acc || !lse || !lse_scratch || (num_launches > 0 && !launch_first))
    return CPATTN_ERR_INVALID_ARG;
  if (!a16(o_acc) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse_scratch) & 3u))
    return CPATTN_ERR_ALIGNMENT;
  for (int i = 0; i < num_launches; ++i)
    if (launch_first[i] < 0 || launch_first[i + 1] < launch_first[i]) return CPATTN_ERR_INVALID_ARG;
  const long long n_l = (long long)num_q_rows * Hq;
  const long long n_o4 = n_l * dv / 4;
  ring_init_kernel<<<4 * 152, 256, 0, stream>>>(reinterpret_cast<float4*>(o_acc), n_o4, lse,
                                                lse_scratch, n_l);
  if (cudaGetLastError() != cudaSuccess) return CPATTN_ERR_CUDA;
  for (int i = 0; i < num_launches; ++i) {
    const int first = launch_first[i], n = launch_first[i + 1] - first;
    if (n == 0) continue;
    // the hop's partials merge into (o_acc, lse) -> (o_acc, lse_scratch); the
    // rows this launch did not hold keep equal values in both LSE buffers once
    // the new values are copied back
    const int rc = cp_attn_partial_accumulate(
        entry_segs_dev + first, n, nullptr, 0, q, num_q_rows, k, k_row_stride, k_head_stride, v,
        v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv, scale, 0, -1,
        entry_windows_dev + 2 * (long long)first, o_acc, lse, lse_scratch, 0, num_q_rows,
        status_dev, stream);
    if (rc != CPATTN_OK) return rc;
    if (cudaMemcpyAsync(lse, lse_scratch, n_l * sizeof(float), cudaMemcpyDeviceToDevice, stream) !=
        cudaSuccess)
      return CPATTN_ERR_CUDA;
  }
  return CPATTN_OK;
}
