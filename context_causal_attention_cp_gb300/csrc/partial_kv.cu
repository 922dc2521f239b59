// Partial-KV (ring-style) decomposition of shard attention in one call.
//
// Blog "什么是 Context Parallelism", §2.1 item 2 and §3.1: when the whole KV
// does not fit, a rank's queries meet the KV one block at a time, each block
// giving a partial output O_j with its log-sum-exp L_j, and the LSE merge
// (§3.6) makes the result equal to attention over all keys.  On one GPU the
// ring's rotation becomes a loop over KV blocks in HBM; here every visible
// (query tile, KV block) pair runs in a single split-KV attention launch.
//
// Three launches on the caller's stream:
//   1. pkv_layout_kernel: per segment, the number of visible KV blocks nb_s
//      and the first workspace row of its partials (slot_s, an exclusive scan
//      of nb_s * q_len_s), plus the running count of segment rows.
//   2. the attention kernel in split mode: CTA (tile, block j, heads) writes
//      its fp32 partial (O_j, L_j) at workspace rows slot_s + j*q_len_s + i.
//   3. pkv_merge_kernel: per (segment row, head), the LSE merge of its nb_s
//      partials, written to output row dst_rows[cat row] (the restore).
//
// Workspace layout (caller-allocated, see cp_partial_kv_workspace_size):
//   int64 slot[num_segs] | int64 rows_before[num_segs + 1] | int64 total
//   (padded to 256 B) | fp32 O partials [cap_rows, Hq, dv] (padded to 256 B) |
//   fp32 L partials [cap_rows, Hq]; cap_rows follows from the byte size.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "attn_common.cuh"
#include "host_plan.h"
#include "trace.h"

namespace cpattn {
namespace {

constexpr int kLayoutThreads = 1024;

__host__ __device__ inline long long round256(long long x) { return (x + 255) & ~255LL; }

struct PkvLayout {
  long long header_bytes, cap_rows, o_off, l_off;
};

inline PkvLayout pkv_layout(int num_segs, int Hq, int dv, long long workspace_bytes) {
  PkvLayout L;
  L.header_bytes = round256((2LL * num_segs + 2) * 8);
  const long long per_row = (long long)Hq * (dv + 1) * 4;
  const long long avail = workspace_bytes - L.header_bytes - 256;
  L.cap_rows = avail > 0 ? avail / per_row : 0;
  L.o_off = L.header_bytes;
  L.l_off = L.o_off + round256(L.cap_rows * Hq * dv * 4);
  return L;
}

// Block-wide exclusive scan of one 64-bit value per thread (blockDim == 1024).
__device__ long long block_scan64(long long v, long long* buf /* >= 33 */, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) buf[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const long long w = lane < (int)(blockDim.x >> 5) ? buf[lane] : 0;
    long long s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    buf[lane] = s - w;
    if (lane == 31) buf[32] = s;
  }
  __syncthreads();
  const long long r = buf[wid] + x - v;
  *total = buf[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kLayoutThreads)
pkv_layout_kernel(const cp_segment_t* __restrict__ segs, int num_segs, int kv_block,
                  int max_blocks, long long cap_rows, long long* __restrict__ slot,
                  long long* __restrict__ rows_before, long long* __restrict__ total,
                  int32_t* status) {
  grid_dep_trigger();  // the attention launch may start its loads and MMAs now
  __shared__ long long buf[33];
  long long slot_carry = 0, row_carry = 0;
  for (int c0 = 0; c0 < num_segs; c0 += kLayoutThreads) {
    const int s = c0 + threadIdx.x;
    long long parts = 0, rows = 0;
    if (s < num_segs) {
      const cp_segment_t sg = segs[s];
      if (sg.q_len <= 0 || sg.q_pos0 < 0 || sg.q_pos_step < 0) {
        set_status(status, CPATTN_ERR_RANGE);
      } else {
        const int nb = segment_blocks(sg, kv_block);
        if (nb > max_blocks) set_status(status, CPATTN_ERR_INVALID_ARG);
        rows = sg.q_len;
        parts = (long long)nb * sg.q_len;
      }
    }
    long long t1, t2;
    const long long so = slot_carry + block_scan64(parts, buf, &t1);
    const long long ro = row_carry + block_scan64(rows, buf, &t2);
    if (s < num_segs) {
      slot[s] = so;
      rows_before[s] = ro;
    }
    slot_carry += t1;
    row_carry += t2;
  }
  if (threadIdx.x == 0) {
    rows_before[num_segs] = row_carry;
    *total = slot_carry;
    if (slot_carry > cap_rows) set_status(status, CPATTN_ERR_INVALID_ARG);
  }
}

constexpr int kMergeThreadsP = 256;
constexpr int kGroupP = 16;
constexpr int kFewLoads = 8;  // partial loads per lane per step with few partials

__device__ __forceinline__ float4 ld_stream4(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Merge of one segment row's partials for all heads, NP <= 8 partials: a
// warp step merges U = 8 / NP heads (at least one) so that each lane has
// about 8 partial loads in flight.  Lane L < U*NP owns L_j of (head h0 + L / NP,
// partial L % NP); the normalised weights are broadcast by shuffles.
//   o_row: partial 0 of the row, all heads ([Hq, dv] fp32); part_stride /
//   l_stride: distance between a row's consecutive partials.
template <bool OUT_F32, int NP>
__device__ __forceinline__ void pkv_merge_row_few(const float* __restrict__ o_row,
                                                  const float* __restrict__ l_row,
                                                  long long part_stride, long long l_stride,
                                                  int Hq, int hb, int he, int dv,
                                                  long long out_row, void* __restrict__ o_out,
                                                  float* __restrict__ lse_out, int lane) {
  constexpr int U = kFewLoads / NP > 0 ? kFewLoads / NP : 1;
  const int ui_l = lane / NP, j_l = lane - ui_l * NP;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int h0 = hb; h0 < he; h0 += U) {
    const int h_l = h0 + ui_l;
    float lj = -INFINITY;
    if (lane < U * NP && h_l < he) lj = __ldg(l_row + j_l * l_stride + h_l);
    float v4[U * NP][4];
    for (int c0 = 0; c0 < dv; c0 += 128) {
      const int c = c0 + lane * 4;
      const bool act = c < dv;
#pragma unroll
      for (int sl = 0; sl < U * NP; ++sl) {
        const int ui = sl / NP, j = sl - ui * NP;
        const float4 v = (act && h0 + ui < he)
                             ? ld_stream4(o_row + j * part_stride + (long long)(h0 + ui) * dv + c)
                             : zero;
        v4[sl][0] = v.x; v4[sl][1] = v.y; v4[sl][2] = v.z; v4[sl][3] = v.w;
      }
      if (c0 == 0) {
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < NP; ++j) m = fmaxf(m, __shfl_sync(0xffffffffu, lj, (ui_l * NP + j) & 31));
        const bool empty = (m == -INFINITY);
        const float w = empty ? 0.f : __expf(lj - m);
        float sw = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) sw += __shfl_sync(0xffffffffu, w, (ui_l * NP + j) & 31);
        lj = empty ? 0.f : w / sw;  // now the normalised weight
        if (lse_out && lane < U * NP && j_l == 0 && h_l < he)
          lse_out[out_row * Hq + h_l] = empty ? -INFINITY : m + __logf(sw);
      }
#pragma unroll
      for (int ui = 0; ui < U; ++ui) {
        float ax = 0.f, ay = 0.f, az = 0.f, aw = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          const float w = __shfl_sync(0xffffffffu, lj, ui * NP + j);
          ax = fmaf(w, v4[ui * NP + j][0], ax);
          ay = fmaf(w, v4[ui * NP + j][1], ay);
          az = fmaf(w, v4[ui * NP + j][2], az);
          aw = fmaf(w, v4[ui * NP + j][3], aw);
        }
        if (!act || h0 + ui >= he) continue;
        const long long oo = (out_row * Hq + h0 + ui) * dv + c;
        if (OUT_F32) {
          __stcs(reinterpret_cast<float4*>(static_cast<float*>(o_out) + oo),
                 make_float4(ax, ay, az, aw));
        } else {
          uint2 pk;
          pk.x = pack_bf16x2(ax, ay);
          pk.y = pack_bf16x2(az, aw);
          __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + oo), pk);
        }
      }
    }
  }
}

// Merge of one segment row's nb (> 8, <= 32) partials, one head per warp
// step: lane j holds L_j; partial loads in groups of kGroupP per lane, the
// first group issued with the L_j load.
template <bool OUT_F32>
__device__ __forceinline__ void pkv_merge_row_many(const float* __restrict__ o_row,
                                                   const float* __restrict__ l_row, int nb,
                                                   long long part_stride, long long l_stride,
                                                   int Hq, int hb, int he, int dv,
                                                   long long out_row, void* __restrict__ o_out,
                                                   float* __restrict__ lse_out, int lane) {
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int h = hb; h < he; ++h) {
    const float* base = o_row + (long long)h * dv;
    float lj = -INFINITY;
    if (lane < nb) lj = __ldg(l_row + lane * l_stride + h);
    float4 v[kGroupP];
    {
      const int c = lane * 4;
      const bool act = c < dv;
#pragma unroll
      for (int jj = 0; jj < kGroupP; ++jj)
        v[jj] = (act && jj < nb) ? ld_stream4(base + jj * part_stride + c) : zero;
    }
    float m = lj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const bool empty = (m == -INFINITY);
    const float wj = (lane < nb && !empty) ? __expf(lj - m) : 0.f;
    float ws = wj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    const float inv = empty ? 0.f : 1.f / ws;
    for (int c0 = 0; c0 < dv; c0 += 128) {
      const int c = c0 + lane * 4;
      const bool act = c < dv;
      float4 acc = zero;
      for (int j0 = 0; j0 < nb; j0 += kGroupP) {
        if (c0 > 0 || j0 > 0) {
#pragma unroll
          for (int jj = 0; jj < kGroupP; ++jj)
            v[jj] = (act && j0 + jj < nb) ? ld_stream4(base + (j0 + jj) * part_stride + c) : zero;
        }
#pragma unroll
        for (int jj = 0; jj < kGroupP; ++jj) {
          const float w = __shfl_sync(0xffffffffu, wj, (j0 + jj) & 31);
          acc.x = fmaf(w, v[jj].x, acc.x);
          acc.y = fmaf(w, v[jj].y, acc.y);
          acc.z = fmaf(w, v[jj].z, acc.z);
          acc.w = fmaf(w, v[jj].w, acc.w);
        }
      }
      if (!act) continue;
      acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      const long long oo = (out_row * Hq + h) * dv + c;
      if (OUT_F32) {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(o_out) + oo), acc);
      } else {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + oo), pk);
      }
    }
    if (lse_out && lane == 0) lse_out[out_row * Hq + h] = empty ? -INFINITY : m + __logf(ws);
  }
}

// One warp per (segment row, slice of hs heads): find the row's segment once
// (binary search on rows_before), check the row's partials and destination,
// then merge its nb partials for the slice's heads.  hs = Hq when there are
// rows enough to fill the GPU, smaller for a few rows (e.g. decode).
template <bool OUT_F32>
__global__ void __launch_bounds__(kMergeThreadsP, 2)
pkv_merge_kernel(const cp_segment_t* __restrict__ segs, int num_segs, int kv_block,
                 const long long* __restrict__ slot, const long long* __restrict__ rows_before,
                 const float* __restrict__ ws_o, const float* __restrict__ ws_l, long long cap_rows,
                 int Hq, int dv, int num_q_rows, const int32_t* __restrict__ dst_rows,
                 void* __restrict__ o_out, float* __restrict__ lse_out, int num_out_rows,
                 int hs, int32_t* status) {
  grid_dep_wait();  // the attention launch before this one wrote the partials
  const int lane = threadIdx.x & 31;
  const int nslices = (Hq + hs - 1) / hs;
  const long long total_tasks = rows_before[num_segs] * nslices;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long task = warp0; task < total_tasks; task += nwarps) {
    const long long gr = task / nslices;
    const int hb = (int)(task - gr * nslices) * hs, he = min(Hq, hb + hs);
    int lo = 0, hi = num_segs;  // last segment with rows_before <= gr
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (rows_before[mid] <= gr) lo = mid; else hi = mid;
    }
    const cp_segment_t sg = segs[lo];
    const int i = (int)(gr - rows_before[lo]);
    const long long cat_row = (long long)sg.q_row0 + i;
    if (i < 0 || i >= sg.q_len || cat_row < 0 || cat_row >= num_q_rows) {
      if (lane == 0) set_status(status, CPATTN_ERR_RANGE);
      continue;
    }
    const int nb = segment_blocks(sg, kv_block);
    const long long first = slot[lo] + i;  // partial 0 of this row
    const long long out_row = dst_rows ? (long long)__ldg(dst_rows + cat_row) : cat_row;
    if (nb < 1 || nb > 32 || first + (long long)(nb - 1) * sg.q_len >= cap_rows || out_row < 0 ||
        out_row >= num_out_rows) {
      if (lane == 0) set_status(status, CPATTN_ERR_RANGE);
      continue;
    }
    const float* o_row = ws_o + first * Hq * dv;
    const float* l_row = ws_l + first * Hq;
    const long long part_stride = (long long)sg.q_len * Hq * dv;
    const long long l_stride = (long long)sg.q_len * Hq;
    switch (nb) {
#define CPATTN_PKV_FEW(NPV)                                                                    \
  case NPV:                                                                                    \
    pkv_merge_row_few<OUT_F32, NPV>(o_row, l_row, part_stride, l_stride, Hq, hb, he, dv,      \
                                    out_row, o_out, lse_out, lane);                            \
    break;
      CPATTN_PKV_FEW(1) CPATTN_PKV_FEW(2) CPATTN_PKV_FEW(3) CPATTN_PKV_FEW(4)
      CPATTN_PKV_FEW(5) CPATTN_PKV_FEW(6) CPATTN_PKV_FEW(7) CPATTN_PKV_FEW(8)
#undef CPATTN_PKV_FEW
      default:
        pkv_merge_row_many<OUT_F32>(o_row, l_row, nb, part_stride, l_stride, Hq, hb, he, dv,
                                    out_row, o_out, lse_out, lane);
    }
  }
}

// SM count of the current device, cached per device.
int num_sms() {
  constexpr int kMaxDev = 64;
  static int cached[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < kMaxDev && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < kMaxDev) cached[dev] = n;
  return n;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

namespace {

// Workspace bytes for `rows` partial rows of `segs` segments (the layout at
// the top of this file).
int64_t pkv_workspace_bytes(long long segs, long long rows, int Hq, int dv) {
  const long long header = round256((2 * segs + 2) * 8);
  return header + round256(rows * Hq * dv * 4) + round256(rows * Hq * 4) + 256;
}

// Running sizes over a segment table: partial rows, segments, the largest
// block count and the longest segment.
struct PkvSizes {
  long long rows = 0, segs = 0, max_blocks = 0, max_rows = 0;
  void add(const cp_segment_t& s, int kv_block) {
    if (s.q_len <= 0) return;
    const long long nb = segment_last_pos(s) / kv_block + 1;
    rows += nb * s.q_len;
    segs += 1;
    max_blocks = std::max(max_blocks, nb);
    max_rows = std::max<long long>(max_rows, s.q_len);
  }
  void write(int Hq, int dv, int64_t* bytes, int32_t* mb, int32_t* msr, long long table_segs) const {
    *bytes = pkv_workspace_bytes(table_segs, rows, Hq, dv);
    if (mb) *mb = (int32_t)std::min<long long>(max_blocks, 0x7fffffff);
    if (msr) *msr = (int32_t)max_rows;
  }
};

}  // namespace

extern "C" int cp_partial_kv_workspace_size(const int32_t* new_lens, const int32_t* prefix_lens,
                                            int num_reqs, int cp_size, int strategy, int kv_block,
                                            int Hq, int dv, int64_t* bytes, int32_t* max_blocks,
                                            int32_t* max_seg_rows) {
  if (kv_block < 1 || Hq < 1 || dv < 4 || (dv % 4) != 0 || !bytes) return CPATTN_ERR_INVALID_ARG;
  PkvSizes sz;
  // the segments cp_shard_plan makes for these lengths
  const int rc = for_each_plan_segment(new_lens, prefix_lens, num_reqs, cp_size, strategy,
                                       [&](int, const cp_segment_t& s) { sz.add(s, kv_block); });
  if (rc != CPATTN_OK) return rc;
  sz.write(Hq, dv, bytes, max_blocks, max_seg_rows, sz.segs);
  return CPATTN_OK;
}

extern "C" int cp_partial_kv_workspace_size_segs(const cp_segment_t* segs_host, int num_segs,
                                                 int kv_block, int Hq, int dv, int64_t* bytes,
                                                 int32_t* max_blocks, int32_t* max_seg_rows) {
  if (num_segs < 0 || kv_block < 1 || Hq < 1 || dv < 4 || (dv % 4) != 0 || !bytes)
    return CPATTN_ERR_INVALID_ARG;
  if (num_segs > 0 && !segs_host) return CPATTN_ERR_INVALID_ARG;
  PkvSizes sz;
  for (int i = 0; i < num_segs; ++i) {
    const cp_segment_t& sg = segs_host[i];
    if (sg.q_len < 0 || sg.q_pos0 < 0 || sg.q_pos_step < 0) return CPATTN_ERR_INVALID_ARG;
    sz.add(sg, kv_block);
  }
  sz.write(Hq, dv, bytes, max_blocks, max_seg_rows, num_segs);
  return CPATTN_OK;
}

extern "C" int cp_attn_partial_kv(const cp_segment_t* segs_dev, int num_segs,
                                  const int32_t* tiles_dev, int num_tiles, const void* q,
                                  int num_q_rows, const void* k, int64_t k_row_stride,
                                  int64_t k_head_stride, const void* v, int64_t v_row_stride,
                                  int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv, int d,
                                  int dv, float scale, int kv_block, int max_blocks,
                                  int max_seg_rows,
                                  const int32_t* dst_rows, void* o_out, int o_is_fp32,
                                  float* lse_out, int num_out_rows, void* workspace,
                                  int64_t workspace_bytes, int32_t* status_dev,
                                  cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_partial_kv");
  if (num_segs < 0 || kv_block < 1 || max_blocks < 0 || max_blocks > 32 || num_out_rows < 0 ||
      max_seg_rows < 0)
    return CPATTN_ERR_INVALID_ARG;
  // no segments (a batch without new tokens): nothing to compute; the sizing
  // calls report max_blocks = 0 for it
  if (num_segs == 0) return CPATTN_OK;
  if (max_blocks < 1) return CPATTN_ERR_INVALID_ARG;
  if (!o_out || !workspace || num_out_rows == 0 || Hq < 1 || dv < 4) return CPATTN_ERR_INVALID_ARG;
  if (!a16(o_out) || !a16(workspace) || (reinterpret_cast<uintptr_t>(lse_out) & 3u) ||
      (reinterpret_cast<uintptr_t>(dst_rows) & 3u))
    return CPATTN_ERR_ALIGNMENT;
  const PkvLayout L = pkv_layout(num_segs, Hq, dv, workspace_bytes);
  if (L.cap_rows <= 0) return CPATTN_ERR_INVALID_ARG;
  auto* base = static_cast<uint8_t*>(workspace);
  long long* slot = reinterpret_cast<long long*>(base);
  long long* rows_before = slot + num_segs;
  long long* total = rows_before + num_segs + 1;
  float* ws_o = reinterpret_cast<float*>(base + L.o_off);
  float* ws_l = reinterpret_cast<float*>(base + L.l_off);

  pkv_layout_kernel<<<1, kLayoutThreads, 0, stream>>>(segs_dev, num_segs, kv_block, max_blocks,
                                                      L.cap_rows, slot, rows_before, total,
                                                      status_dev);
  if (cudaGetLastError() != cudaSuccess) return CPATTN_ERR_CUDA;

  AttnParams prm{};
  prm.kv_lo = 0;
  prm.kv_hi = -1;
  prm.o = ws_o;
  prm.o_f32 = 1;
  prm.lse = ws_l;
  prm.out_row_base = 0;
  prm.num_out_rows = num_q_rows;  // output placement comes from the workspace slots
  prm.status = status_dev;
  prm.split_block = kv_block;
  prm.max_blocks = max_blocks;
  prm.ws_slot = slot;
  prm.ws_rows = L.cap_rows;
  prm.pack_heads = (max_seg_rows >= 1 && max_seg_rows <= BM / 2) ? 1 : 0;
  // the attention overlaps the layout kernel (it reads the slot table only
  // before its stores), and the merge's launch overlaps the attention's tail
  prm.pdl = 1;
  int rc = attn_launch(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k, k_row_stride,
                       k_head_stride, v, v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv,
                       scale, prm, stream);
  if (rc != CPATTN_OK) return rc;

  // heads per merge task: all of a row's heads, unless the rows (at most
  // num_q_rows) are too few to give every resident warp (two blocks per SM)
  // a task.  Each task walks a dependent chain (segment search, slot) before
  // its loads, so fewer, wider tasks beat one task per head on few rows.
  const long long resident_warps = (long long)num_sms() * 2 * (kMergeThreadsP / 32);
  int hs = Hq;
  while (hs > 1 && (long long)num_q_rows * ((Hq + hs - 1) / hs) < resident_warps)
    hs = (hs + 1) / 2;
  const long long tasks = (long long)num_q_rows * ((Hq + hs - 1) / hs);
  const int grid = (int)std::max<long long>(
      1, std::min<long long>((long long)num_sms() * 2 * 8,
                             (tasks + kMergeThreadsP / 32 - 1) / (kMergeThreadsP / 32)));
  const long long* slot_c = slot;
  const long long* rows_c = rows_before;
  const float* ws_o_c = ws_o;
  const float* ws_l_c = ws_l;
  const cudaError_t e =
      launch_kernel(o_is_fp32 ? pkv_merge_kernel<true> : pkv_merge_kernel<false>, (unsigned)grid,
                    kMergeThreadsP, 0, stream, true, segs_dev, num_segs, kv_block, slot_c, rows_c,
                    ws_o_c, ws_l_c, L.cap_rows, Hq, dv, num_q_rows, dst_rows, o_out, lse_out,
                    num_out_rows, hs, status_dev);
  return e == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}
