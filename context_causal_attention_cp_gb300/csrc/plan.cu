// Shard plan: zigzag / interleave query sharding for prefill context
// parallelism, the per-segment causal metadata, the gather / restore indices
// and a heaviest-first list of 128-row query tiles.
//
// Zigzag (SGLang docs, "Prefill Context Parallelism", §Zigzag strategy): each
// request's new tokens are cut into 2C contiguous blocks, early blocks taking
// the remainder (block k has n/2C tokens plus one when k < n mod 2C); rank r
// takes blocks r and 2C-1-r; the split restarts for every request.
// Interleave (same page, §Interleave strategy): rank r takes flattened
// new-token indices r, r+C, r+2C, ... across the whole batch; positions keep
// their original values.
// Restore index (blog "什么是 Context Parallelism", §2.1): flat index -> row of
// the all-gathered (rank-concatenated) buffer.
#include <cstdint>
#include <cstdlib>
#include <vector>

#include "../../include/cpattn.h"
#include "attn_common.cuh"
#include "ptx.cuh"
#include "trace.h"

namespace cpattn {
namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one int per thread (blockDim == kPlanThreads).
// Returns the exclusive prefix; *total receives the block sum.
__device__ int block_excl_scan(int v, int* scratch /* >= 33 ints */, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? scratch[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s - w;  // exclusive warp offsets
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  int res = scratch[wid] + x - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Block-wide exclusive scan of four ints per thread at once (any multiple of
// 32 threads up to 1024): one pass of warp shuffles and two barriers for all
// four.  v[] is replaced by its exclusive prefixes, total[] by the block sums.
__device__ void block_excl_scan4(int (&v)[4], int4* scratch /* >= 33 */, int (&total)[4]) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
  }
  if (lane == 31) scratch[wid] = make_int4(x[0], x[1], x[2], x[3]);
  __syncthreads();
  if (wid == 0) {
    const int nw = (int)(blockDim.x >> 5);
    const int4 w4 = lane < nw ? scratch[lane] : make_int4(0, 0, 0, 0);
    int w[4] = {w4.x, w4.y, w4.z, w4.w}, sacc[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int y = __shfl_up_sync(0xffffffffu, sacc[k], o);
        if (lane >= o) sacc[k] += y;
      }
    }
    scratch[lane] = make_int4(sacc[0] - w[0], sacc[1] - w[1], sacc[2] - w[2], sacc[3] - w[3]);
    if (lane == 31) scratch[32] = make_int4(sacc[0], sacc[1], sacc[2], sacc[3]);
  }
  __syncthreads();
  const int4 off = scratch[wid], tot = scratch[32];
  v[0] = off.x + x[0] - v[0];
  v[1] = off.y + x[1] - v[1];
  v[2] = off.z + x[2] - v[2];
  v[3] = off.w + x[3] - v[3];
  total[0] = tot.x;
  total[1] = tot.y;
  total[2] = tot.z;
  total[3] = tot.w;
  __syncthreads();
}

// Kernel 1: one CTA (a multiple of 32 threads, up to 1024, sized to the
// request count) writes every segment plus the rank offsets.
__global__ void __launch_bounds__(kPlanThreads)
plan_segments_kernel(const int32_t* __restrict__ new_lens, const int32_t* __restrict__ prefix_lens,
                     int num_reqs, int C, int strategy, int total_rows, int total_segs,
                     cp_segment_t* __restrict__ segs, int32_t* __restrict__ seg_offsets,
                     int32_t* __restrict__ row_offsets, int32_t* status) {
  grid_dep_trigger();  // the row and tile kernels may launch and wait for this one
  __shared__ int4 scan_buf[33];
  int row_base = 0, seg_base = 0;  // identical in every thread
  for (int r = 0; r < C; ++r) {
    if (threadIdx.x == 0) {
      row_offsets[r] = row_base;
      seg_offsets[r] = seg_base;
    }
    int flat_carry = 0, kv_carry = 0, row_carry = 0, seg_carry = 0;
    for (int c0 = 0; c0 < num_reqs; c0 += (int)blockDim.x) {
      const int b = c0 + threadIdx.x;
      const bool valid = b < num_reqs;
      int n = valid ? new_lens[b] : 0;
      int p = valid ? prefix_lens[b] : 0;
      if (n < 0 || p < 0) {
        set_status(status, CPATTN_ERR_INVALID_ARG);
        n = 0;
        p = 0;
      }
      // the request's flat start, KV start, and (below) its rows and segments
      // on rank r, as prefix sums over the batch; the flat start decides the
      // interleave counts, so it is scanned first
      int sc[4] = {n, n + p, 0, 0}, tot[4];
      if (strategy == CP_INTERLEAVE) {
        block_excl_scan4(sc, scan_buf, tot);
      } else {
        // zigzag counts do not depend on the flat start: one scan for all four
        const int nb = 2 * C, base = n / nb, rem = n % nb, kl = nb - 1 - r;
        const int e0 = base + (r < rem ? 1 : 0), l0 = base + (kl < rem ? 1 : 0);
        sc[2] = e0 + l0;
        sc[3] = (e0 > 0) + (l0 > 0);
        block_excl_scan4(sc, scan_buf, tot);
      }
      const int flat0 = flat_carry + sc[0];
      flat_carry += tot[0];
      const int kv0 = kv_carry + sc[1];
      kv_carry += tot[1];
      int rows_b = 0, segs_b = 0;
      int e = 0, l = 0, st_e = 0, st_l = 0, i0 = 0;
      if (strategy == CP_ZIGZAG) {
        const int nb = 2 * C, base = n / nb, rem = n % nb;
        const int kl = nb - 1 - r;
        e = base + (r < rem ? 1 : 0);
        l = base + (kl < rem ? 1 : 0);
        st_e = r * base + min(r, rem);
        st_l = kl * base + min(kl, rem);
        rows_b = e + l;
        segs_b = (e > 0) + (l > 0);
      } else {
        i0 = flat0 + ((r - flat0 % C) % C + C) % C;
        const int cnt = (i0 < flat0 + n) ? (flat0 + n - 1 - i0) / C + 1 : 0;
        rows_b = cnt;
        segs_b = cnt > 0;
        e = cnt;
      }
      int row_in_rank, seg_in_rank;
      if (strategy == CP_INTERLEAVE) {
        int sc2[4] = {rows_b, segs_b, 0, 0}, tot2[4];
        block_excl_scan4(sc2, scan_buf, tot2);
        row_in_rank = row_carry + sc2[0];
        row_carry += tot2[0];
        seg_in_rank = seg_carry + sc2[1];
        seg_carry += tot2[1];
      } else {
        row_in_rank = row_carry + sc[2];
        row_carry += tot[2];
        seg_in_rank = seg_carry + sc[3];
        seg_carry += tot[3];
      }
      if (valid) {
        int si = seg_base + seg_in_rank;
        if (si + segs_b > total_segs) {
          set_status(status, CPATTN_ERR_INVALID_ARG);
        } else if (strategy == CP_ZIGZAG) {
          if (e > 0) {
            segs[si++] = cp_segment_t{row_base + row_in_rank, e, p + st_e, 1, kv0,
                                      p + st_e + e, flat0 + st_e, b};
          }
          if (l > 0) {
            segs[si] = cp_segment_t{row_base + row_in_rank + e, l, p + st_l, 1, kv0,
                                    p + st_l + l, flat0 + st_l, b};
          }
        } else if (e > 0) {
          const int last = i0 + (e - 1) * C;
          segs[si] = cp_segment_t{row_base + (i0 - r) / C, e, p + (i0 - flat0), C, kv0,
                                  p + (last - flat0) + 1, i0, b};
        }
      }
    }
    row_base += row_carry;
    seg_base += seg_carry;
  }
  if (threadIdx.x == 0) {
    row_offsets[C] = row_base;
    seg_offsets[C] = seg_base;
    if (row_base != total_rows || seg_base != total_segs) set_status(status, CPATTN_ERR_INVALID_ARG);
  }
}

// Kernel 2: per cat row, find its segment and fill the index arrays.
__global__ void plan_rows_kernel(const cp_segment_t* __restrict__ segs, int total_segs,
                                 int total_rows, int32_t* __restrict__ gather_idx,
                                 int32_t* __restrict__ positions, int32_t* __restrict__ restore_idx,
                                 int32_t* status) {
  grid_dep_wait();  // the segment kernel before this launch wrote segs
  grid_dep_trigger();
  for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < total_rows;
       row += gridDim.x * blockDim.x) {
    int lo = 0, hi = total_segs;  // last segment with q_row0 <= row
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (segs[mid].q_row0 <= row) lo = mid; else hi = mid;
    }
    if (total_segs <= 0) { set_status(status, CPATTN_ERR_INVALID_ARG); return; }
    const cp_segment_t s = segs[lo];
    const int i = row - s.q_row0;
    if (i < 0 || i >= s.q_len) { set_status(status, CPATTN_ERR_INVALID_ARG); continue; }
    const int tok = s.tok0 + i * s.q_pos_step;
    if (tok < 0 || tok >= total_rows) { set_status(status, CPATTN_ERR_INVALID_ARG); continue; }
    gather_idx[row] = tok;
    positions[row] = s.q_pos0 + i * s.q_pos_step;
    restore_idx[tok] = row;
  }
}

constexpr int kTileBins = 4096;

// Kernel 3: list of 128-row query tiles, heaviest first (counting sort on the
// number of 128-key tiles visible to the tile's last row).
__global__ void __launch_bounds__(kPlanThreads)
plan_tiles_kernel(const cp_segment_t* __restrict__ segs, int total_segs, int total_tiles,
                  int32_t* __restrict__ tiles, int32_t* status) {
  grid_dep_wait();  // the kernels before this launch wrote segs
  __shared__ int hist[kTileBins];
  __shared__ int scan_buf[33];
  for (int i = threadIdx.x; i < kTileBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  int ntiles = 0;
  for (int s = threadIdx.x; s < total_segs; s += blockDim.x) {
    const cp_segment_t sg = segs[s];
    const int nt = (sg.q_len + CPATTN_TILE_ROWS - 1) / CPATTN_TILE_ROWS;
    ntiles += nt;
    for (int t = 0; t < nt; ++t) {
      const int last = min(sg.q_len, (t + 1) * CPATTN_TILE_ROWS) - 1;
      const long long keys = (long long)sg.q_pos0 + (long long)last * sg.q_pos_step + 1;
      const int key = (int)min((keys + CPATTN_TILE_ROWS - 1) / CPATTN_TILE_ROWS,
                               (long long)kTileBins - 1);
      atomicAdd(&hist[kTileBins - 1 - key], 1);  // bin 0 = heaviest
    }
  }
  int total;
  block_excl_scan(ntiles, scan_buf, &total);
  if (total != total_tiles) {
    if (threadIdx.x == 0) set_status(status, CPATTN_ERR_INVALID_ARG);
    return;
  }
  // exclusive scan of the histogram, 4 bins per thread
  int local[4], sum = 0;
  for (int j = 0; j < 4; ++j) { local[j] = hist[threadIdx.x * 4 + j]; sum += local[j]; }
  int tot2;
  int off = block_excl_scan(sum, scan_buf, &tot2);
  __syncthreads();
  for (int j = 0; j < 4; ++j) { hist[threadIdx.x * 4 + j] = off; off += local[j]; }
  __syncthreads();
  for (int s = threadIdx.x; s < total_segs; s += blockDim.x) {
    const cp_segment_t sg = segs[s];
    const int nt = (sg.q_len + CPATTN_TILE_ROWS - 1) / CPATTN_TILE_ROWS;
    for (int t = 0; t < nt; ++t) {
      const int last = min(sg.q_len, (t + 1) * CPATTN_TILE_ROWS) - 1;
      const long long keys = (long long)sg.q_pos0 + (long long)last * sg.q_pos_step + 1;
      const int key = (int)min((keys + CPATTN_TILE_ROWS - 1) / CPATTN_TILE_ROWS,
                               (long long)kTileBins - 1);
      const int dst = atomicAdd(&hist[kTileBins - 1 - key], 1);
      tiles[2 * dst] = s;
      tiles[2 * dst + 1] = t;
    }
  }
}

static_assert(kTileBins == 4 * kPlanThreads, "histogram scan assumes 4 bins per thread");

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" int cp_shard_plan_sizes(const int32_t* new_lens, const int32_t* prefix_lens,
                                   int num_reqs, int cp_size, int strategy,
                                   int32_t* rows_per_rank, int32_t* segs_per_rank,
                                   int32_t* tiles_per_rank) {
  if (num_reqs < 0 || num_reqs > CPATTN_MAX_REQS) return CPATTN_ERR_INVALID_ARG;
  if (cp_size < 1 || cp_size > CPATTN_MAX_CP) return CPATTN_ERR_INVALID_ARG;
  if (strategy != CP_ZIGZAG && strategy != CP_INTERLEAVE) return CPATTN_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!new_lens || !prefix_lens)) return CPATTN_ERR_INVALID_ARG;
  const int C = cp_size;
  std::vector<long long> rows(C, 0), segs(C, 0), tiles(C, 0);
  long long flat0 = 0, kv = 0;
  auto ntile = [](long long x) { return (x + CPATTN_TILE_ROWS - 1) / CPATTN_TILE_ROWS; };
  for (int b = 0; b < num_reqs; ++b) {
    const long long n = new_lens[b], p = prefix_lens[b];
    if (n < 0 || p < 0) return CPATTN_ERR_INVALID_ARG;
    if (strategy == CP_ZIGZAG) {
      const long long nb = 2LL * C, base = n / nb, rem = n % nb;
      for (int r = 0; r < C; ++r) {
        const long long e = base + (r < rem), l = base + ((nb - 1 - r) < rem);
        rows[r] += e + l;
        segs[r] += (e > 0) + (l > 0);
        tiles[r] += ntile(e) + ntile(l);
      }
    } else {
      for (int r = 0; r < C; ++r) {
        const long long i0 = flat0 + (((r - flat0 % C) % C) + C) % C;
        const long long cnt = (i0 < flat0 + n) ? (flat0 + n - 1 - i0) / C + 1 : 0;
        rows[r] += cnt;
        segs[r] += cnt > 0;
        tiles[r] += ntile(cnt);
      }
    }
    flat0 += n;
    kv += n + p;
  }
  long long tr = 0, ts = 0, tt = 0;
  for (int r = 0; r < C; ++r) { tr += rows[r]; ts += segs[r]; tt += tiles[r]; }
  if (tr >= (1LL << 31) || kv >= (1LL << 31) || ts >= (1LL << 31) || tt >= (1LL << 31))
    return CPATTN_ERR_INVALID_ARG;
  for (int r = 0; r < C; ++r) {
    if (rows_per_rank) rows_per_rank[r] = (int32_t)rows[r];
    if (segs_per_rank) segs_per_rank[r] = (int32_t)segs[r];
    if (tiles_per_rank) tiles_per_rank[r] = (int32_t)tiles[r];
  }
  return CPATTN_OK;
}

static bool misaligned(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u); }

extern "C" int cp_shard_plan(const int32_t* new_lens_dev, const int32_t* prefix_lens_dev,
                             int num_reqs, int cp_size, int strategy, int total_rows,
                             int total_segs, int total_tiles, cp_segment_t* segs_dev,
                             int32_t* seg_offsets_dev, int32_t* row_offsets_dev,
                             int32_t* gather_idx_dev, int32_t* positions_dev,
                             int32_t* restore_idx_dev, int32_t* tiles_dev, int32_t* status_dev,
                             cudaStream_t stream) {
  CPATTN_TRACE("cp_shard_plan");
  if (num_reqs < 0 || num_reqs > CPATTN_MAX_REQS) return CPATTN_ERR_INVALID_ARG;
  if (cp_size < 1 || cp_size > CPATTN_MAX_CP) return CPATTN_ERR_INVALID_ARG;
  if (strategy != CP_ZIGZAG && strategy != CP_INTERLEAVE) return CPATTN_ERR_INVALID_ARG;
  if (total_rows < 0 || total_segs < 0 || total_tiles < 0) return CPATTN_ERR_INVALID_ARG;
  if (!seg_offsets_dev || !row_offsets_dev) return CPATTN_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!new_lens_dev || !prefix_lens_dev)) return CPATTN_ERR_INVALID_ARG;
  if (total_segs > 0 && !segs_dev) return CPATTN_ERR_INVALID_ARG;
  if (total_rows > 0 && (!gather_idx_dev || !positions_dev || !restore_idx_dev))
    return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(segs_dev) & 15u) return CPATTN_ERR_ALIGNMENT;
  if (misaligned(new_lens_dev) || misaligned(prefix_lens_dev) || misaligned(gather_idx_dev) ||
      misaligned(positions_dev) || misaligned(restore_idx_dev) || misaligned(tiles_dev) ||
      misaligned(seg_offsets_dev) || misaligned(row_offsets_dev) || misaligned(status_dev))
    return CPATTN_ERR_ALIGNMENT;
  // one warp per 32 requests (at least one, at most the 1024-thread block)
  const int seg_threads = std::min(kPlanThreads, std::max(32, (num_reqs + 31) / 32 * 32));
  plan_segments_kernel<<<1, seg_threads, 0, stream>>>(new_lens_dev, prefix_lens_dev, num_reqs,
                                                      cp_size, strategy, total_rows, total_segs,
                                                      segs_dev, seg_offsets_dev, row_offsets_dev,
                                                      status_dev);
  if (cudaGetLastError() != cudaSuccess) return CPATTN_ERR_CUDA;
  // the row and tile kernels are launched to overlap the kernel before them
  // and wait for it before their first read (programmatic dependent launch)
  if (total_rows > 0 && total_segs > 0) {
    const int threads = 256;
    const int blocks = (int)std::min<long long>(((long long)total_rows + threads - 1) / threads, 4096);
    const cp_segment_t* segs_c = segs_dev;
    if (launch_kernel(plan_rows_kernel, (unsigned)blocks, threads, 0, stream, true, segs_c,
                      total_segs, total_rows, gather_idx_dev, positions_dev, restore_idx_dev,
                      status_dev) != cudaSuccess)
      return CPATTN_ERR_CUDA;
  }
  if (tiles_dev && total_tiles > 0) {
    const cp_segment_t* segs_c = segs_dev;
    if (launch_kernel(plan_tiles_kernel, 1u, kPlanThreads, 0, stream, true, segs_c, total_segs,
                      total_tiles, tiles_dev, status_dev) != cudaSuccess)
      return CPATTN_ERR_CUDA;
  }
  return CPATTN_OK;
}
