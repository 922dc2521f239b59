// LSE merge of partial attention results and the restore (row gather).
//
// Merge (blog "什么是 Context Parallelism", §3.6, the shared component of
// pass-KV and pass-Q): partial j carries a normalised output O_j and its
// log-sum-exp L_j; with m = max_j L_j and w_j = exp(L_j - m) the exact result
// is L = m + ln(sum_j w_j) and O = sum_j w_j O_j / sum_j w_j.
// Restore (same blog, §2.1): a restore index puts the all-gathered shard rows
// back into causal token order.
//
// Both are HBM-bound streams: a warp merges one (row, head) unit per step
// (or, with at most 8 partials, 16 / n units so that every lane still has 16
// loads in flight), with groups of 16-byte partial loads issued before any
// use; the gather is a flat grid-stride 16-byte copy.
#include <algorithm>
#include <cstdint>

#include <cuda_bf16.h>

#include "../../include/cpattn.h"
#include "ptx.cuh"
#include "trace.h"

namespace cpattn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kMaxParts = 32;

__device__ __forceinline__ float4 ld_stream(const float* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// Each warp merges one (row, head) unit per iteration; lane j < num_parts
// holds L_j.  dv is split in 128-float chunks, one float4 per lane, and the
// partials are streamed in groups of kGroup 16-byte loads that are all issued
// before any is used (the first group together with the L_j load).  Two
// 256-thread blocks share an SM: 16 warps, about 128 KB of loads in flight.
constexpr int kGroup = 16;

template <bool OUT_F32>
__global__ void __launch_bounds__(kMergeThreads, 2)
lse_merge_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                 int num_parts, int64_t o_stride, int64_t l_stride, int rows, int Hq, int dv,
                 const int32_t* __restrict__ dst_rows, void* __restrict__ o_out,
                 float* __restrict__ lse_out, int num_out_rows, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long units = (long long)rows * Hq;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long u = warp0; u < units; u += nwarps) {
    const int row = (int)(u / Hq), h = (int)(u % Hq);
    int out_row = row;
    if (dst_rows) {
      out_row = __ldg(dst_rows + row);
      if (out_row < 0 || out_row >= num_out_rows) {
        if (lane == 0) set_status(status, CPATTN_ERR_RANGE);
        continue;
      }
    }
    const float* base = o_parts + u * dv;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    // issue the L_j load and the first group of partial loads together, so a
    // unit with up to kGroup partials costs one memory round trip
    float lj = -INFINITY;
    if (lane < num_parts) lj = __ldg(lse_parts + lane * l_stride + u);
    float4 v[kGroup];
    {
      const int c = lane * 4;
      const bool act = c < dv;
#pragma unroll
      for (int jj = 0; jj < kGroup; ++jj)
        v[jj] = (act && jj < num_parts) ? ld_stream(base + jj * o_stride + c) : zero;
    }
    float m = lj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const bool empty = (m == -INFINITY);
    const float wj = (lane < num_parts && !empty) ? __expf(lj - m) : 0.f;
    float ws = wj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    const float inv = empty ? 0.f : 1.f / ws;
    // every lane runs the same number of chunks and groups so that the weight
    // shuffles always see the full warp; lanes past dv load and store nothing
    for (int c0 = 0; c0 < dv; c0 += 128) {
      const int c = c0 + lane * 4;
      const bool act = c < dv;
      float4 acc = zero;
      for (int j0 = 0; j0 < num_parts; j0 += kGroup) {
        if (c0 > 0 || j0 > 0) {
#pragma unroll
          for (int jj = 0; jj < kGroup; ++jj)
            v[jj] = (act && j0 + jj < num_parts) ? ld_stream(base + (j0 + jj) * o_stride + c)
                                                 : zero;
        }
#pragma unroll
        for (int jj = 0; jj < kGroup; ++jj) {
          const float w = __shfl_sync(0xffffffffu, wj, (j0 + jj) & 31);
          acc.x = fmaf(w, v[jj].x, acc.x);
          acc.y = fmaf(w, v[jj].y, acc.y);
          acc.z = fmaf(w, v[jj].z, acc.z);
          acc.w = fmaf(w, v[jj].w, acc.w);
        }
      }
      if (!act) continue;
      acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      const long long oo = ((long long)out_row * Hq + h) * dv + c;
      if (OUT_F32) {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(o_out) + oo), acc);
      } else {
        uint2 pk;
        pk.x = pack_bf16x2(acc.x, acc.y);
        pk.y = pack_bf16x2(acc.z, acc.w);
        __stcs(reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o_out) + oo), pk);
      }
    }
    if (lse_out && lane == 0)
      lse_out[(long long)out_row * Hq + h] = empty ? -INFINITY : m + __logf(ws);
  }
}

// Few partials (NP <= 8): a warp step merges U = 16 / NP consecutive units so that
// every lane still has about 16 partial loads in flight.  Lane L < U*NP owns
// L_j of (unit L / NP, part L % NP); weights are normalised in the owning lane
// and broadcast by shuffles.
template <bool OUT_F32, int NP>
__global__ void __launch_bounds__(kMergeThreads, 2)
lse_merge_batched_kernel(const float* __restrict__ o_parts, const float* __restrict__ lse_parts,
                         int64_t o_stride, int64_t l_stride, int rows, int Hq, int dv,
                         const int32_t* __restrict__ dst_rows, void* __restrict__ o_out,
                         float* __restrict__ lse_out, int num_out_rows, int32_t* status) {
  constexpr int U = kGroup / NP;
  const int lane = threadIdx.x & 31;
  const long long units = (long long)rows * Hq;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const int ui_l = lane / NP, j_l = lane - ui_l * NP;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (long long ub = warp0 * U; ub < units; ub += nwarps * U) {
    // output unit (out row * Hq + head) of each unit of this step, -1 when out
    // of range or past the end (the host keeps num_out_rows * Hq < 2^31 here)
    int orow[U];
#pragma unroll
    for (int ui = 0; ui < U; ++ui) {
      const long long u = ub + ui;
      int r = -1;
      if (u < units) {
        const int row = (int)(u / Hq), h = (int)(u % Hq);
        const int dr = dst_rows ? __ldg(dst_rows + row) : row;
        if (dr >= 0 && dr < num_out_rows) r = dr * Hq + h;
        else if (lane == 0) set_status(status, CPATTN_ERR_RANGE);
      }
      orow[ui] = r;
    }
    const long long u_l = ub + ui_l;
    float lj = -INFINITY;
    if (lane < U * NP && u_l < units) lj = __ldg(lse_parts + j_l * l_stride + u_l);
    float v4[U * NP][4];
    for (int c0 = 0; c0 < dv; c0 += 128) {
      const int c = c0 + lane * 4;
      const bool act = c < dv;
#pragma unroll
      for (int sl = 0; sl < U * NP; ++sl) {
        const int ui = sl / NP, j = sl - ui * NP;
        const float4 v = (act && orow[ui] >= 0)
                             ? ld_stream(o_parts + j * o_stride + (ub + ui) * dv + c)
                             : zero;
        v4[sl][0] = v.x; v4[sl][1] = v.y; v4[sl][2] = v.z; v4[sl][3] = v.w;
      }
      if (c0 == 0) {
        // per-unit max and normalised weight of the owned (unit, part)
        float m = -INFINITY;
#pragma unroll
        for (int j = 0; j < NP; ++j)
          m = fmaxf(m, __shfl_sync(0xffffffffu, lj, (ui_l * NP + j) & 31));
        const bool empty = (m == -INFINITY);
        const float w = empty ? 0.f : __expf(lj - m);
        float sw = 0.f;
#pragma unroll
        for (int j = 0; j < NP; ++j) sw += __shfl_sync(0xffffffffu, w, (ui_l * NP + j) & 31);
        lj = empty ? 0.f : w / sw;  // lj now holds the normalised weight
        if (lse_out && lane < U * NP && j_l == 0 && u_l < units) {
          int r = -1;
#pragma unroll
          for (int ui = 0; ui < U; ++ui)
            if (ui == ui_l) r = orow[ui];
          if (r >= 0) lse_out[r] = empty ? -INFINITY : m + __logf(sw);
        }
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
        if (!act || orow[ui] < 0) continue;
        const long long oo = (long long)orow[ui] * dv + c;
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

// dst[i] = src[idx[i]]: vector chunks of type V (16 or 4 bytes), consecutive
// threads on consecutive chunks of the same row.
template <typename V>
__global__ void __launch_bounds__(256)
row_gather_kernel(const V* __restrict__ src, int num_src_rows, const int32_t* __restrict__ idx,
                  int rows, long long chunks_per_row, V* __restrict__ dst, int32_t* status) {
  const long long total = (long long)rows * chunks_per_row;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    const long long row = e / chunks_per_row, col = e - row * chunks_per_row;
    const int s = __ldg(idx + row);
    if (s < 0 || s >= num_src_rows) {
      if (col == 0) set_status(status, CPATTN_ERR_RANGE);
      continue;
    }
    const V v = __ldcs(src + (long long)s * chunks_per_row + col);
    __stcs(dst + e, v);
  }
}

// SM count of the current device, cached per device.
int sm_count() {
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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace cpattn

using namespace cpattn;

extern "C" int cp_lse_merge(const float* o_parts, const float* lse_parts, int num_parts,
                            int64_t o_part_stride, int64_t lse_part_stride, int rows, int Hq,
                            int dv, const int32_t* dst_rows, void* o_out, int o_out_is_fp32,
                            float* lse_out, int num_out_rows, int32_t* status_dev,
                            cudaStream_t stream) {
  CPATTN_TRACE("cp_lse_merge");
  if (num_parts < 1 || num_parts > kMaxParts) return CPATTN_ERR_INVALID_ARG;
  if (rows < 0 || Hq < 1 || dv < 4 || dv > 1024 || (dv % 4) != 0) return CPATTN_ERR_INVALID_ARG;
  if (num_out_rows < 0 || (!dst_rows && num_out_rows < rows)) return CPATTN_ERR_INVALID_ARG;
  if (rows == 0) return CPATTN_OK;
  if (!o_parts || !lse_parts || !o_out) return CPATTN_ERR_INVALID_ARG;
  if (num_parts > 1 && (o_part_stride < (int64_t)rows * Hq * dv ||
                        lse_part_stride < (int64_t)rows * Hq))
    return CPATTN_ERR_INVALID_ARG;
  if (!aligned16(o_parts) || !aligned16(o_out) || (o_part_stride % 4) != 0 ||
      (reinterpret_cast<uintptr_t>(lse_parts) & 3u) || (reinterpret_cast<uintptr_t>(lse_out) & 3u))
    return CPATTN_ERR_ALIGNMENT;
  const long long units = (long long)rows * Hq;
  const long long want = (units + (kMergeThreads / 32) - 1) / (kMergeThreads / 32);
  const int grid = (int)std::min<long long>(want, (long long)sm_count() * 2 * 8);
  if (num_parts <= kGroup / 2 && (long long)num_out_rows * Hq < (1LL << 31) &&
      (long long)rows * Hq < (1LL << 31)) {
#define CPATTN_BATCHED(NPV)                                                                      \
  case NPV:                                                                                      \
    if (o_out_is_fp32)                                                                           \
      lse_merge_batched_kernel<true, NPV><<<grid, kMergeThreads, 0, stream>>>(                   \
          o_parts, lse_parts, o_part_stride, lse_part_stride, rows, Hq, dv, dst_rows, o_out,     \
          lse_out, num_out_rows, status_dev);                                                    \
    else                                                                                         \
      lse_merge_batched_kernel<false, NPV><<<grid, kMergeThreads, 0, stream>>>(                  \
          o_parts, lse_parts, o_part_stride, lse_part_stride, rows, Hq, dv, dst_rows, o_out,     \
          lse_out, num_out_rows, status_dev);                                                    \
    break;
    switch (num_parts) {
      CPATTN_BATCHED(1) CPATTN_BATCHED(2) CPATTN_BATCHED(3) CPATTN_BATCHED(4)
      CPATTN_BATCHED(5) CPATTN_BATCHED(6) CPATTN_BATCHED(7) CPATTN_BATCHED(8)
      default: break;
    }
#undef CPATTN_BATCHED
  } else if (o_out_is_fp32) {
    lse_merge_kernel<true><<<grid, kMergeThreads, 0, stream>>>(
        o_parts, lse_parts, num_parts, o_part_stride, lse_part_stride, rows, Hq, dv, dst_rows,
        o_out, lse_out, num_out_rows, status_dev);
  } else {
    lse_merge_kernel<false><<<grid, kMergeThreads, 0, stream>>>(
        o_parts, lse_parts, num_parts, o_part_stride, lse_part_stride, rows, Hq, dv, dst_rows,
        o_out, lse_out, num_out_rows, status_dev);
  }
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

extern "C" int cp_restore(const void* src, int num_src_rows, const int32_t* idx_dev, int rows,
                          int64_t row_bytes, void* dst, int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_restore");
  if (rows < 0 || num_src_rows < 0 || row_bytes <= 0 || (row_bytes % 4) != 0)
    return CPATTN_ERR_INVALID_ARG;
  if (rows == 0) return CPATTN_OK;
  if (!src || !dst || !idx_dev) return CPATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 3u) || (reinterpret_cast<uintptr_t>(dst) & 3u) ||
      (reinterpret_cast<uintptr_t>(idx_dev) & 3u))
    return CPATTN_ERR_ALIGNMENT;
  const bool wide = (row_bytes % 16) == 0 && aligned16(src) && aligned16(dst);
  const long long cpr = wide ? row_bytes / 16 : row_bytes / 4;
  const long long total = (long long)rows * cpr;
  const int grid = (int)std::min<long long>((total + 255) / 256, (long long)sm_count() * 8);
  if (wide)
    row_gather_kernel<uint4><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src), num_src_rows,
                                                       idx_dev, rows, cpr,
                                                       static_cast<uint4*>(dst), status_dev);
  else
    row_gather_kernel<uint32_t><<<grid, 256, 0, stream>>>(
        static_cast<const uint32_t*>(src), num_src_rows, idx_dev, rows, cpr,
        static_cast<uint32_t*>(dst), status_dev);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

extern "C" const char* cp_status_string(int status) {
  switch (status) {
    case CPATTN_OK: return "ok";
    case CPATTN_ERR_INVALID_ARG: return "invalid argument";
    case CPATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case CPATTN_ERR_CUDA: return "CUDA error";
    case CPATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case CPATTN_ERR_ALIGNMENT: return "misaligned pointer or stride";
    case CPATTN_ERR_RANGE: return "index or segment out of range";
    case CPATTN_ERR_TOO_LARGE: return "problem needs more scratch than the static buffer";
    default: return "unknown status";
  }
}
