// Shard partial attention, absorbed-MLA shape (sm_103a).
//
// Query and key rows are the 576-wide absorbed latent (512 latent + 64 rope
// columns) and the value is the latent itself, V = K[:, :512] (blog "什么是
// Context Parallelism", §4.2: CP for MLA gathers the compressed latent, and the
// absorbed form attends directly on it).  The semantics are those of
// cp_attn_partial: causal / windowed softmax attention per query row giving O
// and its log-sum-exp.
//
// Tensor memory holds 512 fp32 columns per SM, exactly a 128 x 512 output,
// so the output is split in two 256-column halves computed by sibling CTAs
// that each recompute S = Q K^T.  One CTA: 128 query rows of one head, one
// output half, keys in tiles of 64.
//   shared memory: Q tile 128 x 576 (9 swizzled 64-column chunks, 144 KB) and
//     one K tile 64 x 576 (9 chunks, 72 KB) with a barrier pair per chunk.  The
//     K tile also serves as V: the four chunks of this CTA's output half are
//     the B operand (MN-major) of P V.
//   tensor memory: S double-buffered (2 x 64 columns, P aliased as bf16) and
//     the 256-column O half.
//   order of the MMA thread for key tile j: Q K_j^T over the five chunks that
//     P V does not read (they were released as soon as S_{j-1} was done),
//     then P_{j-1} V_{j-1}, which frees the V chunks of tile j-1 for the
//     producer, then the rest of Q K_j^T on those chunks.  Softmax of tile
//     j-1 overlaps the first part.
#include <algorithm>
#include <cstdint>

#include "attn_common.cuh"

namespace cpattn {
namespace {

constexpr int kD = 576, kDV = 512, kDVH = 256, kBNm = 64, kChunks = kD / 64;
constexpr int kThreadsM = 192;  // 4 softmax warps, producer warp, MMA warp
constexpr int kQBytes = BM * kD * 2;          // 147456
constexpr int kKChunkBytes = kBNm * 128;      // 8192 (64 keys x 64 bf16)
constexpr int kKOffM = kQBytes;
constexpr int kBarOffM = kKOffM + kChunks * kKChunkBytes;
constexpr int kNumBarsM = 1 + 2 * kChunks + 2 + 2 + 1 + 1;
constexpr int kSmemM = kBarOffM + kNumBarsM * 8 + 16 + 1024;
static_assert(kSmemM <= 232448, "MLA tile exceeds shared memory");

__global__ void __launch_bounds__(kThreadsM, 1)
attn_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffM);
  uint64_t* bar_q = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kChunks;
  uint64_t* s_full = k_empty + kChunks;  // [2]
  uint64_t* p_full = s_full + 2;         // [2]
  uint64_t* o_full = p_full + 2;
  uint64_t* bar_drain = o_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBarsM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work item: (128-row tile, query head, output half) ----
  const int half = blockIdx.x & 1;
  const int h = (blockIdx.x >> 1) % p.Hq;
  const int rest = (blockIdx.x >> 1) / p.Hq;
  const int jblk = p.split_block > 0 ? rest % p.max_blocks : 0;
  const int tile_idx = p.split_block > 0 ? rest / p.max_blocks : rest;
  cp_segment_t sg;
  int t, seg_id, kv_lo, kv_hi;
  long long out_row0;
  if (!resolve_tile(p, tile_idx, sg, t, seg_id)) return;
  if (!split_window(p, sg, seg_id, jblk, kv_lo, kv_hi, out_row0)) return;
  const int r0 = t * BM;
  const int rows_valid = min(BM, sg.q_len - r0);
  const int pos_max = sg.q_pos0 + (r0 + rows_valid - 1) * sg.q_pos_step;
  const int win_lo = max(kv_lo, 0);
  const int win_hi_tile = kv_hi < 0 ? pos_max + 1 : min(kv_hi, pos_max + 1);
  const int j0 = win_lo / kBNm;
  const int n_kv = win_hi_tile > win_lo ? (win_hi_tile + kBNm - 1) / kBNm - j0 : 0;
  const int kv_head = h / p.g;
  // chunk order: the five chunks P V does not read, then this half's V chunks
  int order[kChunks];
  {
    int n = 0;
    for (int c = 0; c < kChunks; ++c)
      if (c < 4 * half || c >= 4 * half + 4) order[n++] = c;
    for (int c = 4 * half; c < 4 * half + 4; ++c) order[n++] = c;
  }
  constexpr int kNonV = kChunks - 4;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int c = 0; c < kChunks; ++c) {
      mbar_init(k_full + c, 1);
      mbar_init(k_empty + c, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full + b, 1);
      mbar_init(p_full + b, 128);
    }
    mbar_init(o_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    tmem_slot[2] = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // producer's issued chunk-load count, kept in shared memory for the abort drain
  volatile int* issued_ctr = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const uint32_t q_base = smem_u32(smem);
  const uint32_t k_base = smem_u32(smem + kKOffM);
  constexpr uint32_t kOCol = 256;

  if (warp == 4) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_kv > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      int issued = 0;
      if (!p.withhold_q) {
        mbar_arrive_expect_tx(bar_q, kQBytes);
        for (int c = 0; c < kChunks; ++c)
          tma_load_3d(smem + c * (BM * 128), &tm_q, bar_q, c * 64, h, sg.q_row0 + r0);
      }
      bool ok = true;
      for (int it = 0; it < n_kv && ok; ++it) {
        const int kv_row = sg.kv_row0 + (j0 + it) * kBNm;
        for (int i = 0; i < kChunks; ++i) {
          const int c = order[i];
          ok = mbar_wait(k_empty + c, (it & 1) ^ 1, abort_flag, p.timeout_ns);
          if (!ok) break;
          mbar_arrive_expect_tx(k_full + c, kKChunkBytes);
          tma_load_3d(smem + kKOffM + c * kKChunkBytes, &tm_k, k_full + c, c * 64, kv_head, kv_row);
          ++issued;
        }
      }
      *issued_ctr = issued;
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, kBNm, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, kDVH, 0, 1);
      // descriptors built once; per MMA only a constant offset is added
      const uint64_t dq0 = smem_desc_sw128(q_base, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(k_base, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(k_base + 4 * half * kKChunkBytes, kKChunkBytes, 1024);
      auto qk_chunk = [&](int c, uint32_t s_col, bool first) {
        const uint64_t qd = dq0 + (uint64_t)((c * (BM * 128)) >> 4);
        const uint64_t kd = dk0 + (uint64_t)((c * kKChunkBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tmem_base + s_col, qd + (uint64_t)(kk * 2), kd + (uint64_t)(kk * 2), kIdescQK,
                 (first && kk == 0) ? 0u : 1u);
      };
      auto pv = [&](int j) {
        const uint32_t p_col = (j & 1) * kBNm;
#pragma unroll
        for (int kk = 0; kk < kBNm / 16; ++kk)
          mma_ts(tmem_base + kOCol, tmem_base + p_col + kk * 8,
                 dv0 + (uint64_t)(kk * ((16 * 128) >> 4)), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.timeout_ns);
      for (int j = 0; j < n_kv && ok; ++j) {
        const uint32_t s_col = (j & 1) * kBNm;
        for (int i = 0; i < kNonV && ok; ++i) {
          const int c = order[i];
          ok = mbar_wait(k_full + c, j & 1, abort_flag, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          qk_chunk(c, s_col, i == 0);
          mma_commit(k_empty + c);
        }
        if (!ok) break;
        if (j > 0) {
          ok = mbar_wait(p_full + ((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          pv(j - 1);
          for (int i = kNonV; i < kChunks; ++i) mma_commit(k_empty + order[i]);
        }
        for (int i = kNonV; i < kChunks && ok; ++i) {
          const int c = order[i];
          ok = mbar_wait(k_full + c, j & 1, abort_flag, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          qk_chunk(c, s_col, false);
        }
        if (!ok) break;
        mma_commit(s_full + (j & 1));
      }
      if (ok) {
        const int j = n_kv - 1;
        ok = mbar_wait(p_full + (j & 1), (j >> 1) & 1, abort_flag, p.timeout_ns);
        if (ok) {
          tc_fence_after();
          pv(j);
          mma_commit(o_full);
        }
      }
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      mma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------- softmax --
    const int row = warp * 32 + lane;
    const bool valid = row < rows_valid;
    const int pos = valid ? sg.q_pos0 + (r0 + row) * sg.q_pos_step : -1;
    const int row_hi = valid ? (kv_hi < 0 ? pos + 1 : min(kv_hi, pos + 1)) : 0;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f, m_use = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = mbar_wait_warp(s_full + b, (j >> 1) & 1, abort_flag, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      float x[kBNm];
      {
        uint32_t r[kBNm];
        tmem_ld32p(lane_addr + b * kBNm, r);
        tmem_ld32p(lane_addr + b * kBNm + 32, r + 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kBNm; ++c) x[c] = __uint_as_float(r[c]);
      }
      const int key0 = (j0 + j) * kBNm;
      if (key0 < win_lo || key0 + kBNm > row_hi) {
#pragma unroll
        for (int c = 0; c < kBNm; ++c) {
          const int key = key0 + c;
          if (key < win_lo || key >= row_hi) x[c] = -INFINITY;
        }
      }
      float mx0 = x[0], mx1 = x[1];
#pragma unroll
      for (int c = 2; c < kBNm; c += 4) {
        mx0 = fmax3(mx0, x[c], x[c + 1]);
        mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
      }
      const float mx = fmaxf(mx0, mx1) * sl2;
      const bool move = mx > m_run + kMaxSlack;
      const float m_new = move ? mx : m_run;
      const float m_new_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = move ? ex2_approx(m_run - m_new_use) : 1.f;
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int q = 0; q < kBNm / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float a, bb;
          ffma2(a, bb, x[q * 32 + c], x[q * 32 + c + 1], sl2, sl2, -m_new_use, -m_new_use);
          a = ex2_approx(a);
          bb = ex2_approx(bb);
          fadd2(sum0, sum1, sum0, sum1, a, bb);
          pk[c >> 1] = pack_bf16x2(a, bb);
        }
        tmem_st16(lane_addr + b * kBNm + q * 16, pk);
      }
      l_run = l_run * alpha + (sum0 + sum1);
      // P_{j-1} V_{j-1} has completed: S_j was committed after it was issued
      const bool need = (j > 0) && move;
      if (__any_sync(0xffffffffu, need)) {
        const float a = need ? alpha : 1.f;
#pragma unroll 1
        for (int q = 0; q < kDVH / 32; ++q) {
          uint32_t r[32];
          tmem_ld32p(lane_addr + kOCol + q * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * a);
          tmem_st32(lane_addr + kOCol + q * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + b);
      m_run = m_new;
      m_use = m_new_use;
    }
    if (ok && n_kv > 0) ok = mbar_wait_warp(o_full, 0, abort_flag, p.timeout_ns);
    if (!ok) {
      if (lane == 0) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      tc_fence_after();
      const long long out_row = out_row0 + r0 + row;
      const bool has = l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
#pragma unroll 1
      for (int q = 0; q < kDVH / 32; ++q) {
        uint32_t r[32];
        if (n_kv > 0) {
          tmem_ld32p(lane_addr + kOCol + q * 32, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
        }
        if (valid) {
          const long long off = (out_row * p.Hq + h) * kDV + half * kDVH + q * 32;
          if (p.o_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + off);
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_float4(__uint_as_float(r[4 * c]) * inv, __uint_as_float(r[4 * c + 1]) * inv,
                                   __uint_as_float(r[4 * c + 2]) * inv,
                                   __uint_as_float(r[4 * c + 3]) * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + off);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(
                  pack_bf16x2(__uint_as_float(r[8 * c]) * inv, __uint_as_float(r[8 * c + 1]) * inv),
                  pack_bf16x2(__uint_as_float(r[8 * c + 2]) * inv, __uint_as_float(r[8 * c + 3]) * inv),
                  pack_bf16x2(__uint_as_float(r[8 * c + 4]) * inv, __uint_as_float(r[8 * c + 5]) * inv),
                  pack_bf16x2(__uint_as_float(r[8 * c + 6]) * inv, __uint_as_float(r[8 * c + 7]) * inv));
          }
        }
      }
      if (valid && half == 0)
        p.lse[out_row * p.Hq + h] = has ? (m_use + lg2_approx(l_run)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    if (lane == 0 && *abort_flag && n_kv > 0) {
      // after an abort, let this CTA's own copies land before its shared
      // memory is released: Q, and the last load of every chunk
      const int issued = *issued_ctr;
      if (!p.withhold_q) mbar_wait(bar_q, 0, nullptr, p.timeout_ns);
      const int it_last = (issued - 1) / kChunks;
      for (int i = 0; i < kChunks && issued > 0; ++i) {
        const int c = order[i];
        const int it_c = (i < issued - it_last * kChunks) ? it_last : it_last - 1;
        if (it_c >= 0) mbar_wait(k_full + c, it_c & 1, nullptr, p.timeout_ns);
      }
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

int launch_attn_mla(const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                    int64_t k_head_stride, int num_kv_rows, int Hkv, AttnParams prm,
                    long long tiles, cudaStream_t stream) {
  CUtensorMap mq, mk;
  if (!make_map(&mq, q, kD, prm.Hq, num_q_rows, kD, (long long)prm.Hq * kD) ||
      !make_map(&mk, k, kD, Hkv, num_kv_rows, k_head_stride, k_row_stride, kBNm))
    return CPATTN_ERR_CUDA;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(attn_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemM) != cudaSuccess)
      return CPATTN_ERR_CUDA;
    configured = true;
  }
  const long long grid = tiles * prm.Hq * 2;  // tiles x KV blocks (split mode) x heads x halves
  if (grid <= 0) return CPATTN_OK;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_INVALID_ARG;
  attn_mla_kernel<<<(unsigned)grid, kThreadsM, kSmemM, stream>>>(mq, mk, prm);
  return cudaGetLastError() == cudaSuccess ? CPATTN_OK : CPATTN_ERR_CUDA;
}

}  // namespace cpattn
