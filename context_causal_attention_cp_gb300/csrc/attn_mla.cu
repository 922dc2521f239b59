// Shard partial attention, absorbed-MLA shape (sm_103a).
//
// Query and key rows are the 576-wide absorbed latent (512 latent + 64 rope
// columns) and the value is the latent itself, V = K[:, :512] (blog "什么是
// Context Parallelism", §4.2: CP for MLA gathers the compressed latent, and the
// absorbed form attends directly on it).  The semantics are those of
// cp_attn_partial: causal / windowed softmax attention per query row giving O
// and its log-sum-exp.
//
// This single-SM kernel serves an odd number of query heads; with an even
// number the pair kernel of attn_mla2.cu runs instead (MMAs issued for two
// SMs at once over 128-key tiles).
//
// Tensor memory holds 512 fp32 columns per SM, exactly a 128 x 512 output,
// so the output is split in two 256-column halves computed by sibling CTAs
// that each recompute S = Q K^T.  One CTA: 128 query rows of one head, one
// output half, keys in tiles of 64.
//   tensor memory (512 columns): S double-buffered (2 x 64, P aliased as
//     bf16), query chunks 5..8 as the A operand of their Q K^T MMAs (4 x 32
//     columns of packed bf16) and the 256-column O half.
//   shared memory: query chunks 0..4 (5 x 16 KB) and K tiles of 64 x 576 in
//     two double-buffered rings of 64-column swizzled chunks: the four chunks
//     of this CTA's output half (the V ring; they double as V, the B operand
//     of P V, MN-major) and the other five (the non-V ring).
//   MMA order per tile j: Q K_j^T over the non-V chunks (their stage is
//     released right after), P_{j-1} V_{j-1} (releases the V stage of tile
//     j-1), then Q K_j^T over the V chunks, so a stage's reload has a whole
//     tile of MMAs to land.  A rescale of O (rare: lazy max) first waits for
//     the P V in flight (o_ready).
#include <algorithm>
#include <cstdint>

#include "attn_common.cuh"

namespace cpattn {
namespace {

constexpr int kD = 576, kDV = 512, kDVH = 256, kBNm = 64, kChunks = kD / 64;
constexpr int kQSmemChunks = 5;                       // query chunks 0..4 in shared memory
constexpr int kQTmemChunks = kChunks - kQSmemChunks;  // chunks 5..8 in tensor memory
constexpr int kThreadsM = 192;  // 4 softmax warps, producer warp, MMA warp
constexpr int kQChunkBytes = BM * 128;               // 16384
constexpr int kKChunkBytes = kBNm * 128;             // 8192 (64 keys x 64 bf16)
constexpr int kVChunks = 4, kNChunks = kChunks - kVChunks;  // per K tile: V part, non-V part
constexpr int kNOff = kQSmemChunks * kQChunkBytes;            // non-V ring: 2 x 5 chunks
constexpr int kVOff = kNOff + 2 * kNChunks * kKChunkBytes;    // V ring: 2 x 4 chunks
constexpr int kBarOffM = kVOff + 2 * kVChunks * kKChunkBytes;  // 229376
// bar_q, qt_full, n_full[2], n_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2],
// o_ready, o_full, drain
constexpr int kNumBarsM = 17;
constexpr int kSmemM = kBarOffM + kNumBarsM * 8 + 16 + 1024;
static_assert(kSmemM <= 232448, "MLA tile exceeds shared memory");
constexpr uint32_t kSCol = 0, kQtCol = 128, kOCol = 256;  // TMEM column map

// Chunk c of a K tile is one of output half HALF's four V chunks iff
// 4*HALF <= c < 4*HALF+4; the other five are the non-V chunks, numbered
// 0..4 in increasing c.  Both lists are compile-time so that every MMA of a
// tile is issued with immediate descriptor offsets.
template <int HALF>
__device__ __forceinline__ constexpr bool mla_is_v(int c) {
  return c >= kVChunks * HALF && c < kVChunks * (HALF + 1);
}
template <int HALF>
__device__ __forceinline__ constexpr int mla_n_slot(int c) {
  return c < kVChunks * HALF ? c : c - kVChunks;
}

// Q K^T over chunk C of the tile whose non-V / V chunks start at descriptors
// dn / dkv (this stage), into S at s_tm.
template <int HALF, int C>
__device__ __forceinline__ void mla_qk_chunk(uint32_t s_tm, uint32_t qt_base, uint64_t dq0,
                                             uint64_t dn, uint64_t dkv, bool first) {
  constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, kBNm, 0, 0);
  uint64_t kd;
  if constexpr (mla_is_v<HALF>(C))
    kd = dkv + (uint64_t)(((C - kVChunks * HALF) * kKChunkBytes) >> 4);
  else
    kd = dn + (uint64_t)((mla_n_slot<HALF>(C) * kKChunkBytes) >> 4);
  if constexpr (C < kQSmemChunks) {
    const uint64_t qd = dq0 + (uint64_t)((C * kQChunkBytes) >> 4);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ss(s_tm, qd + kk * 2, kd + kk * 2, kIdescQK, (first && kk == 0) ? 0u : 1u);
  } else {
    const uint32_t qt = qt_base + (C - kQSmemChunks) * 32;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      mma_ts(s_tm, qt + kk * 8, kd + kk * 2, kIdescQK, (first && kk == 0) ? 0u : 1u);
  }
}

// Q K^T over the non-V chunks (PART 0) or the V chunks (PART 1) of a tile.
template <int HALF, int PART, int C = 0>
__device__ __forceinline__ void mla_qk_part(uint32_t s_tm, uint32_t qt_base, uint64_t dq0,
                                            uint64_t dn, uint64_t dkv, bool first) {
  if constexpr (C < kChunks) {
    constexpr bool mine = (PART == 1) == mla_is_v<HALF>(C);
    if constexpr (mine) mla_qk_chunk<HALF, C>(s_tm, qt_base, dq0, dn, dkv, first);
    mla_qk_part<HALF, PART, C + 1>(s_tm, qt_base, dq0, dn, dkv, first && !mine);
  }
}

// The MMA issuer of one CTA (one thread).  Per tile j: Q K_j^T on the non-V
// chunks (their stage is released right after), then P_{j-1} V_{j-1} (frees
// the V chunks of tile j-1), then Q K_j^T on the V chunks; the V reload of a
// stage has a whole tile of MMAs to land.
template <int HALF>
__device__ __noinline__ void mla_mma_issue(const AttnParams& p, uint8_t* smem, uint32_t q_base,
                                           uint32_t tmem_base, int n_kv, uint64_t* bars,
                                           volatile int* abort_flag) {
  constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, kDVH, 0, 1);
  uint64_t* bar_q = bars;
  uint64_t* qt_full = bars + 1;
  uint64_t* n_full = bars + 2;
  uint64_t* n_empty = bars + 4;
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 8;
  uint64_t* s_full = bars + 10;
  uint64_t* p_full = bars + 12;
  uint64_t* o_ready = bars + 14;
  uint64_t* o_full = bars + 15;
  uint64_t* bar_drain = bars + 16;
  const uint64_t dq0 = smem_desc_sw128(q_base, 16, 1024);
  const uint64_t dn0 = smem_desc_sw128(smem_u32(smem + kNOff), 16, 1024);
  const uint64_t dkv0 = smem_desc_sw128(smem_u32(smem + kVOff), 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + kVOff), kKChunkBytes, 1024);
  constexpr uint64_t kNStage = (kNChunks * kKChunkBytes) >> 4;  // descriptor step per stage
  constexpr uint64_t kVStage = (kVChunks * kKChunkBytes) >> 4;
  const uint32_t qt_base = tmem_base + kQtCol;
  auto pv = [&](int j) {
    const uint32_t p_tm = tmem_base + kSCol + (j & 1) * kBNm;
    const uint64_t vd = dv0 + (j & 1) * kVStage;
#pragma unroll
    for (int kk = 0; kk < kBNm / 16; ++kk)
      mma_ts(tmem_base + kOCol, p_tm + kk * 8, vd + (uint64_t)(kk * ((16 * 128) >> 4)),
             kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
  };
  bool ok = mbar_wait(bar_q, 0, abort_flag, p.timeout_ns);
  if (ok) ok = mbar_wait(qt_full, 0, abort_flag, p.timeout_ns);
  for (int j = 0; j < n_kv && ok; ++j) {
    const int st = j & 1;
    const uint32_t s_tm = tmem_base + kSCol + st * kBNm;
    const uint64_t dn = dn0 + st * kNStage, dkv = dkv0 + st * kVStage;
    ok = mbar_wait(n_full + st, (j >> 1) & 1, abort_flag, p.timeout_ns);
    if (!ok) break;
    tc_fence_after();
    mla_qk_part<HALF, 0>(s_tm, qt_base, dq0, dn, dkv, true);
    mma_commit(n_empty + st);
    if (j > 0) {
      const int jp = j - 1;
      ok = mbar_wait(p_full + (jp & 1), (jp >> 1) & 1, abort_flag, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      pv(jp);
      mma_commit(o_ready);
      mma_commit(v_empty + (jp & 1));
    }
    ok = mbar_wait(v_full + st, (j >> 1) & 1, abort_flag, p.timeout_ns);
    if (!ok) break;
    tc_fence_after();
    mla_qk_part<HALF, 1>(s_tm, qt_base, dq0, dn, dkv, false);
    mma_commit(s_full + st);
  }
  if (ok) {
    const int jp = n_kv - 1;
    ok = mbar_wait(p_full + (jp & 1), (jp >> 1) & 1, abort_flag, p.timeout_ns);
    if (ok) {
      tc_fence_after();
      pv(jp);
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

__global__ void __launch_bounds__(kThreadsM, 1)
attn_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOffM);
  uint64_t* bar_q = bars;
  uint64_t* qt_full = bars + 1;
  uint64_t* n_full = bars + 2;    // [2] non-V chunks of a K tile
  uint64_t* n_empty = bars + 4;   // [2]
  uint64_t* v_full = bars + 6;    // [2] this half's V chunks of a K tile
  uint64_t* v_empty = bars + 8;   // [2]
  uint64_t* s_full = bars + 10;   // [2]
  uint64_t* p_full = bars + 12;   // [2]
  uint64_t* o_ready = bars + 14;
  uint64_t* o_full = bars + 15;
  uint64_t* bar_drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBarsM);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* issued_n = reinterpret_cast<volatile int*>(tmem_slot + 2);  // non-V loads issued
  volatile int* issued_v = reinterpret_cast<volatile int*>(tmem_slot + 3);  // V loads issued
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_trigger();  // a dependent merge may launch once every CTA is resident

  // ---- work item: (128-row tile [, KV block], query head, output half) ----
  const int half = blockIdx.x & 1;
  const int h = (blockIdx.x >> 1) % p.Hq;
  const int rest = (blockIdx.x >> 1) / p.Hq;
  const int jblk = p.split_block > 0 ? rest % p.max_blocks : 0;
  const int tile_idx = p.split_block > 0 ? rest / p.max_blocks : rest;
  cp_segment_t sg;
  int t, seg_id, kv_lo, kv_hi;
  long long out_row0;
  if (!resolve_tile(p, tile_idx, sg, t, seg_id) ||
      !split_window(p, sg, seg_id, jblk, kv_lo, kv_hi, out_row0)) {
    grid_dep_wait();  // no CTA ends before the kernel this launch may overlap
    return;
  }
  const int r0 = t * BM;
  const int rows_valid = min(BM, sg.q_len - r0);
  const int pos_max = sg.q_pos0 + (r0 + rows_valid - 1) * sg.q_pos_step;
  const int win_lo = max(kv_lo, 0);
  const int win_hi_tile = kv_hi < 0 ? pos_max + 1 : min(kv_hi, pos_max + 1);
  const int j0 = win_lo / kBNm;
  const int n_kv = win_hi_tile > win_lo ? (win_hi_tile + kBNm - 1) / kBNm - j0 : 0;
  const int kv_head = h / p.g;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(qt_full, 128);
    for (int st = 0; st < 2; ++st) {
      mbar_init(n_full + st, 1);
      mbar_init(n_empty + st, 1);
      mbar_init(v_full + st, 1);
      mbar_init(v_empty + st, 1);
      mbar_init(s_full + st, 1);
      mbar_init(p_full + st, 128);
    }
    mbar_init(o_ready, 1);
    mbar_init(o_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    tmem_slot[2] = 0;
    tmem_slot[3] = 0;
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
  const uint32_t q_base = smem_u32(smem);
  // chunk c of the K tile is a V chunk of this half iff 4*half <= c < 4*half+4;
  // non-V chunks are numbered 0..4 in increasing c
  auto is_v = [&](int c) { return c >= kVChunks * half && c < kVChunks * (half + 1); };
  auto n_slot = [&](int c) { return c < kVChunks * half ? c : c - kVChunks; };

  if (warp == 4) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_kv > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      if (!p.withhold_q) {
        mbar_arrive_expect_tx(bar_q, kQSmemChunks * kQChunkBytes);
        for (int c = 0; c < kQSmemChunks; ++c)
          tma_load_3d(smem + c * kQChunkBytes, &tm_q, bar_q, c * 64, h, sg.q_row0 + r0);
      }
      bool ok = true;
      int in = 0, iv = 0;  // loads issued per ring
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        const int kv_row = sg.kv_row0 + (j0 + j) * kBNm;
        ok = mbar_wait(n_empty + st, ((j >> 1) & 1) ^ 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        mbar_arrive_expect_tx(n_full + st, kNChunks * kKChunkBytes);
        for (int c = 0; c < kChunks; ++c)
          if (!is_v(c))
            tma_load_3d(smem + kNOff + (st * kNChunks + n_slot(c)) * kKChunkBytes, &tm_k,
                        n_full + st, c * 64, kv_head, kv_row);
        ++in;
        ok = mbar_wait(v_empty + st, ((j >> 1) & 1) ^ 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        mbar_arrive_expect_tx(v_full + st, kVChunks * kKChunkBytes);
        for (int c = kVChunks * half; c < kVChunks * (half + 1); ++c)
          tma_load_3d(smem + kVOff + (st * kVChunks + c - kVChunks * half) * kKChunkBytes, &tm_k,
                      v_full + st, c * 64, kv_head, kv_row);
        ++iv;
      }
      *issued_n = in;
      *issued_v = iv;
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_kv > 0) {
      if (half == 0)
        mla_mma_issue<0>(p, smem, q_base, tmem_base, n_kv, bars, abort_flag);
      else
        mla_mma_issue<1>(p, smem, q_base, tmem_base, n_kv, bars, abort_flag);
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
    if (n_kv > 0) {
      // query chunks 5..8 of this row into tensor memory (packed bf16 pairs,
      // the A-operand layout: row = lane, K along columns)
      const long long qrow = (long long)sg.q_row0 + r0 + row;
      const bool in_q = qrow < p.num_q_rows;
      const uint4* src = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(p.q) + (in_q ? qrow * p.Hq + h : 0) * kD);
#pragma unroll
      for (int c = 0; c < kQTmemChunks; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 w = in_q ? __ldg(src + (kQSmemChunks + c) * 8 + v) : make_uint4(0, 0, 0, 0);
          r[4 * v] = w.x;
          r[4 * v + 1] = w.y;
          r[4 * v + 2] = w.z;
          r[4 * v + 3] = w.w;
        }
        tmem_st32(lane_addr + kQtCol + c * 32, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qt_full);
    }
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = mbar_wait_warp(s_full + b, (j >> 1) & 1, abort_flag, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      float x[kBNm];
      {
        uint32_t r[kBNm];
        tmem_ld32p(lane_addr + kSCol + b * kBNm, r);
        tmem_ld32p(lane_addr + kSCol + b * kBNm + 32, r + 32);
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
      // O rescale (rare: lazy max): P V of tile j-1 may still be in flight,
      // so wait for it first (o_ready completes once per P V)
      const bool need = (j > 0) && move;
      if (__any_sync(0xffffffffu, need)) {
        ok = mbar_wait_warp(o_ready, (j - 1) & 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
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
        tmem_st16(lane_addr + kSCol + b * kBNm + q * 16, pk);
      }
      l_run = l_run * alpha + (sum0 + sum1);
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
      out_row0 = split_slot_row0(p, sg, seg_id, jblk, out_row0);
      const long long out_row = valid ? output_row(p, sg, r0, row, out_row0) : -1;
      const bool has = l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
      const bool acc_mode = p.lse_acc != nullptr;
      MergeCoef mc{0.f, inv, has ? (m_use + lg2_approx(l_run)) * kLn2 : -INFINITY};
      if (acc_mode && out_row >= 0)
        mc = merge_coef(__ldg(p.lse_acc + out_row * p.Hq + h), has, m_use, l_run);
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
        if (out_row >= 0) {
          const long long off = (out_row * p.Hq + h) * kDV + half * kDVH + q * 32;
          float v[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(r[c]) * mc.c_new;
          if (p.o_f32) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) + off);
            if (acc_mode) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const float4 a = dst[c];
                v[4 * c] += mc.c_old * a.x;
                v[4 * c + 1] += mc.c_old * a.y;
                v[4 * c + 2] += mc.c_old * a.z;
                v[4 * c + 3] += mc.c_old * a.w;
              }
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
              dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.o) + off);
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c] = make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]),
                                  pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                  pack_bf16x2(v[8 * c + 4], v[8 * c + 5]),
                                  pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
          }
        }
      }
      // both halves read lse_acc; only half 0 writes the LSE (the accumulate
      // entry point requires lse_acc and lse not to overlap)
      if (out_row >= 0 && half == 0) p.lse[out_row * p.Hq + h] = mc.lse;
    }
  }

  tc_fence_before();
  grid_dep_wait();  // (already returned in the epilogue unless this CTA aborted)
  __syncthreads();
  if (warp == 4) {
    if (lane == 0 && *abort_flag && n_kv > 0) {
      // after an abort, let this CTA's own copies land before its shared
      // memory is released: Q and the last load of each stage of both rings
      const int in = *issued_n, iv = *issued_v;
      if (!p.withhold_q) mbar_wait(bar_q, 0, nullptr, p.timeout_ns);
      for (int j = max(0, in - 2); j < in; ++j)
        mbar_wait(n_full + (j & 1), (j >> 1) & 1, nullptr, p.timeout_ns);
      for (int j = max(0, iv - 2); j < iv; ++j)
        mbar_wait(v_full + (j & 1), (j >> 1) & 1, nullptr, p.timeout_ns);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace

// The pair kernel (attn_mla2.cu) for an even number of query heads.
int launch_attn_mla_pair(const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                         int64_t k_head_stride, int num_kv_rows, int Hkv, AttnParams prm,
                         long long tiles, cudaStream_t stream);

int launch_attn_mla(const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                    int64_t k_head_stride, int num_kv_rows, int Hkv, AttnParams prm,
                    long long tiles, cudaStream_t stream) {
  if (prm.Hq % 2 == 0)
    return launch_attn_mla_pair(q, num_q_rows, k, k_row_stride, k_head_stride, num_kv_rows, Hkv,
                                prm, tiles, stream);
  CUtensorMap mq, mk;
  if (!make_map(&mq, q, kD, prm.Hq, num_q_rows, kD, (long long)prm.Hq * kD) ||
      !make_map(&mk, k, kD, Hkv, num_kv_rows, k_head_stride, k_row_stride, kBNm))
    return CPATTN_ERR_CUDA;
  prm.q = q;
  if (!allow_smem(attn_mla_kernel, kSmemM)) return CPATTN_ERR_CUDA;
  const long long grid = tiles * prm.Hq * 2;  // tiles x KV blocks (split mode) x heads x halves
  if (grid <= 0) return CPATTN_OK;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_INVALID_ARG;
  return launch_kernel(attn_mla_kernel, (unsigned)grid, kThreadsM, kSmemM, stream, prm.pdl != 0,
                       mq, mk, prm) == cudaSuccess
             ? CPATTN_OK
             : CPATTN_ERR_CUDA;
}

}  // namespace cpattn
