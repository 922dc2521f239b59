// Shard partial attention for prefill context parallelism on sm_103a.
//
// Computes, for every query row of every segment and every query head, the
// causal attention output O and its log-sum-exp L against the gathered KV
// (blog "什么是 Context Parallelism", §3.1/§3.3: each rank's queries against a
// KV block give a partial O_j with L_j; SGLang docs, "Prefill Context
// Parallelism", §Attention backend integration: the early and late zigzag
// blocks run with their own query and KV lengths, including any cached
// prefix).  One launch covers every segment of every shard.
//
// Design (one CTA = one 128-row query tile of one segment, for NQ query
// heads that share one KV head):
//   warp 4*NQ      TMA producer: Q tiles once, then K and V tiles of 128 keys
//                  through KST / VST-stage rings (128-byte swizzled boxes).
//   warp 4*NQ+1    MMA issuer (one thread): S_s = Q_s K^T into TMEM
//                  (tcgen05.mma, both operands from shared memory) and
//                  O_s += P_s V with P_s read from TMEM.  For NQ = 2 the two
//                  tiles ping-pong: while tile 0's softmax runs, the tensor
//                  core works on tile 1 and vice versa.
//   warps 0..4NQ-1 softmax, one warpgroup per query tile, one thread per row:
//                  tcgen05.ld of the S row, causal/window mask only on tiles
//                  that cross the diagonal or the window edge, online softmax
//                  in base 2, O rescale in TMEM when the row max grows, P
//                  written back to TMEM as bf16 (aliasing the S columns), and
//                  the epilogue (O / l, L = ln(sum)) straight to global memory.
// Every mbarrier wait is bounded; a wait that runs out sets
// CPATTN_ERR_TIMEOUT, the CTA drains its own in-flight work and frees TMEM.
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "attn_common.cuh"
#include "trace.h"

namespace cpattn {
namespace {

constexpr int BN = 128;  // keys per KV tile (MMA N of Q K^T)

template <int D, int DV, int NQ, int KST, int VST>
struct Cfg {
  // NQ = 2: two softmax warpgroups plus one warpgroup holding the producer and
  // MMA warps, so that setmaxnreg can move registers to the softmax warps
  // (168 x 384 at launch >= 104 x 128 + 200 x 256 after the split).
  static constexpr int kThreads = NQ == 2 ? 384 : NQ * 128 + 64;
  static constexpr bool kSplitRegs = NQ == 2;
  static constexpr int kRegsLaunch = 168, kRegsSoftmax = 200, kRegsOther = 104;
  static_assert(!kSplitRegs || kRegsOther * 128 + kRegsSoftmax * 256 <= kRegsLaunch * kThreads,
                "register split exceeds the launch allocation");
  static constexpr int kProducerWarp = NQ * 4;
  static constexpr int kMmaWarp = NQ * 4 + 1;
  static constexpr int kQTileBytes = BM * D * 2;
  static constexpr int kKTileBytes = BN * D * 2;
  static constexpr int kVTileBytes = BN * DV * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + NQ * kQTileBytes;
  static constexpr int kVOff = kKOff + KST * kKTileBytes;
  // epilogue staging: 32 rows x 128 bytes per softmax warp
  static constexpr int kStageOff = kVOff + VST * kVTileBytes;
  static constexpr int kStageBytes = 4 * NQ * 32 * 128;
  static constexpr int kBarOff = kStageOff + kStageBytes;
  static constexpr int kNumBars = 1 + 2 * KST + 2 * VST + 3 * NQ + 1;
  // barriers, then TMEM slot, abort flag and two issued-load counters
  static constexpr int kSmemBytes = kBarOff + kNumBars * 8 + 16 + 1024;  // + align slack
  static constexpr int kTmemNeed = NQ * (BN + DV);
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "TMEM budget");
  static_assert(D % 64 == 0 && DV % 64 == 0 && DV <= 256, "head dims");
};

// After an abort, let a CTA's own TMA copies land before its shared memory is
// released: the query load and the last `stages` loads of each ring (every
// wait is bounded).  Cold path, kept out of line.
__device__ __noinline__ void drain_after_abort(uint64_t* bar_q, bool q_issued, uint64_t* k_full,
                                               int kst, int k_issued, uint64_t* v_full, int vst,
                                               int v_issued, unsigned long long timeout) {
  if (q_issued) mbar_wait(bar_q, 0, nullptr, timeout);
  for (int i = max(0, k_issued - kst); i < k_issued; ++i)
    mbar_wait(k_full + i % kst, (i / kst) & 1, nullptr, timeout);
  for (int i = max(0, v_issued - vst); i < v_issued; ++i)
    mbar_wait(v_full + i % vst, (i / vst) & 1, nullptr, timeout);
}

template <int D, int DV, int NQ, int KST, int VST>
__global__ void __launch_bounds__(Cfg<D, DV, NQ, KST, VST>::kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D, DV, NQ, KST, VST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* bar_q = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + KST;
  uint64_t* v_full = k_empty + KST;
  uint64_t* v_empty = v_full + VST;
  uint64_t* s_full = v_empty + VST;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_full = p_full + NQ;
  uint64_t* bar_drain = o_full + NQ;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_trigger();  // a dependent merge may launch once every CTA is resident

  // ---- work item: (tile of 128 rows of one segment, group of NQ heads) ----
  const int hg = blockIdx.x % p.n_hgroups;
  const int rest = blockIdx.x / p.n_hgroups;
  // split-KV mode: block-major (the grid is query-tile units x KV blocks x
  // head groups), so that the CTAs running together read the same KV block:
  // one block of every head fits L2, all blocks do not
  const int tile_units = p.split_block > 0 ? (int)(gridDim.x / p.n_hgroups) / p.max_blocks : 1;
  const int jblk = p.split_block > 0 ? rest / tile_units : 0;
  const int tile_idx = p.split_block > 0 ? rest % tile_units : rest;
  cp_segment_t sg;
  int t, seg_id, kv_lo, kv_hi;
  long long out_row0;
  if (!resolve_tile(p, tile_idx, sg, t, seg_id) ||
      !split_window(p, sg, seg_id, jblk, kv_lo, kv_hi, out_row0)) {
    grid_dep_wait();  // no CTA ends before the kernel this launch may overlap
    return;
  }
  // packed heads: BM / 2 query rows per head, two heads per tile
  const int HP = p.pack_heads ? 2 : 1;
  if (p.pack_heads && sg.q_len > BM / 2) {
    if (threadIdx.x == 0) set_status(p.status, CPATTN_ERR_RANGE);
    grid_dep_wait();
    return;
  }
  const int r0 = t * BM;
  const int rows_valid = min(BM / HP, sg.q_len - r0);
  const int pos_max = sg.q_pos0 + (r0 + rows_valid - 1) * sg.q_pos_step;
  const int win_lo = max(kv_lo, 0);
  const int win_hi_tile = kv_hi < 0 ? pos_max + 1 : min(kv_hi, pos_max + 1);
  const int j0 = win_lo / BN;
  const int n_kv = win_hi_tile > win_lo ? (win_hi_tile + BN - 1) / BN - j0 : 0;
  const int head0 = hg * NQ * HP;       // query heads head0 .. head0+NQ*HP-1
  const int kv_head = head0 / p.g;      // shared by all of them (g % (NQ*HP) == 0)

  // ---- setup: barriers, TMEM ----
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < KST; ++i) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(v_full + i, 1); mbar_init(v_empty + i, 1); }
    for (int s = 0; s < NQ; ++s) {
      mbar_init(s_full + s, 1);
      mbar_init(p_full + s, 128);
      mbar_init(o_full + s, 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    tmem_slot[2] = 0;
    tmem_slot[3] = 0;
    fence_barrier_init();
  }
  if (warp == C::kProducerWarp) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // producer's issued-load counts, kept in shared memory for the abort drain
  volatile int* issued_kv = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const uint32_t q_base = smem_u32(smem + C::kQOff);
  const uint32_t k_base = smem_u32(smem + C::kKOff);
  const uint32_t v_base = smem_u32(smem + C::kVOff);

  if (warp >= 4 * NQ) {
    if constexpr (C::kSplitRegs)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::kRegsOther));
  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0 && n_kv > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      int k_issued = 0, v_issued = 0;
      if (!p.withhold_q) {
        mbar_arrive_expect_tx(bar_q, NQ * C::kQTileBytes);
        // HP boxes of BM / HP rows per 64-column chunk (one per packed head)
        for (int s = 0; s < NQ; ++s)
          for (int hp = 0; hp < HP; ++hp)
            for (int c = 0; c < D / 64; ++c)
              tma_load_3d(smem + C::kQOff + s * C::kQTileBytes + c * BM * 128 +
                              hp * (BM / HP) * 128,
                          &tm_q, bar_q, c * 64, head0 + s * HP + hp, sg.q_row0 + r0);
      }
      bool ok = true;
      for (int it = 0; it < n_kv && ok; ++it) {
        const int kv_row = sg.kv_row0 + (j0 + it) * BN;
        const int ks = it % KST;
        ok = mbar_wait(k_empty + ks, ((it / KST) & 1) ^ 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        mbar_arrive_expect_tx(k_full + ks, C::kKTileBytes);
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(smem + C::kKOff + ks * C::kKTileBytes + c * BN * 128, &tm_k, k_full + ks,
                      c * 64, kv_head, kv_row);
        ++k_issued;
        const int vs = it % VST;
        ok = mbar_wait(v_empty + vs, ((it / VST) & 1) ^ 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        mbar_arrive_expect_tx(v_full + vs, C::kVTileBytes);
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(smem + C::kVOff + vs * C::kVTileBytes + c * BN * 128, &tm_v, v_full + vs,
                      c * 64, kv_head, kv_row);
        ++v_issued;
      }
      issued_kv[0] = k_issued;
      issued_kv[1] = v_issued;
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (warp == C::kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0 && n_kv > 0) {
      constexpr uint32_t kIdescQK = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(BM, DV, 0, 1);
      // Descriptors are built once; each MMA adds a compile-time offset
      // (start address >> 4 in the low bits), so the single issuing thread
      // spends a few independent instructions per MMA instead of a long
      // dependent chain.
      const uint64_t dq0 = smem_desc_sw128(q_base, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(k_base, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(v_base, BN * 128, 1024);
      auto issue_qk = [&](int s, int ks) {
        const uint64_t qd = dq0 + (uint64_t)((s * C::kQTileBytes) >> 4);
        const uint64_t kd = dk0 + (uint64_t)((ks * C::kKTileBytes) >> 4);
        const uint32_t dt = tmem_base + s * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          constexpr int kQChunk = (BM * 128) >> 4, kKChunk = (BN * 128) >> 4;
          const uint64_t oq = (uint64_t)((kk >> 2) * kQChunk + (kk & 3) * 2);
          const uint64_t ok_ = (uint64_t)((kk >> 2) * kKChunk + (kk & 3) * 2);
          mma_ss(dt, qd + oq, kd + ok_, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int s, int vs, bool acc) {
        const uint64_t vd = dv0 + (uint64_t)((vs * C::kVTileBytes) >> 4);
        const uint32_t dt = tmem_base + NQ * BN + s * DV;
        const uint32_t pt = tmem_base + s * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(dt, pt + kk * 8, vd + (uint64_t)(kk * ((16 * 128) >> 4)), kIdescPV,
                 (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.timeout_ns);
      if (ok) ok = mbar_wait(k_full, 0, abort_flag, p.timeout_ns);
      if (ok) {
        tc_fence_after();
        for (int s = 0; s < NQ; ++s) {
          issue_qk(s, 0);
          mma_commit(s_full + s);
        }
        mma_commit(k_empty);
      }
      for (int it = 0; it < n_kv && ok; ++it) {
        const int vs = it % VST;
        ok = mbar_wait(v_full + vs, (it / VST) & 1, abort_flag, p.timeout_ns);
        if (!ok) break;
        const int ks_next = (it + 1) % KST;
        for (int s = 0; s < NQ && ok; ++s) {
          ok = mbar_wait(p_full + s, it & 1, abort_flag, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          issue_pv(s, vs, it > 0);
          if (it == n_kv - 1) mma_commit(o_full + s);
          if (it + 1 < n_kv) {
            if (s == 0) {
              ok = mbar_wait(k_full + ks_next, ((it + 1) / KST) & 1, abort_flag, p.timeout_ns);
              if (!ok) break;
              tc_fence_after();
            }
            issue_qk(s, ks_next);
            mma_commit(s_full + s);
          }
        }
        if (!ok) break;
        mma_commit(v_empty + vs);
        if (it + 1 < n_kv) mma_commit(k_empty + ks_next);
      }
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      // drain: every MMA and commit issued by this thread has completed
      mma_commit(bar_drain);
      mbar_wait(bar_drain, 0, nullptr, p.timeout_ns);
    }
  }
  } else {
    if constexpr (C::kSplitRegs)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::kRegsSoftmax));
    // ------------------------------------------------------------- softmax --
    const int s = warp >> 2;               // query tile of this warpgroup
    const int wq = warp & 3;               // TMEM lane quarter
    const int trow = wq * 32 + lane;       // row within the tile
    // query row and head of this thread (packed: two heads per tile, the
    // head uniform across a warp)
    const int row = p.pack_heads ? (trow & (BM / 2 - 1)) : trow;
    const int h = head0 + s * HP + (p.pack_heads ? trow / (BM / 2) : 0);
    const bool valid = row < rows_valid;
    const int pos = valid ? sg.q_pos0 + (r0 + row) * sg.q_pos_step : -1;
    const int row_hi = valid ? (kv_hi < 0 ? pos + 1 : min(kv_hi, pos + 1)) : 0;
    // output row, computed before the KV loop (fewer live registers in the
    // loop than at the store); split-KV mode: known only at the store
    long long out_row = valid ? output_row(p, sg, r0, row, out_row0) : -1;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_col = s * BN, o_col = NQ * BN + s * DV;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f, m_use = 0.f;
    bool ok = true;
    for (int it = 0; it < n_kv; ++it) {
      ok = mbar_wait_warp(s_full + s, it & 1, abort_flag, p.timeout_ns);
      if (!ok) break;
      tc_fence_after();
      float x[BN];
      {
        uint32_t r[BN];
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) tmem_ld32p(lane_addr + s_col + q * 32, r + q * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < BN; ++c) x[c] = __uint_as_float(r[c]);
      }
      const int key0 = (j0 + it) * BN;
      if (key0 < win_lo || key0 + BN > row_hi) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = key0 + c;
          if (key < win_lo || key >= row_hi) x[c] = -INFINITY;
        }
      }
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int c = 4; c < BN; c += 8) {
        mx0 = fmax3(mx0, x[c], x[c + 1]);
        mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
        mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
        mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      // Lazy max: keep the running max unless the tile raises it by more than
      // kMaxSlack (log2 units).  Exponentials against a stale max are at most
      // 2^kMaxSlack, and l is accumulated against the same max, so O / l and
      // L are unchanged; O in TMEM is rescaled only when the max moves.
      const bool move = mx > m_run + kMaxSlack;
      const float m_new = move ? mx : m_run;
      const float m_new_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = move ? ex2_approx(m_run - m_new_use) : 1.f;  // 0 while m_run = -inf
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int q = 0; q < BN / 32; ++q) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float a, b;
          ffma2(a, b, x[q * 32 + c], x[q * 32 + c + 1], sl2, sl2, -m_new_use, -m_new_use);
          a = ex2_approx(a);
          b = ex2_approx(b);
          fadd2(sum0, sum1, sum0, sum1, a, b);
          pk[c >> 1] = pack_bf16x2(a, b);
        }
        tmem_st16(lane_addr + s_col + q * 16, pk);
      }
      l_run = l_run * alpha + (sum0 + sum1);
      // rescale the running O (its previous PV has completed: S of this
      // iteration was committed after it)
      const bool need = (it > 0) && move;
      if (__any_sync(0xffffffffu, need)) {
        const float a = need ? alpha : 1.f;
        uint32_t r[32];
#pragma unroll
        for (int q = 0; q < DV / 32; ++q) {
          tmem_ld32(lane_addr + o_col + q * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * a);
          tmem_st32(lane_addr + o_col + q * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full + s);
      m_run = m_new;
      m_use = m_new_use;
    }
    if (ok && n_kv > 0) ok = mbar_wait_warp(o_full + s, 0, abort_flag, p.timeout_ns);
    if (!ok) {
      if (lane == 0) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      tc_fence_after();
      if (p.split_block > 0) {
        const long long w0 = split_slot_row0(p, sg, seg_id, jblk, out_row0);
        out_row = (valid && w0 >= 0) ? w0 + r0 + row : -1;
      }
      const bool has = l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
      MergeCoef mc{0.f, inv, has ? (m_use + lg2_approx(l_run)) * kLn2 : -INFINITY};
      if (p.lse_acc) {
        // accumulate mode (fp32 O): merge into the partial already stored
        if (out_row >= 0) mc = merge_coef(__ldg(p.lse_acc + out_row * p.Hq + h), has, m_use, l_run);
#pragma unroll 1
        for (int q = 0; q < DV / 32; ++q) {
          uint32_t r[32];
          if (n_kv > 0) {
            tmem_ld32(lane_addr + o_col + q * 32, r);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = 0u;
          }
          if (out_row >= 0) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.o) +
                                                    (out_row * p.Hq + h) * DV + q * 32);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 a = dst[c];
              dst[c] = make_float4(mc.c_old * a.x + mc.c_new * __uint_as_float(r[4 * c]),
                                   mc.c_old * a.y + mc.c_new * __uint_as_float(r[4 * c + 1]),
                                   mc.c_old * a.z + mc.c_new * __uint_as_float(r[4 * c + 2]),
                                   mc.c_old * a.w + mc.c_new * __uint_as_float(r[4 * c + 3]));
            }
          }
        }
      } else {
        // Plain store, staged per warp through shared memory: each thread
        // puts 128 bytes of its row in the warp's 32-row buffer (16-byte
        // chunks XOR-swizzled by row, so neither side has bank conflicts),
        // then every store instruction writes 4 rows x 128 contiguous bytes.
        uint8_t* stage = smem + C::kStageOff + warp * (32 * 128);
        const int row_bytes = DV * (p.o_f32 ? 4 : 2);
        for (int b0 = 0; b0 < row_bytes; b0 += 128) {
          uint32_t pk[32];  // 128 bytes of this thread's row
          if (p.o_f32) {
            uint32_t r[32];
            if (n_kv > 0) {
              tmem_ld32(lane_addr + o_col + b0 / 4, r);
              tmem_wait_ld();
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = 0u;
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = __float_as_uint(__uint_as_float(r[c]) * inv);
          } else {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t r[32];
              if (n_kv > 0) {
                tmem_ld32(lane_addr + o_col + b0 / 2 + hh * 32, r);
                tmem_wait_ld();
              } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) r[c] = 0u;
              }
#pragma unroll
              for (int c = 0; c < 16; ++c)
                pk[hh * 16 + c] = pack_bf16x2(__uint_as_float(r[2 * c]) * inv,
                                              __uint_as_float(r[2 * c + 1]) * inv);
            }
          }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) * 16)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3), ch = lane & 7;
            const long long orr = __shfl_sync(0xffffffffu, out_row, rr);
            const uint4 val =
                *reinterpret_cast<const uint4*>(stage + rr * 128 + ((ch ^ (rr & 7)) * 16));
            if (orr >= 0) {
              uint8_t* dst = reinterpret_cast<uint8_t*>(p.o) + (orr * p.Hq + h) * row_bytes +
                             b0 + ch * 16;
              *reinterpret_cast<uint4*>(dst) = val;
            }
          }
          __syncwarp();
        }
      }
      if (out_row >= 0) p.lse[out_row * p.Hq + h] = mc.lse;
    }
  }

  // ---- teardown ----
  grid_dep_wait();  // (already returned in the epilogue unless this CTA aborted)
  tc_fence_before();
  __syncthreads();
  if (warp == C::kProducerWarp) {
    if (lane == 0 && *abort_flag && n_kv > 0)
      drain_after_abort(bar_q, !p.withhold_q, k_full, KST, issued_kv[0], v_full, VST,
                        issued_kv[1], p.timeout_ns);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int D, int DV, int NQ, int KST, int VST>
int launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const AttnParams& prm, long long tiles, cudaStream_t stream) {
  using C = Cfg<D, DV, NQ, KST, VST>;
  auto kern = attn_fwd_kernel<D, DV, NQ, KST, VST>;
  if (!allow_smem(kern, C::kSmemBytes)) return CPATTN_ERR_CUDA;
  // setmaxnreg.inc waits until the block's launch allocation can cover the
  // split; refuse a build whose register count could not.  The count is a
  // property of this binary, the same in every context: 0 not checked yet,
  // 1 ok, -1 refused.
  static int regs_ok = 0;
  if (regs_ok == 0) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return CPATTN_ERR_CUDA;
    regs_ok = (!C::kSplitRegs ||
               fa.numRegs * C::kThreads >= C::kRegsOther * 128 + C::kRegsSoftmax * 256)
                  ? 1
                  : -1;
  }
  if (regs_ok < 0) return CPATTN_ERR_UNSUPPORTED;
  const long long grid = tiles * prm.n_hgroups;  // tiles x KV blocks (split mode) x head groups
  if (grid <= 0) return CPATTN_OK;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_INVALID_ARG;
  return launch_kernel(kern, (unsigned)grid, C::kThreads, C::kSmemBytes, stream, prm.pdl != 0,
                       mq, mk, mv, prm) == cudaSuccess
             ? CPATTN_OK
             : CPATTN_ERR_CUDA;
}

}  // namespace
}  // namespace cpattn

using namespace cpattn;

AttnDebug& cpattn::attn_debug() {
  static AttnDebug d;
  return d;
}

extern "C" int cp_attn_debug(int knob, long long value) {
  switch (knob) {
    case CPATTN_DEBUG_WAIT_LIMIT_NS:
      if (value <= 0) return CPATTN_ERR_INVALID_ARG;
      attn_debug().timeout_ns = (unsigned long long)value;
      return CPATTN_OK;
    case CPATTN_DEBUG_WITHHOLD_Q:
      attn_debug().withhold_q = value ? 1 : 0;
      return CPATTN_OK;
    case CPATTN_DEBUG_NVTX:
      nvtx_flag().store(value ? 1 : 0);
      return CPATTN_OK;
    default:
      return CPATTN_ERR_INVALID_ARG;
  }
}

int cpattn::attn_launch(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                        int num_tiles, const void* q, int num_q_rows, const void* k,
                        int64_t k_row_stride, int64_t k_head_stride, const void* v,
                        int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                        int Hkv, int d, int dv, float scale, AttnParams& prm,
                        cudaStream_t stream) {
  if (num_segs < 0 || num_q_rows < 0 || num_kv_rows < 0) return CPATTN_ERR_INVALID_ARG;
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || !(scale > 0.f)) return CPATTN_ERR_INVALID_ARG;
  const bool mla = (d == 576 && dv == 512);
  const bool shape_ok = (d == 64 && dv == 64) || (d == 128 && dv == 128) || mla;
  if (!shape_ok) return CPATTN_ERR_UNSUPPORTED;
  // absorbed MLA: the value is the first 512 columns of the key rows
  if (mla && (v != k || v_row_stride != k_row_stride || v_head_stride != k_head_stride))
    return CPATTN_ERR_UNSUPPORTED;
  if (tiles_dev && num_tiles < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_segs == 0 || (tiles_dev && num_tiles == 0)) return CPATTN_OK;
  if (!segs_dev || !q || !k || !v) return CPATTN_ERR_INVALID_ARG;
  if (num_q_rows == 0 || num_kv_rows == 0) return CPATTN_ERR_INVALID_ARG;
  if (!a16(segs_dev) || !a16(q) || !a16(k) || !a16(v) ||
      (reinterpret_cast<uintptr_t>(tiles_dev) & 7u))
    return CPATTN_ERR_ALIGNMENT;
  if ((k_row_stride * 2) % 16 || (k_head_stride * 2) % 16 || (v_row_stride * 2) % 16 ||
      (v_head_stride * 2) % 16)
    return CPATTN_ERR_ALIGNMENT;
  if (k_head_stride < d || v_head_stride < dv ||
      k_row_stride < (int64_t)(Hkv - 1) * k_head_stride + d ||
      v_row_stride < (int64_t)(Hkv - 1) * v_head_stride + dv)
    return CPATTN_ERR_INVALID_ARG;

  const int g = Hq / Hkv;
  const int nq = (g % 2 == 0) ? 2 : 1;
  // head packing (segments of at most BM / 2 rows): both tiles of a CTA hold
  // two heads each, so the head group spans 4 heads of one KV head
  if (prm.pack_heads && (mla || nq != 2 || g % 4 != 0)) prm.pack_heads = 0;
  prm.segs = segs_dev;
  prm.tiles = tiles_dev;
  prm.num_segs = num_segs;
  prm.num_tiles = tiles_dev ? num_tiles : 0;
  prm.Hq = Hq;
  prm.g = g;
  prm.n_hgroups = Hq / (nq * (prm.pack_heads ? 2 : 1));
  prm.scale_log2 = scale * kLog2e;
  prm.num_q_rows = num_q_rows;
  prm.num_kv_rows = num_kv_rows;
  prm.timeout_ns = attn_debug().timeout_ns;
  prm.withhold_q = attn_debug().withhold_q;
  long long units =
      tiles_dev ? num_tiles : ((long long)num_q_rows + BM - 1) / BM + (long long)num_segs;
  if (prm.split_block > 0) units *= prm.max_blocks;
  if (mla)
    return launch_attn_mla(q, num_q_rows, k, k_row_stride, k_head_stride, num_kv_rows, Hkv, prm,
                           units, stream);
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, d, Hq, num_q_rows, d, (long long)Hq * d, prm.pack_heads ? BM / 2 : BM) ||
      !make_map(&mk, k, d, Hkv, num_kv_rows, k_head_stride, k_row_stride) ||
      !make_map(&mv, v, dv, Hkv, num_kv_rows, v_head_stride, v_row_stride))
    return CPATTN_ERR_CUDA;
  if (d == 128) {
    if (nq == 2) return launch_attn<128, 128, 2, 2, 2>(mq, mk, mv, prm, units, stream);
    return launch_attn<128, 128, 1, 2, 2>(mq, mk, mv, prm, units, stream);
  }
  if (nq == 2) return launch_attn<64, 64, 2, 3, 3>(mq, mk, mv, prm, units, stream);
  return launch_attn<64, 64, 1, 3, 3>(mq, mk, mv, prm, units, stream);
}

extern "C" int cp_attn_partial(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev,
                               int num_tiles, const void* q, int num_q_rows, const void* k,
                               int64_t k_row_stride, int64_t k_head_stride, const void* v,
                               int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq,
                               int Hkv, int d, int dv, float scale, int kv_lo, int kv_hi, void* o,
                               int o_is_fp32, float* lse, int out_row_base, int num_out_rows,
                               int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_partial");
  if (num_out_rows < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_segs > 0 && (!o || !lse || num_out_rows == 0)) return CPATTN_ERR_INVALID_ARG;
  if (o && (!a16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))) return CPATTN_ERR_ALIGNMENT;
  AttnParams prm{};
  prm.kv_lo = kv_lo;
  prm.kv_hi = kv_hi;
  prm.o = o;
  prm.o_f32 = o_is_fp32 ? 1 : 0;
  prm.lse = lse;
  prm.out_row_base = out_row_base;
  prm.num_out_rows = num_out_rows;
  prm.status = status_dev;
  prm.split_block = 0;
  return attn_launch(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k, k_row_stride,
                     k_head_stride, v, v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv,
                     scale, prm, stream);
}

extern "C" int cp_attn_prefill(const cp_segment_t* segs_dev, int num_segs,
                               const int32_t* tiles_dev, int num_tiles, const void* q,
                               int num_tokens, const void* k, int64_t k_row_stride,
                               int64_t k_head_stride, const void* v, int64_t v_row_stride,
                               int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv, int d,
                               int dv, float scale, void* o, int o_is_fp32, float* lse,
                               int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_prefill");
  if (num_tokens < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_segs > 0 && (!o || !lse || num_tokens == 0)) return CPATTN_ERR_INVALID_ARG;
  if (o && (!a16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))) return CPATTN_ERR_ALIGNMENT;
  AttnParams prm{};
  prm.kv_lo = 0;
  prm.kv_hi = -1;
  prm.o = o;
  prm.o_f32 = o_is_fp32 ? 1 : 0;
  prm.lse = lse;
  prm.out_row_base = 0;
  prm.num_out_rows = num_tokens;
  prm.q_token_rows = 1;
  prm.status = status_dev;
  prm.split_block = 0;
  return attn_launch(segs_dev, num_segs, tiles_dev, num_tiles, q, num_tokens, k, k_row_stride,
                     k_head_stride, v, v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv,
                     scale, prm, stream);
}

extern "C" int cp_attn_partial_restore(
    const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev, int num_tiles,
    const void* q, int num_q_rows, const void* k, int64_t k_row_stride, int64_t k_head_stride,
    const void* v, int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv,
    int d, int dv, float scale, int kv_lo, int kv_hi, const int32_t* dst_rows, void* o,
    int o_is_fp32, float* lse, int num_out_rows, int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_partial_restore");
  if (num_out_rows < 0) return CPATTN_ERR_INVALID_ARG;
  if (num_segs > 0 && (!o || !lse || !dst_rows || num_out_rows == 0))
    return CPATTN_ERR_INVALID_ARG;
  if (o && (!a16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u))) return CPATTN_ERR_ALIGNMENT;
  AttnParams prm{};
  prm.kv_lo = kv_lo;
  prm.kv_hi = kv_hi;
  prm.o = o;
  prm.o_f32 = o_is_fp32 ? 1 : 0;
  prm.lse = lse;
  prm.out_row_base = 0;
  prm.num_out_rows = num_q_rows;  // segment rows are checked against the query rows
  prm.dst_rows = dst_rows;
  prm.dst_limit = num_out_rows;
  prm.status = status_dev;
  prm.split_block = 0;
  return attn_launch(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k, k_row_stride,
                     k_head_stride, v, v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv,
                     scale, prm, stream);
}

extern "C" int cp_attn_partial_accumulate(
    const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev, int num_tiles,
    const void* q, int num_q_rows, const void* k, int64_t k_row_stride, int64_t k_head_stride,
    const void* v, int64_t v_row_stride, int64_t v_head_stride, int num_kv_rows, int Hq, int Hkv,
    int d, int dv, float scale, int kv_lo, int kv_hi, const int32_t* seg_windows_dev,
    float* o_acc, const float* lse_acc, float* lse_out, int out_row_base, int num_out_rows,
    int32_t* status_dev, cudaStream_t stream) {
  CPATTN_TRACE("cp_attn_partial_accumulate");
  if (num_out_rows < 0 || Hq <= 0) return CPATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(seg_windows_dev) & 3u) return CPATTN_ERR_ALIGNMENT;
  if (num_segs > 0 && (!o_acc || !lse_acc || !lse_out || num_out_rows == 0))
    return CPATTN_ERR_INVALID_ARG;
  if (o_acc && (!a16(o_acc) || (reinterpret_cast<uintptr_t>(lse_acc) & 3u) ||
                (reinterpret_cast<uintptr_t>(lse_out) & 3u)))
    return CPATTN_ERR_ALIGNMENT;
  if (lse_acc && lse_out) {
    // both LSE buffers span num_out_rows * Hq floats and must not overlap
    const uintptr_t a = reinterpret_cast<uintptr_t>(lse_acc), b = reinterpret_cast<uintptr_t>(lse_out);
    const uintptr_t n = (uintptr_t)num_out_rows * (uintptr_t)Hq * sizeof(float);
    if (a < b + n && b < a + n) return CPATTN_ERR_INVALID_ARG;
  }
  AttnParams prm{};
  prm.kv_lo = kv_lo;
  prm.kv_hi = kv_hi;
  prm.o = o_acc;
  prm.o_f32 = 1;
  prm.lse = lse_out;
  prm.lse_acc = lse_acc;
  prm.seg_windows = seg_windows_dev;
  prm.out_row_base = out_row_base;
  prm.num_out_rows = num_out_rows;
  prm.status = status_dev;
  prm.split_block = 0;
  return attn_launch(segs_dev, num_segs, tiles_dev, num_tiles, q, num_q_rows, k, k_row_stride,
                     k_head_stride, v, v_row_stride, v_head_stride, num_kv_rows, Hq, Hkv, d, dv,
                     scale, prm, stream);
}
