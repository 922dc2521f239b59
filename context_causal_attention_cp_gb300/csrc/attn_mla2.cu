// Shard partial attention, absorbed-MLA shape, on pairs of SMs (sm_103a).
//
// The same computation as attn_mla.cu (query and key rows are the 576-wide
// absorbed latent, V = K[:, :512]; blog "什么是 Context Parallelism", §4.2)
// with every MMA issued for two SMs at once (tcgen05 cta_group::2): a cluster
// of two CTAs holds the same 128 query rows of two query heads (2h', 2h'+1;
// all heads share the one latent KV head) for one 256-column output half, and
// one thread of the even CTA issues M = 256 MMAs that read each CTA's own
// operands.  Keys come in tiles of 128.
//
// Why pairs: one SM's tensor and shared memory cannot hold a 128-key S tile
// next to the 576-wide query and the 256-column O half, and with 64-key tiles
// the single issuing thread, not the tensor core, sets the pace (an N = 64
// MMA executes in less time than it takes to issue).  A pair splits the key
// tile of Q K^T (each CTA stores 64 of its 128 keys) and the value columns of
// P V (each CTA stores 128 of the 256), so every MMA has N = 128 or 256.
//
// Per CTA:
//   tensor memory (512 columns): S_0 and S_1 (128 x 128 fp32 each; tile j
//     uses S_{j mod 2}, and P_j is written over it as bf16, the A operand of
//     P_j V_j) and the O half.
//   shared memory: the whole 576-wide query (nine 64-column chunks), a ring
//     of two slots of three K chunks (64 keys x 64 columns each, one barrier
//     per slot) and one buffer of this CTA's V columns (128 keys x 128).
//   MMA order: Q K_0^T, Q K_1^T, then per tile j: P_j V_j, Q K_{j+2}^T.  With
//     S double-buffered the tensor cores compute the next tile's scores while
//     the softmax of this one runs, and P_j has all of Q K_{j+1}^T and
//     P_{j-1} V_{j-1} to be produced.
//   softmax: two warpgroups, each thread taking 64 of its row's 128 scores
//     (and 128 of its 256 output columns); the halves of a row exchange their
//     maxima (and, at the end, their sums) through shared memory.
// Loads: each CTA's TMA copies land in its own shared memory and complete on
// the even CTA's barriers (the .cta_group::2 form of the copy), which the even
// CTA's producer arms with both CTAs' bytes.
// Every wait is bounded; a wait that runs out sets CPATTN_ERR_TIMEOUT and
// aborts both CTAs of the pair, which let their copies land, meet and free
// tensor memory.
#include <algorithm>
#include <cstdint>

#include "attn_common.cuh"
#include "pair.cuh"

namespace cpattn {
namespace {

using namespace pair;

constexpr int kD2 = 576, kDV2 = 512, kDVH2 = 256, kBN2 = 128, kCh2 = kD2 / 64;
constexpr int kSoftWarps2 = 8;          // two warpgroups: half h of every row
constexpr int kProducerWarp2 = kSoftWarps2, kMmaWarp2 = kSoftWarps2 + 1;
constexpr int kThreads2 = (kSoftWarps2 + 2) * 32;
constexpr int kKSlots2 = 2;             // slots of kKGroup chunks
constexpr int kKGroup = 3;
constexpr int kQChunk2 = BM * 128;      // 16 KB: 128 rows x 64 columns
constexpr int kKChunk2 = 64 * 128;      // 8 KB: this CTA's 64 keys x 64 columns
constexpr int kVChunk2 = kBN2 * 128;    // 16 KB: 128 keys x 64 columns
constexpr int kQOff2 = 0;
constexpr int kKOff2 = kQOff2 + kCh2 * kQChunk2;
constexpr int kVOff2 = kKOff2 + kKSlots2 * kKGroup * kKChunk2;
constexpr int kXOff2 = kVOff2 + 2 * kVChunk2;   // row exchange: [2 rounds][2 halves][BM] floats
constexpr int kBarOff2 = kXOff2 + 2 * 2 * BM * 4;
// barriers ("pair" ones are used in the even CTA and count both CTAs)
constexpr int kBQ = 0;                    // pair: the query of both CTAs
constexpr int kBKF = 1;                   // pair [2]: K slot full in both CTAs
constexpr int kBKE = kBKF + kKSlots2;     // local [2]: K slot free (multicast commit)
constexpr int kBVF = kBKE + kKSlots2;     // pair: V buffer full in both CTAs
constexpr int kBVE = kBVF + 1;            // local: V buffer free (multicast commit)
constexpr int kBSF = kBVE + 1;            // local [2]: S_b ready (multicast commit)
constexpr int kBPF = kBSF + 2;            // pair [2]: P_b written by both CTAs' softmax
constexpr int kBPD = kBPF + 2;            // local: P V of a tile done (multicast commit)
constexpr int kBDR = kBPD + 1;            // even CTA: every MMA complete
constexpr int kBX = kBDR + 1;             // local [4]: the two halves of a row quarter met
constexpr int kNumBars2 = kBX + 4;
// The dynamic shared memory is declared 1024-byte aligned (the 128-byte
// swizzle atoms of the TMA boxes and MMA descriptors need it), so no slack is
// requested; the kernel checks the alignment and reports a misaligned base.
constexpr int kSmem2 = kBarOff2 + kNumBars2 * 8 + 16;
static_assert(kSmem2 <= 232448, "MLA pair tile exceeds shared memory");
constexpr uint32_t kOCol2 = 2 * kBN2;  // TMEM: S_0 at 0, S_1 at 128, O at 256

// The MMA issuer (one thread of the even CTA).
__device__ __noinline__ void mla2_mma_issue(const AttnParams& p, uint8_t* smem, uint32_t tmem_base,
                                            int n_kv, uint64_t* bars, volatile int* abort_flag,
                                            uint32_t peer_abort) {
  constexpr uint32_t kIdescQK = idesc_bf16_f32(2 * BM, kBN2, 0, 0);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(2 * BM, kDVH2, 0, 1);
  const uint64_t dq0 = smem_desc_sw128(smem_u32(smem + kQOff2), 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(smem_u32(smem + kKOff2), 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(smem_u32(smem + kVOff2), kVChunk2, 1024);
  const uint32_t o_tm = tmem_base + kOCol2;
  int g = 0;  // K chunk groups consumed
  // S_{j mod 2} = Q K_j^T over the nine chunks, three per K slot
  auto qk = [&](int j) -> bool {
    const uint32_t s_tm = tmem_base + (j & 1) * kBN2;
#pragma unroll
    for (int grp = 0; grp < kCh2 / kKGroup; ++grp, ++g) {
      const int slot = g % kKSlots2;
      if (!mbar_wait(bars + kBKF + slot, (g / kKSlots2) & 1, abort_flag, p.timeout_ns))
        return false;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < kKGroup; ++cc) {
        const int c = grp * kKGroup + cc;
        const uint64_t qd = dq0 + (uint64_t)((c * kQChunk2) >> 4);
        const uint64_t kd = dk0 + (uint64_t)(((slot * kKGroup + cc) * kKChunk2) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma2_ss(s_tm, qd + kk * 2, kd + kk * 2, kIdescQK, (c == 0 && kk == 0) ? 0u : 1u);
      }
      commit2_both(bars + kBKE + slot);
    }
    commit2_both(bars + kBSF + (j & 1));
    return true;
  };
  bool ok = mbar_wait(bars + kBQ, 0, abort_flag, p.timeout_ns);
  if (ok) ok = qk(0);
  if (ok && n_kv > 1) ok = qk(1);
  for (int j = 0; j < n_kv && ok; ++j) {
    // O += P_j V_j, P_j read from tensor memory over S_{j mod 2}
    ok = wait_pair(bars + kBPF + (j & 1), (j >> 1) & 1, abort_flag, p.timeout_ns);
    if (!ok) break;
    ok = mbar_wait(bars + kBVF, j & 1, abort_flag, p.timeout_ns);
    if (!ok) break;
    tc_fence_after();
    const uint32_t p_tm = tmem_base + (j & 1) * kBN2;
#pragma unroll
    for (int kk = 0; kk < kBN2 / 16; ++kk)
      mma2_ts(o_tm, p_tm + kk * 8, dv0 + (uint64_t)(kk * ((16 * 128) >> 4)), kIdescPV,
              (j > 0 || kk > 0) ? 1u : 0u);
    commit2_both(bars + kBVE);
    commit2_both(bars + kBPD);
    // the scores two tiles ahead overwrite S_{j mod 2} after P_j V_j has read it
    if (j + 2 < n_kv) ok = qk(j + 2);
  }
  if (!ok) {
    set_status(p.status, CPATTN_ERR_TIMEOUT);
    *abort_flag = 1;
    store_cluster_u32(peer_abort, 1);
  }
  // drain: every MMA issued by this thread has completed
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bars + kBDR))
               : "memory");
  mbar_wait(bars + kBDR, 0, nullptr, p.timeout_ns);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads2, 1)
attn_mla_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_trigger();  // a dependent merge may launch once every CTA is resident
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const uint32_t peer_abort = peer_addr((const void*)abort_flag, peer);

  // ---- work item: (128-row tile [, KV block], head pair, output half); CTA
  // `rank` of the pair takes head 2 * pair_head + rank ----
  const int pair_id = blockIdx.x >> 1;
  const int half = pair_id & 1;
  const int n_hp = p.Hq >> 1;
  const int hp = (pair_id >> 1) % n_hp;
  const int rest = (pair_id >> 1) / n_hp;
  const int h = 2 * hp + (int)rank;
  const int jblk = p.split_block > 0 ? rest % p.max_blocks : 0;
  const int tile_idx = p.split_block > 0 ? rest / p.max_blocks : rest;
  cp_segment_t sg;
  int t, seg_id, kv_lo, kv_hi;
  long long out_row0;
  // both CTAs of a pair resolve the same tile and window, so they leave together
  if (!resolve_tile(p, tile_idx, sg, t, seg_id) ||
      !split_window(p, sg, seg_id, jblk, kv_lo, kv_hi, out_row0)) {
    grid_dep_wait();  // no CTA ends before the kernel this launch may overlap
    return;
  }
  // the swizzled layouts need a 1024-byte aligned base (declared above; both
  // CTAs see the same layout, so both leave here together)
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(p.status, CPATTN_ERR_ALIGNMENT);
    grid_dep_wait();
    return;
  }
  const int r0 = t * BM;
  const int rows_valid = min(BM, sg.q_len - r0);
  const int pos_max = sg.q_pos0 + (r0 + rows_valid - 1) * sg.q_pos_step;
  const int win_lo = max(kv_lo, 0);
  const int win_hi_tile = kv_hi < 0 ? pos_max + 1 : min(kv_hi, pos_max + 1);
  const int j0 = win_lo / kBN2;
  const int n_kv = win_hi_tile > win_lo ? (win_hi_tile + kBN2 - 1) / kBN2 - j0 : 0;
  const int kv_head = h / p.g;  // both heads share it (the latent head)

  if (threadIdx.x == 0) {
    mbar_init(bars + kBQ, 1);
    for (int sl = 0; sl < kKSlots2; ++sl) {
      mbar_init(bars + kBKF + sl, 1);
      mbar_init(bars + kBKE + sl, 1);
    }
    mbar_init(bars + kBVF, 1);
    mbar_init(bars + kBVE, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars + kBSF + b, 1);
      mbar_init(bars + kBPF + b, 2 * kSoftWarps2);
    }
    mbar_init(bars + kBPD, 1);
    mbar_init(bars + kBDR, 1);
    for (int i = 0; i < 4; ++i) mbar_init(bars + kBX + i, 2);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // barriers and tensor memory of both CTAs are ready
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint64_t to = p.timeout_ns;

  if (warp == kProducerWarp2) {
    // ------------------------------------------------------------ producer --
    // Every copy lands in this CTA's shared memory and completes on the even
    // CTA's barrier, which the even CTA's producer arms with both CTAs' bytes.
    // Loads follow the MMAs' order: K of tiles 0 and 1, then per tile j the V
    // of tile j and the K of tile j + 2; K chunk group g (three chunks) goes to
    // slot g % 2 once the MMAs of group g - 2 have released it.
    if (lane == 0 && n_kv > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      const bool lead = rank == 0;
      if (!p.withhold_q) {
        if (lead) mbar_arrive_expect_tx(bars + kBQ, 2 * kCh2 * kQChunk2);
        const uint32_t fq = peer_addr(bars + kBQ, 0);
        for (int c = 0; c < kCh2; ++c)
          tma_load_pair(smem + kQOff2 + c * kQChunk2, &tm_q, fq, c * 64, h, sg.q_row0 + r0);
      }
      bool ok = true;
      int g = 0;
      auto load_k = [&](int j) -> bool {
        const int kv_row = sg.kv_row0 + (j0 + j) * kBN2;
        for (int grp = 0; grp < kCh2 / kKGroup; ++grp, ++g) {
          const int slot = g % kKSlots2;
          if (!mbar_wait(bars + kBKE + slot, ((g / kKSlots2) & 1) ^ 1, abort_flag, to))
            return false;
          if (lead) mbar_arrive_expect_tx(bars + kBKF + slot, 2 * kKGroup * kKChunk2);
          for (int cc = 0; cc < kKGroup; ++cc)
            tma_load_pair(smem + kKOff2 + (slot * kKGroup + cc) * kKChunk2, &tm_k,
                          peer_addr(bars + kBKF + slot, 0), (grp * kKGroup + cc) * 64, kv_head,
                          kv_row + 64 * (int)rank);
        }
        return true;
      };
      ok = load_k(0);
      if (ok && n_kv > 1) ok = load_k(1);
      for (int j = 0; j < n_kv && ok; ++j) {
        ok = mbar_wait(bars + kBVE, (j & 1) ^ 1, abort_flag, to);  // P_{j-1} V_{j-1} done
        if (!ok) break;
        if (lead) mbar_arrive_expect_tx(bars + kBVF, 2 * 2 * kVChunk2);
        const int kv_row = sg.kv_row0 + (j0 + j) * kBN2;
        for (int t2 = 0; t2 < 2; ++t2)
          tma_load_pair(smem + kVOff2 + t2 * kVChunk2, &tm_v, peer_addr(bars + kBVF, 0),
                        (4 * half + 2 * (int)rank + t2) * 64, kv_head, kv_row);
        if (j + 2 < n_kv) ok = load_k(j + 2);
      }
      if (!ok) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
        store_cluster_u32(peer_abort, 1);
      }
    }
  } else if (warp == kMmaWarp2) {
    // ---------------------------------------------- MMA issuer (even CTA) --
    if (lane == 0 && n_kv > 0 && rank == 0)
      mla2_mma_issue(p, smem, tmem_base, n_kv, bars, abort_flag, peer_abort);
  } else {
    // ------------------------------------------------------------- softmax --
    const int wq = warp & 3;               // TMEM lane quarter
    const int hf = warp >> 2;              // half of the row: scores, P and O columns
    const int row = wq * 32 + lane;
    const bool valid = row < rows_valid;
    const int pos = valid ? sg.q_pos0 + (r0 + row) * sg.q_pos_step : -1;
    const int row_hi = valid ? (kv_hi < 0 ? pos + 1 : min(kv_hi, pos + 1)) : 0;
    const uint32_t lane_addr = tmem_base + ((uint32_t)(wq * 32) << 16);
    const uint32_t o_col = kOCol2 + hf * (kDVH2 / 2);
    const float sl2 = p.scale_log2;
    const uint32_t bar_pf0 = peer_addr(bars + kBPF, 0), bar_pf1 = peer_addr(bars + kBPF + 1, 0);
    float* xchg = reinterpret_cast<float*>(smem + kXOff2);
    uint64_t* xb = bars + kBX + wq;
    bool ok = true;
    // exchange a per-row value with the other half (round r, two buffers): both
    // halves write, meet at the quarter's barrier, read the other's
    auto exchange = [&](float v, int r) -> float {
      float* buf = xchg + (r & 1) * 2 * BM;
      buf[hf * BM + row] = v;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(xb);
      ok = mbar_wait_warp(xb, r & 1, abort_flag, to);
      tc_fence_after();
      return buf[(hf ^ 1) * BM + row];
    };
    float m_run = -INFINITY, l_run = 0.f, m_use = 0.f;
    for (int j = 0; j < n_kv; ++j) {
      const int b = j & 1;
      ok = wait_pair_warp(bars + kBSF + b, (j >> 1) & 1, abort_flag, to);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_col = b * kBN2 + hf * (kBN2 / 2);
      float x[kBN2 / 2];
      {
        uint32_t r[kBN2 / 2];
#pragma unroll
        for (int q = 0; q < kBN2 / 64; ++q) tmem_ld32p(lane_addr + s_col + q * 32, r + q * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kBN2 / 2; ++c) x[c] = __uint_as_float(r[c]);
      }
      const int key0 = (j0 + j) * kBN2 + hf * (kBN2 / 2);
      if (key0 < win_lo || key0 + kBN2 / 2 > row_hi) {
#pragma unroll
        for (int c = 0; c < kBN2 / 2; ++c) {
          const int key = key0 + c;
          if (key < win_lo || key >= row_hi) x[c] = -INFINITY;
        }
      }
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int c = 4; c < kBN2 / 2; c += 8) {
        mx0 = fmax3(mx0, x[c], x[c + 1]);
        mx1 = fmax3(mx1, x[c + 2], x[c + 3]);
        mx2 = fmax3(mx2, x[c + 4], x[c + 5]);
        mx3 = fmax3(mx3, x[c + 6], x[c + 7]);
      }
      // the row max over both halves; the meeting also orders this half's
      // read of S before the other half's P store, which overwrites it
      float mxr = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      mxr = fmaxf(mxr, exchange(mxr, j));
      if (!ok) break;
      const float mx = mxr * sl2;
      // lazy max (see attn.cu); both halves take the same decisions
      const bool move = mx > m_run + kMaxSlack;
      const float m_new = move ? mx : m_run;
      const float m_new_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = move ? ex2_approx(m_run - m_new_use) : 1.f;
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int q = 0; q < kBN2 / 64; ++q) {
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
        // P_j as bf16 pairs over the first 64 columns of S_b: key k at column k / 2
        tmem_st16(lane_addr + b * kBN2 + hf * (kBN2 / 4) + q * 16, pk);
      }
      l_run = l_run * alpha + (sum0 + sum1);
      // P_{j-1} V_{j-1} must be done before O is rescaled; waited every tile
      // so that this barrier's phases are followed one by one
      if (j > 0) {
        ok = wait_pair_warp(bars + kBPD, (j - 1) & 1, abort_flag, to);
        if (!ok) break;
        tc_fence_after();
      }
      const bool need = (j > 0) && move;
      if (__any_sync(0xffffffffu, need)) {
        const float a = need ? alpha : 1.f;
#pragma unroll 1
        for (int q = 0; q < kDVH2 / 64; ++q) {
          uint32_t r[32];
          tmem_ld32p(lane_addr + o_col + q * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * a);
          tmem_st32(lane_addr + o_col + q * 32, r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_cluster(b ? bar_pf1 : bar_pf0);
      m_run = m_new;
      m_use = m_new_use;
    }
    // the last P V completes O
    if (ok && n_kv > 0) ok = wait_pair_warp(bars + kBPD, (n_kv - 1) & 1, abort_flag, to);
    // the row sum over both halves
    if (ok && n_kv > 0) l_run += exchange(l_run, n_kv);
    if (!ok) {
      if (lane == 0) {
        set_status(p.status, CPATTN_ERR_TIMEOUT);
        *abort_flag = 1;
        store_cluster_u32(peer_abort, 1);
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
      for (int q = 0; q < kDVH2 / 64; ++q) {
        uint32_t r[32];
        if (n_kv > 0) {
          tmem_ld32p(lane_addr + o_col + q * 32, r);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) r[c] = 0u;
        }
        if (out_row >= 0) {
          const long long off =
              (out_row * p.Hq + h) * kDV2 + half * kDVH2 + hf * (kDVH2 / 2) + q * 32;
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
      // both halves read lse_acc; only output half 0, row half 0 writes the LSE
      if (out_row >= 0 && half == 0 && hf == 0) p.lse[out_row * p.Hq + h] = mc.lse;
    }
  }

  // ---- teardown: meet, let in-flight copies land after an abort, free ----
  grid_dep_wait();  // (already returned in the epilogue unless this CTA aborted)
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs have stopped issuing copies and MMAs
  if (*abort_flag && n_kv > 0 && threadIdx.x == 0) {
    // copies issued before the abort complete on barriers that may never be
    // armed, so they cannot be waited for: give them time to land (a copy
    // takes microseconds) before either CTA releases its shared memory
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  __syncthreads();
  cluster_sync_all();  // neither CTA frees memory the other's MMAs or copies still use
  if (warp == kProducerWarp2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512)
                 : "memory");
  }
}

}  // namespace

// Launch the pair kernel for the absorbed-MLA shape (Hq even).  Same contract
// as launch_attn_mla.
int launch_attn_mla_pair(const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                         int64_t k_head_stride, int num_kv_rows, int Hkv, AttnParams prm,
                         long long tiles, cudaStream_t stream) {
  if (prm.Hq % 2 != 0) return CPATTN_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, kD2, prm.Hq, num_q_rows, kD2, (long long)prm.Hq * kD2) ||
      !make_map(&mk, k, kD2, Hkv, num_kv_rows, k_head_stride, k_row_stride, 64) ||
      !make_map(&mv, k, kD2, Hkv, num_kv_rows, k_head_stride, k_row_stride, kBN2))
    return CPATTN_ERR_CUDA;
  if (!allow_smem(attn_mla_pair_kernel, kSmem2)) return CPATTN_ERR_CUDA;
  // tiles x KV blocks (split mode) x head pairs x halves x 2 CTAs
  const long long grid = tiles * (prm.Hq / 2) * 2 * 2;
  if (grid <= 0) return CPATTN_OK;
  if (grid > 0x7fffffffLL) return CPATTN_ERR_INVALID_ARG;
  return launch_kernel(attn_mla_pair_kernel, (unsigned)grid, kThreads2, kSmem2, stream,
                       prm.pdl != 0, mq, mk, mv, prm) == cudaSuccess
             ? CPATTN_OK
             : CPATTN_ERR_CUDA;
}

}  // namespace cpattn
