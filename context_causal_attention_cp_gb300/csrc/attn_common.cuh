// Shared pieces of the shard-attention kernels (sm_103a): launch parameters,
// bounded warp-uniform waits, TMEM and packed-fp32 helpers, work-item
// resolution and tensor-map encoding.
#pragma once
#include <utility>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "../../include/cpattn.h"
#include "ptx.cuh"

namespace cpattn {

constexpr int BM = CPATTN_TILE_ROWS;  // query rows per tile (MMA M)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kMaxSlack = 8.0f;  // lazy-rescale threshold, log2 units

struct AttnParams {
  const cp_segment_t* segs;
  const int32_t* tiles;
  int num_segs, num_tiles;
  int Hq, g, n_hgroups;
  float scale_log2;
  int kv_lo, kv_hi;
  void* o;
  int o_f32;
  float* lse;
  int out_row_base, num_out_rows, num_q_rows, num_kv_rows;
  int32_t* status;
  unsigned long long timeout_ns;
  int withhold_q;  // test hook: the producer skips the Q load (see cp_attn_debug)
  // split-KV mode (cp_attn_partial_kv): split_block > 0 splits every segment's
  // keys into blocks [j*split_block, (j+1)*split_block); the CTA for block j
  // writes its fp32 partial at workspace row ws_slot[seg] + j*q_len + row.
  int split_block, max_blocks;
  const long long* ws_slot;
  long long ws_rows;  // capacity of the partial buffers, rows
  const void* q;      // query rows (read directly by kernels that stage part of Q in TMEM)
  // Output placement and mode of the normal (non-split) path:
  //   dst_rows: when set, query row i writes output row dst_rows[i] (the
  //     restore scatter done by the store), which must lie in [0, dst_limit);
  //     then out_row_base = 0 and num_out_rows = num_q_rows.  Otherwise row i
  //     writes row i - out_row_base.
  //   lse_acc: when set, the store merges this call's partial into the fp32 O
  //     already at the output row, whose LSE is lse_acc[row], by the pairwise
  //     log-sum-exp rule: merged O in place, merged LSE to lse.
  const int32_t* dst_rows;
  long long dst_limit;
  const float* lse_acc;
  // q_token_rows: query and output rows are token (flat) indices: segment row
  // i reads query row tok0 + i and writes output row tok0 + i (the shard
  // gather and the restore both done by the kernel's own loads and stores);
  // every segment must be a run of consecutive tokens (q_pos_step == 1).
  int q_token_rows;
  // seg_windows (normal mode): when set, segment s uses the key window
  // [seg_windows[2s], seg_windows[2s+1]) in place of the call's kv_lo / kv_hi
  // (an upper end < 0 is unbounded), so that one launch can merge every
  // segment against its own resident KV block (the pass-Q ring hop).
  const int32_t* seg_windows;
  // pack_heads (d = 64 / 128 kernel, two query tiles per CTA): every segment
  // has at most BM / 2 rows, and each 128-row tile holds two query heads:
  // tile row r is query row r % (BM / 2) of head 2 * tile + r / (BM / 2)
  // within the CTA's head group (which then spans 4 heads).  The Q tensor map
  // then has boxes of BM / 2 rows.  A longer segment sets CPATTN_ERR_RANGE.
  int pack_heads;
  // pdl (host side): launch with programmatic stream serialization, so that
  // the kernel's set-up and main loop overlap the kernel before it on the
  // stream (split-KV mode, where that kernel writes only the slot table read
  // by split_slot_row0).
  int pdl;
};

// Number of split_block-key blocks a segment sees (key 0 is always visible).
__host__ __device__ __forceinline__ int segment_blocks(const cp_segment_t& s, int split_block) {
  const long long last = (long long)s.q_pos0 + (long long)(s.q_len - 1) * s.q_pos_step;
  return (int)(last / split_block) + 1;
}

// Host-side settings of the test hook (cp_attn_debug); defaults: 4 s, off.
struct AttnDebug {
  unsigned long long timeout_ns = 4000000000ull;
  int withhold_q = 0;
};
AttnDebug& attn_debug();

// Warp-uniform bounded wait: every lane polls, the give-up decision is lane 0's.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               const volatile int* abort, uint64_t timeout) {
  const int lane = threadIdx.x & 31;
  uint64_t t0 = lane == 0 ? global_timer_ns() : 0;
  for (uint32_t i = 0;; ++i) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((i & 63u) == 63u) {
      int give_up = 0;
      if (lane == 0) give_up = (*abort != 0) || (global_timer_ns() - t0 > timeout);
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
    }
  }
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld32p(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

// Three-input maximum (sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Paired fp32 FMA and add (one instruction for two lanes of work, sm_100+).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Resolve this CTA's query tile (segment, tile-in-segment) and check the
// segment against the buffers.  Returns false (the whole CTA returns) when
// there is no work or the metadata is out of range (then CPATTN_ERR_RANGE).
__device__ __forceinline__ bool resolve_tile(const AttnParams& p, int tile_idx, cp_segment_t& sg,
                                             int& t, int& seg_id) {
  seg_id = -1;
  t = 0;
  if (p.tiles) {
    if (tile_idx >= p.num_tiles) return false;
    seg_id = __ldg(p.tiles + 2 * tile_idx);
    t = __ldg(p.tiles + 2 * tile_idx + 1);
    if (seg_id < 0 || seg_id >= p.num_segs) {
      if (threadIdx.x == 0) set_status(p.status, CPATTN_ERR_RANGE);
      return false;
    }
  } else {
    int acc = 0;
    for (int s = 0; s < p.num_segs; ++s) {
      const int ql = __ldg(&p.segs[s].q_len);
      const int nt = ql > 0 ? (ql + BM - 1) / BM : 0;
      if (tile_idx < acc + nt) {
        seg_id = s;
        t = tile_idx - acc;
        break;
      }
      acc += nt;
    }
    if (seg_id < 0) return false;
  }
  sg = p.segs[seg_id];
  bool not_run = false;
  if (p.q_token_rows) {  // rows of a consecutive token run, addressed by token index
    not_run = sg.q_pos_step != 1;
    sg.q_row0 = sg.tok0;
  }
  const long long last_pos = (long long)sg.q_pos0 + (long long)(sg.q_len - 1) * sg.q_pos_step;
  const bool bad = not_run || sg.q_len <= 0 || sg.q_row0 < 0 ||
                   (long long)sg.q_row0 + sg.q_len > p.num_q_rows || sg.q_pos0 < 0 ||
                   sg.q_pos_step < 0 || sg.kv_row0 < 0 ||
                   (long long)sg.kv_row0 + sg.kv_len > p.num_kv_rows ||
                   (long long)sg.q_row0 - p.out_row_base < 0 ||
                   (long long)sg.q_row0 + sg.q_len - p.out_row_base > p.num_out_rows ||
                   last_pos + 1 > sg.kv_len || t < 0 || (long long)t * BM >= sg.q_len;
  if (bad) {
    if (threadIdx.x == 0) set_status(p.status, CPATTN_ERR_RANGE);
    return false;
  }
  return true;
}

// The key window and output placement of this CTA.  Normal mode: the call's
// window (or the segment's own, with seg_windows), output row = cat row -
// out_row_base.  Split-KV mode: block j of the
// segment's keys, output row = ws_slot[seg] + j * q_len + row-in-segment.
// Returns false when the CTA has no block to do.
__device__ __forceinline__ bool split_window(const AttnParams& p, const cp_segment_t& sg, int seg_id,
                                             int j, int& kv_lo, int& kv_hi, long long& out_row0) {
  if (p.split_block <= 0) {
    if (p.seg_windows) {
      kv_lo = __ldg(p.seg_windows + 2 * seg_id);
      kv_hi = __ldg(p.seg_windows + 2 * seg_id + 1);
    } else {
      kv_lo = p.kv_lo;
      kv_hi = p.kv_hi;
    }
    out_row0 = (long long)sg.q_row0 - p.out_row_base;  // output row of segment row 0
    return true;
  }
  const int nb = segment_blocks(sg, p.split_block);
  if (j >= nb) return false;
  if (nb > p.max_blocks) {
    if (threadIdx.x == 0) set_status(p.status, CPATTN_ERR_INVALID_ARG);
    return false;
  }
  kv_lo = j * p.split_block;
  kv_hi = kv_lo + p.split_block;
  out_row0 = -1;  // the workspace slot is read by split_slot_row0 before the store
  return true;
}

// Split-KV mode: workspace row of segment row 0 of block j, read from the
// slot table that the layout kernel before this launch writes (the launch may
// overlap that kernel, so the read waits for it), or -1 with CPATTN_ERR_RANGE
// when the slot is out of range.  Normal mode: out_row0 unchanged.
__device__ __forceinline__ long long split_slot_row0(const AttnParams& p, const cp_segment_t& sg,
                                                     int seg_id, int j, long long out_row0) {
  if (p.split_block <= 0) return out_row0;
  grid_dep_wait();
  const long long r = p.ws_slot[seg_id] + (long long)j * sg.q_len;
  if (r < 0 || r + sg.q_len > p.ws_rows) {
    set_status(p.status, CPATTN_ERR_RANGE);
    return -1;
  }
  return r;
}

// Output row of row `row` of query tile r0 of segment sg (normal mode), or -1
// with CPATTN_ERR_RANGE when the destination index is out of range.
__device__ __forceinline__ long long output_row(const AttnParams& p, const cp_segment_t& sg,
                                                int r0, int row, long long out_row0) {
  if (out_row0 < 0) return -1;  // split-KV slot out of range (status already set)
  if (!p.dst_rows) return out_row0 + r0 + row;
  const long long d = __ldg(p.dst_rows + sg.q_row0 + r0 + row);
  if (d < 0 || d >= p.dst_limit) {
    set_status(p.status, CPATTN_ERR_RANGE);
    return -1;
  }
  return d;
}

// Pairwise log-sum-exp merge of the store in accumulate mode.  This call's
// partial for a row is (acc / l_run, n) with n = m_use + log2(l_run) in log2
// units (no visible key: n = -inf); the accumulator holds (O_old, L_old) with
// L_old a natural log.  With m = max, w_old = 2^(L_old*log2e - m) and
// w_new = 2^(n - m): O = (w_old O_old + w_new acc / l_run) / (w_old + w_new),
// L = (m + log2(w_old + w_new)) ln 2.  Both sides empty: O = 0, L = -inf.
struct MergeCoef {
  float c_old, c_new, lse;  // O = c_old * O_old + c_new * acc
};
__device__ __forceinline__ MergeCoef merge_coef(float l_old, bool has, float m_use, float l_run) {
  const float n2 = has ? m_use + lg2_approx(l_run) : -INFINITY;
  const float o2 = l_old * kLog2e;
  const float m = fmaxf(n2, o2);
  MergeCoef c;
  if (m == -INFINITY) {
    c.c_old = 0.f;
    c.c_new = 0.f;
    c.lse = -INFINITY;
    return c;
  }
  const float wo = ex2_approx(o2 - m), wn = ex2_approx(n2 - m);
  const float iw = 1.f / (wo + wn);
  c.c_old = wo * iw;
  c.c_new = has ? wn * iw * (1.f / l_run) : 0.f;
  c.lse = (m + lg2_approx(wo + wn)) * kLn2;
  return c;
}

// ------------------------------------------------------------------- host --
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D bf16 map (cols, heads, rows) with a 64-column x 1-head x 128-row box,
// 128-byte swizzle; out-of-range rows read as zero.
inline bool make_map(CUtensorMap* m, const void* base, int cols, int heads, long long rows,
                     long long head_stride_el, long long row_stride_el, int box_rows = 128) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)(head_stride_el * 2), (cuuint64_t)(row_stride_el * 2)};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


inline bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Opt `kern` in to `smem` bytes of dynamic shared memory.  The attribute
// belongs to the CUDA context that is current, so it is set on every launch
// (a host-side call of about a microsecond): a new context on the device
// (after cudaDeviceReset, or a caller's own context) never sees a launch
// without it.
template <typename... Params>
inline bool allow_smem(void (*kern)(Params...), int smem) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
         cudaSuccess;
}

// Launch `kern` on `stream`, with programmatic stream serialization when pdl
// is set (the kernel may then start before the previous kernel on the stream
// has finished; see grid_dep_wait).
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(Params...), unsigned grid, unsigned block,
                                 size_t smem, cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Absorbed-MLA variant (d = 576, dv = 512 with V the first 512 columns of K);
// defined in attn_mla.cu.
int launch_attn_mla(const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                    int64_t k_head_stride, int num_kv_rows, int Hkv, AttnParams prm,
                    long long tiles, cudaStream_t stream);

// Shared host front end of cp_attn_partial and cp_attn_partial_kv: validates
// the shape arguments, fills prm (everything but the split fields and the
// output pointers) and launches the kernel for the shape.
int attn_launch(const cp_segment_t* segs_dev, int num_segs, const int32_t* tiles_dev, int num_tiles,
                const void* q, int num_q_rows, const void* k, int64_t k_row_stride,
                int64_t k_head_stride, const void* v, int64_t v_row_stride, int64_t v_head_stride,
                int num_kv_rows, int Hq, int Hkv, int d, int dv, float scale, AttnParams& prm,
                cudaStream_t stream);

}  // namespace cpattn
