// Host mirror of the shard plan's segment table.
//
// cp_shard_plan builds the plan on the device; several host entry points
// (workspace sizing, the pass-Q ring schedule, the host-to-host prefill)
// need the same segments on the host before anything is launched.  This
// enumerator produces them in the table order of cp_shard_plan (rank by rank;
// within a rank request by request, zigzag early block before late block) and
// with the same field values.  Zigzag: SGLang docs, "Prefill Context
// Parallelism", §Zigzag strategy (2C blocks per request, early blocks take
// the remainder, rank r takes blocks r and 2C-1-r); interleave: same page,
// §Interleave strategy (flat index i on rank i mod C, positions kept).
#pragma once
#include <cstdint>

#include "../../include/cpattn.h"

namespace cpattn {

// Calls fn(rank, segment) for every segment of the plan, in table order.
// Returns CPATTN_OK, or CPATTN_ERR_INVALID_ARG for bad arguments or totals
// that do not fit the plan's int32 fields.
template <class F>
int for_each_plan_segment(const int32_t* new_lens, const int32_t* prefix_lens, int num_reqs,
                          int cp_size, int strategy, F&& fn) {
  if (num_reqs < 0 || num_reqs > CPATTN_MAX_REQS || cp_size < 1 || cp_size > CPATTN_MAX_CP)
    return CPATTN_ERR_INVALID_ARG;
  if (strategy != CP_ZIGZAG && strategy != CP_INTERLEAVE) return CPATTN_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!new_lens || !prefix_lens)) return CPATTN_ERR_INVALID_ARG;
  long long tot_new = 0, tot_kv = 0;
  for (int b = 0; b < num_reqs; ++b) {
    if (new_lens[b] < 0 || prefix_lens[b] < 0) return CPATTN_ERR_INVALID_ARG;
    tot_new += new_lens[b];
    tot_kv += (long long)new_lens[b] + prefix_lens[b];
  }
  if (tot_new > 0x7fffffffLL || tot_kv > 0x7fffffffLL) return CPATTN_ERR_INVALID_ARG;
  const long long C = cp_size;
  long long row_base = 0;
  for (long long r = 0; r < C; ++r) {
    long long flat0 = 0, kv0 = 0, row_in_rank = 0;
    for (int b = 0; b < num_reqs; ++b) {
      const long long n = new_lens[b], p = prefix_lens[b];
      if (strategy == CP_ZIGZAG) {
        const long long nb = 2 * C, base = n / nb, rem = n % nb, kl = nb - 1 - r;
        const long long e = base + (r < rem), l = base + (kl < rem);
        const long long st_e = r * base + (r < rem ? r : rem);
        const long long st_l = kl * base + (kl < rem ? kl : rem);
        if (e > 0)
          fn((int)r, cp_segment_t{(int32_t)(row_base + row_in_rank), (int32_t)e, (int32_t)(p + st_e),
                                  1, (int32_t)kv0, (int32_t)(p + st_e + e),
                                  (int32_t)(flat0 + st_e), (int32_t)b});
        if (l > 0)
          fn((int)r, cp_segment_t{(int32_t)(row_base + row_in_rank + e), (int32_t)l,
                                  (int32_t)(p + st_l), 1, (int32_t)kv0, (int32_t)(p + st_l + l),
                                  (int32_t)(flat0 + st_l), (int32_t)b});
        row_in_rank += e + l;
      } else {
        const long long i0 = flat0 + (((r - flat0 % C) % C) + C) % C;
        const long long cnt = (i0 < flat0 + n) ? (flat0 + n - 1 - i0) / C + 1 : 0;
        if (cnt > 0) {
          const long long last = i0 + (cnt - 1) * C;
          fn((int)r, cp_segment_t{(int32_t)(row_base + (i0 - r) / C), (int32_t)cnt,
                                  (int32_t)(p + (i0 - flat0)), (int32_t)C, (int32_t)kv0,
                                  (int32_t)(p + (last - flat0) + 1), (int32_t)i0, (int32_t)b});
        }
        row_in_rank += cnt;
      }
      flat0 += n;
      kv0 += n + p;
    }
    row_base += row_in_rank;
  }
  return CPATTN_OK;
}

// Last position of a segment's rows.
inline long long segment_last_pos(const cp_segment_t& s) {
  return (long long)s.q_pos0 + (long long)(s.q_len - 1) * s.q_pos_step;
}

}  // namespace cpattn
