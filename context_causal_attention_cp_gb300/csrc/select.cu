// Host-side choice between the two exact ring variants of context
// parallelism: pass-KV (KV blocks travel, partials merged at the end) and
// pass-Q (query blocks travel with a carried accumulator).  Blog "什么是
// Context Parallelism", §3.5 (the pass-KV / pass-Q switch of the Meta CP
// system).  Host code only.
#include <cmath>
#include <cstdint>

#include "../../include/cpattn.h"

extern "C" int cp_select_pass(int64_t new_tokens, int64_t cached_tokens, int Hq, int Hkv,
                              int rule, double* score) {
  constexpr int64_t kMaxTokens = int64_t(1) << 40;  // keeps the integer products below 2^63
  if (new_tokens <= 0 || cached_tokens < 0 || new_tokens > kMaxTokens ||
      cached_tokens > kMaxTokens || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq > (1 << 20))
    return CPATTN_ERR_INVALID_ARG;
  const double T = (double)new_tokens, P = (double)cached_tokens;
  const double miss = T / (T + P);
  if (rule == CP_SELECT_MESSAGE) {
    // the query message of pass-Q (T rows x Hq heads) is no larger than the
    // KV message of pass-KV (T+P rows x Hkv heads, K and V)
    const double thr = 2.0 * (double)Hkv / (double)Hq;
    if (score) *score = miss - thr;
    // exact: T * Hq <= 2 * (T + P) * Hkv
    return new_tokens * Hq <= 2 * (new_tokens + cached_tokens) * Hkv ? CP_PASS_Q : CP_PASS_KV;
  }
  if (rule == CP_SELECT_FITTED) {
    const double h = -1.059 * std::log(T) + 1.145 * std::log(miss) + 12.112;
    if (score) *score = h;
    return h > 0.0 ? CP_PASS_KV : CP_PASS_Q;
  }
  return CPATTN_ERR_INVALID_ARG;
}

// Cost rule: the page's message comparison with its roofline condition laid
// over it (pass-KV is preferred when its SendRecv hides behind the hop's
// attention) and the All2All that pass-Q needs to bring its scattered partial
// results home before the LSE merge.  Times per rank of a ring of C ranks:
//   F     = 2 Hq (d + d) (T P + T (T + 1) / 2)   attention flops of the step
//   t_a   = F / C^2 / R                           attention of one hop (R: rate)
//   t_kv  = 2 ceil((T+P)/C) Hkv d 2 B / L        one pass-KV hop's K and V
//   t_q   = ceil(T/C) Hq d 2 B / L               one pass-Q hop's query block
//   t_a2a = (C-1)/C ceil(T/C) Hq (d+1) 4 B / L   pass-Q's All2All of partials
//   t_m   = C ceil(T/C) Hq (d+1) 4 B / M         pass-Q's final merge (M: rate)
//   E_kv  = (C-1) max(0, t_kv - t_a)             exposed pass-KV communication
//   E_q   = (C-1) max(0, t_q - t_a) + t_a2a + t_m
// pass-KV iff E_kv <= E_q.  Pass-KV merges each hop's partial inside the
// hop's attention, so it has no separate merge term.
extern "C" int cp_select_pass_cost(int64_t new_tokens, int64_t cached_tokens, int Hq, int Hkv,
                                   int head_dim, int cp_size, double attn_tflops,
                                   double link_gbs, double merge_gbs, double* exposed_kv_s,
                                   double* exposed_q_s) {
  constexpr int64_t kMaxTokens = int64_t(1) << 40;
  if (new_tokens <= 0 || cached_tokens < 0 || new_tokens > kMaxTokens ||
      cached_tokens > kMaxTokens || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq > (1 << 20) ||
      head_dim <= 0 || head_dim > 4096 || cp_size < 1 || cp_size > CPATTN_MAX_CP ||
      !(attn_tflops > 0.0) || !(link_gbs > 0.0) || !(merge_gbs > 0.0) ||
      !std::isfinite(attn_tflops) || !std::isfinite(link_gbs) || !std::isfinite(merge_gbs))
    return CPATTN_ERR_INVALID_ARG;
  const double T = (double)new_tokens, P = (double)cached_tokens, C = (double)cp_size;
  const double d = (double)head_dim;
  const double R = attn_tflops * 1e12, L = link_gbs * 1e9, M = merge_gbs * 1e9;
  const double t_blk = std::ceil(T / C), kv_blk = std::ceil((T + P) / C);
  const double F = 2.0 * Hq * (2.0 * d) * (T * P + T * (T + 1.0) / 2.0);
  const double t_a = F / (C * C) / R;
  const double t_kv = 2.0 * kv_blk * Hkv * d * 2.0 / L;
  const double t_q = t_blk * Hq * d * 2.0 / L;
  const double part_bytes = t_blk * Hq * (d + 1.0) * 4.0;
  const double t_a2a = (C - 1.0) / C * part_bytes / L;
  const double t_m = C * part_bytes / M;
  const double e_kv = (C - 1.0) * std::fmax(0.0, t_kv - t_a);
  const double e_q = (C - 1.0) * std::fmax(0.0, t_q - t_a) + t_a2a + t_m;
  if (exposed_kv_s) *exposed_kv_s = e_kv;
  if (exposed_q_s) *exposed_q_s = e_q;
  return e_kv <= e_q ? CP_PASS_KV : CP_PASS_Q;
}
