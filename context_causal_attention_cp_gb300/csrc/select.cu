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
