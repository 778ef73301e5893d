// kda_host.h -- host-side helpers shared by the C entry points: problem-size
// limits and the exception barrier in front of every call that allocates host
// memory.
#pragma once

#include <cstdint>
#include <new>

#include "../../include/kda.h"

namespace kda {

void set_last_error(const char* msg);

// Upper bounds on a problem, checked before anything is sized from it, so that no
// byte count or index product overflows 64 bits and no host table is built from an
// absurd count: at most 2^40 tokens, 2^40 token-heads and 2^20 value heads, and no
// more sequences than tokens. Expects B, T, Hv >= 1; num_seqs is 0 for the fixed
// layout. Returns a description of the first bound broken, or nullptr.
inline const char* size_limit_violation(int64_t B, int64_t T, int64_t Hv, int64_t num_seqs) {
  constexpr int64_t kMaxTokens = int64_t(1) << 40, kMaxHeads = int64_t(1) << 20;
  if (Hv > kMaxHeads) return "more than 2^20 value heads";
  if (T > kMaxTokens / B) return "more than 2^40 tokens";
  if (B * T > kMaxTokens / Hv) return "more than 2^40 token-heads";
  if (num_seqs > B * T) return "more sequences than tokens";
  return nullptr;
}

// Runs the body of a C entry point. A host exception (std::bad_alloc while
// building the launch plan, say) becomes a status and a message instead of
// crossing the C ABI, where it would end the process.
template <typename F>
kda_status guarded(F&& body) {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    set_last_error("host memory exhausted while validating or planning the call");
    return KDA_ERR_INVALID_ARGUMENT;
  } catch (...) {
    set_last_error("unexpected host-side exception");
    return KDA_ERR_INVALID_ARGUMENT;
  }
}

}  // namespace kda
