// Host-side argument checks shared by the C entry points (include/kda.h).
#pragma once
#include <stdint.h>

#include "kda.h"

namespace kda {
namespace checks {

// Most tokens a call may hold: the per-chunk tasks address tokens with 32-bit
// offsets (plus a chunk of headroom).
constexpr int64_t kMaxTokens = 0x7fffffffLL - 64;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The strip products form factors up to 2^(8 |lower_bound| / ln 2); the bound
// lies in [-10, 0) so that they stay below 2^126 (finite in bf16 and fp32)
// with a margin.
inline bool lower_bound_ok(float lb) { return lb >= -10.0f && lb < 0.0f; }

inline bool scale_ok(float s) { return s == s; }

// A host copy of cu_seqlens: starts at 0, never decreases, ends at T.
inline bool host_seqlens_ok(const int32_t *cu, int32_t N, int64_t T) {
    if (!cu || N < 0 || cu[0] != 0 || cu[N] != T) return false;
    for (int32_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return false;
    return true;
}

// The host-side checks of kda_chunk_fwd's arguments (everything but the
// workspace pair), in the order the entry point applies them: KDA_OK when the
// call may proceed (num_seqs == 0 with total_tokens == 0 included: a call with
// nothing to do), otherwise the status the entry point returns.
kda_status_t fwd_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                      int32_t head_dim_k, int32_t head_dim_v, const float *initial_state, float scale,
                      float lower_bound, const float *o, const float *final_state, const int32_t *status_dev);

}  // namespace checks
}  // namespace kda
