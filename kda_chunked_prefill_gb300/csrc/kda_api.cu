// Host side of the C ABI declared in include/kda.h: argument validation,
// status zeroing and the launch of the chunked-prefill kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

#include "kda_checks.h"
#include "kda_persistent.h"

namespace {

constexpr int32_t kVersion = 100;  // 0.1.0
using kda::checks::aligned;

}  // namespace

namespace kda {
namespace checks {
kda_status_t fwd_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                      int32_t head_dim_k, int32_t head_dim_v, const float *initial_state, float scale,
                      float lower_bound, const float *o, const float *final_state, const int32_t *status_dev) {
    if (head_dim_k != KDA_HEAD_DIM || head_dim_v != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || num_heads < 1) return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_seqs) * num_heads > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (total_tokens > (int64_t{1} << 40) / (static_cast<int64_t>(num_heads) * KDA_HEAD_DIM))
        return KDA_ERR_INVALID_ARG;
    if (total_tokens > kMaxTokens) return KDA_ERR_UNSUPPORTED;  // task token offsets are 32-bit
    if (!scale_ok(scale) || !lower_bound_ok(lower_bound)) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (!cu_seqlens || !aligned(cu_seqlens, 4)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(o, 16) ||
            !aligned(beta, 4))
            return KDA_ERR_INVALID_ARG;
    }
    if ((initial_state && !aligned(initial_state, 16)) || (final_state && !aligned(final_state, 16)) ||
        (status_dev && !aligned(status_dev, 4)))
        return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}
}  // namespace checks
}  // namespace kda

namespace {
// The options the entry points add to the plain forward.
struct Extras {
    uint32_t debug = 0;                 // KDA_DEBUG_* flags
    bool raw = false;                   // g and beta are raw projections (kda_chunk_fwd_raw_gates)
    const float *A_log = nullptr, *dt_bias = nullptr;
    const void *norm_gate = nullptr;    // gated RMSNorm of o (kda_chunk_fwd_gated_norm)
    const float *norm_weight = nullptr;
    float norm_eps = 0.f;
};

kda_status_t fwd_impl(const void *q, const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                      int32_t head_dim_k, int32_t head_dim_v, const float *initial_state, float scale,
                      float lower_bound, float *o, float *final_state, int32_t *status_dev, void *workspace,
                      size_t workspace_bytes, kda_stream_t stream, const Extras &x = Extras()) {
    const float *A_log = x.A_log, *dt_bias = x.dt_bias;
    if (x.norm_gate || x.norm_weight) {
        if (!x.norm_gate || !x.norm_weight || !aligned(x.norm_gate, 16) || !aligned(x.norm_weight, 16))
            return KDA_ERR_INVALID_ARG;
        if (!(x.norm_eps > 0.f && x.norm_eps < 3.0e38f)) return KDA_ERR_INVALID_ARG;
    }
    const kda_status_t args = kda::checks::fwd_args(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                                                    head_dim_k, head_dim_v, initial_state, scale, lower_bound, o,
                                                    final_state, status_dev);
    if (args != KDA_OK) return args;
    if (num_seqs == 0) return KDA_OK;
    if ((A_log && !aligned(A_log, 4)) || (dt_bias && !aligned(dt_bias, 16))) return KDA_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 16)) return KDA_ERR_INVALID_ARG;
    const size_t need = kda::pers::workspace_bytes(static_cast<int64_t>(num_seqs) * num_heads);
    if (need == 0) return KDA_ERR_CUDA;
    if (workspace_bytes < need) return KDA_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int32_t), s) != cudaSuccess)
        return KDA_ERR_CUDA;
    kda::pers::Params p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = g;
    p.beta = beta;
    p.cu = cu_seqlens;
    p.N = num_seqs;
    p.T = total_tokens;
    p.seq_bos = nullptr;
    p.Ttok = total_tokens;
    p.H = num_heads;
    p.s0 = initial_state;
    p.scale = scale;
    p.lb = lower_bound;
    p.o = o;
    p.sT = final_state;
    p.status = status_dev;
    p.ws = static_cast<unsigned char *>(workspace);
    p.C = 0;
    p.debug = x.debug;
    p.spin = 0;
    p.raw = x.raw ? 1 : 0;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.ngate = static_cast<const __nv_bfloat16 *>(x.norm_gate);
    p.nweight = x.norm_weight;
    p.neps = x.norm_eps;
    const cudaError_t e = kda::pers::launch(p, workspace_bytes, s);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

extern "C" {

kda_status_t kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                           int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                           int32_t head_dim_v, const float *initial_state, float scale,
                           float lower_bound, float *o, float *final_state,
                           int32_t *status_dev, void *workspace, size_t workspace_bytes,
                           kda_stream_t stream) {
    return fwd_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k, head_dim_v,
                    initial_state, scale, lower_bound, o, final_state, status_dev, workspace, workspace_bytes,
                    stream);
}

kda_status_t kda_chunk_fwd_plan(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t num_sms,
                                int32_t plain_device_o, int32_t *consumers, int32_t *wy_on_consumers,
                                int32_t *split_columns) {
    if (num_seqs < 1 || num_heads < 1 || total_tokens < 0 || num_sms < 0 || !consumers || !wy_on_consumers ||
        !split_columns)
        return KDA_ERR_INVALID_ARG;
    int sms = num_sms;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return KDA_ERR_CUDA;
        }
    }
    if (sms < 2) return KDA_ERR_UNSUPPORTED;
    // the same two choices the launch makes (one CTA per SM)
    const int64_t chains = static_cast<int64_t>(num_seqs) * num_heads;
    const int C = kda::pers::consumers_for(chains, total_tokens, num_seqs, sms);
    const bool split = kda::pers::split_for(chains, total_tokens, num_seqs, C, sms);
    *consumers = split ? static_cast<int32_t>(chains) : C;
    *split_columns = split ? 1 : 0;
    *wy_on_consumers = (!split && plain_device_o && kda::pers::wy_for(chains, total_tokens, num_seqs, C, sms)) ? 1 : 0;
    return KDA_OK;
}

kda_status_t kda_chunk_fwd_debug(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                                 int32_t head_dim_v, const float *initial_state, float scale,
                                 float lower_bound, float *o, float *final_state,
                                 int32_t *status_dev, void *workspace, size_t workspace_bytes,
                                 kda_stream_t stream, uint32_t debug_flags) {
    constexpr uint32_t known = KDA_DEBUG_WITHHOLD_READY | KDA_DEBUG_WY_PRODUCER | KDA_DEBUG_WY_CONSUMER |
                               KDA_DEBUG_SPLIT_COLUMNS | KDA_DEBUG_WHOLE_COLUMNS;
    auto both = [&](uint32_t a, uint32_t b) { return (debug_flags & a) && (debug_flags & b); };
    if ((debug_flags & ~known) || both(KDA_DEBUG_WY_PRODUCER, KDA_DEBUG_WY_CONSUMER) ||
        both(KDA_DEBUG_SPLIT_COLUMNS, KDA_DEBUG_WHOLE_COLUMNS) || both(KDA_DEBUG_SPLIT_COLUMNS, KDA_DEBUG_WY_CONSUMER))
        return KDA_ERR_INVALID_ARG;
    Extras x;
    x.debug = debug_flags;
    return fwd_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k, head_dim_v,
                    initial_state, scale, lower_bound, o, final_state, status_dev, workspace, workspace_bytes,
                    stream, x);
}

kda_status_t kda_chunk_fwd_raw_gates(const void *q, const void *k, const void *v, const float *g_raw,
                                     const float *beta_raw, const float *A_log, const float *dt_bias,
                                     const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                     int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                     const float *initial_state, float scale, float lower_bound, float *o,
                                     float *final_state, int32_t *status_dev, void *workspace,
                                     size_t workspace_bytes, kda_stream_t stream) {
    Extras x;
    x.raw = true;
    x.A_log = A_log;
    x.dt_bias = dt_bias;
    return fwd_impl(q, k, v, g_raw, beta_raw, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k,
                    head_dim_v, initial_state, scale, lower_bound, o, final_state, status_dev, workspace,
                    workspace_bytes, stream, x);
}

kda_status_t kda_chunk_fwd_gated_norm(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                      int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                                      int32_t head_dim_v, const float *initial_state, float scale,
                                      float lower_bound, const void *gate, const float *norm_weight,
                                      float norm_eps, float *o, float *final_state, int32_t *status_dev,
                                      void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    if (!gate || !norm_weight) return KDA_ERR_INVALID_ARG;
    Extras x;
    x.norm_gate = gate;
    x.norm_weight = norm_weight;
    x.norm_eps = norm_eps;
    return fwd_impl(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k, head_dim_v,
                    initial_state, scale, lower_bound, o, final_state, status_dev, workspace, workspace_bytes,
                    stream, x);
}

size_t kda_chunk_fwd_workspace_size(int32_t num_seqs, int32_t num_heads) {
    if (num_seqs < 1 || num_heads < 1) return 0;
    return kda::pers::workspace_bytes(static_cast<int64_t>(num_seqs) * num_heads);
}

int32_t kda_chunk_fwd_launches(int32_t num_seqs, int64_t total_tokens, int32_t num_heads) {
    (void)total_tokens;
    return (num_seqs > 0 && num_heads > 0) ? 1 : 0;
}

const char *kda_status_string(int32_t status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported head dimension (only 128 is built)";
        case KDA_ERR_CUDA: return "CUDA runtime or launch error";
        case KDA_ERR_GATE_RANGE: return "gate g outside [lower_bound, 0] or not finite";
        case KDA_ERR_BAD_SEQLENS: return "cu_seqlens not nondecreasing from 0 to total_tokens";
        case KDA_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
        case KDA_ERR_VALUE_RANGE: return "a value entering an fp16 tensor-core operand exceeded 6e4 or was not finite";
        case KDA_ERR_SCRATCH_TOO_SMALL: return "problem needs more scratch than the static scratch array holds";
        case KDA_ERR_BOUNDS: return "an index checked before a global-memory access was out of bounds (KDA_DEBUG_BOUNDS build)";
        default: return "unknown status";
    }
}

int32_t kda_version(void) { return kVersion; }

}  // extern "C"
