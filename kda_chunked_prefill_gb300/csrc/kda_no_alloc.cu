// kda_chunk_fwd_static_scratch: the chunked-prefill forward for callers that
// cannot allocate device memory at all.
//
// kda_chunk_fwd itself allocates nothing, but it needs a scratch workspace that
// the caller must provide. Some callers cannot produce one: a runtime whose
// device memory is a fixed arena planned before the model starts, an embedded
// or real-time host that forbids allocation after start-up, or a plugin that is
// handed its input and output tensors but no way to request memory. For them
// this entry point takes its scratch from a fixed array compiled into the
// library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds KDA_STATIC_SCRATCH_BYTES of it until the process exits. In host
// code the array's name only stands in for the symbol; its device address is
// looked up with cudaGetSymbolAddress on every call, with the call's device
// current, and passed to the kernel. (A cached address would go stale when the
// device's primary context is reset and the module reloaded at a new address;
// the lookup is a cheap query once the module is loaded.)
#include <cuda_runtime.h>

#include "kda.h"

#include "kda_checks.h"

static __device__ __align__(256) unsigned char kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

extern "C" kda_status_t kda_chunk_fwd_static_scratch(
    const void *q, const void *k, const void *v, const float *g, const float *beta,
    const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
    int32_t head_dim_k, int32_t head_dim_v, const float *initial_state, float scale,
    float lower_bound, float *o, float *final_state, int32_t *status_dev, kda_stream_t stream) {
    // the same argument checks, in the same order, as kda_chunk_fwd
    const kda_status_t args = kda::checks::fwd_args(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                                                    head_dim_k, head_dim_v, initial_state, scale, lower_bound, o,
                                                    final_state, status_dev);
    if (args != KDA_OK) return args;
    if (num_seqs == 0) return KDA_OK;  // nothing to schedule
    const size_t need = kda_chunk_fwd_workspace_size(num_seqs, num_heads);
    if (need == 0) return KDA_ERR_CUDA;  // no usable device is current
    if (need > static_cast<size_t>(KDA_STATIC_SCRATCH_BYTES)) return KDA_ERR_SCRATCH_TOO_SMALL;
    void *scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, kda_static_scratch) != cudaSuccess || !scratch) return KDA_ERR_CUDA;
    // kda_chunk_fwd clears the scratch's flag area on the stream before its launch,
    // so nothing left in the array by an earlier call is read as valid.
    return kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k,
                         head_dim_v, initial_state, scale, lower_bound, o, final_state, status_dev,
                         scratch, static_cast<size_t>(KDA_STATIC_SCRATCH_BYTES), stream);
}
