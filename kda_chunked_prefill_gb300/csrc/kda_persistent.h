// Internal interface of the persistent producer/consumer kernel (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {
namespace pers {

constexpr int RING = 4;              // ring slots per consumer
constexpr int SLOT_BYTES = 82944;    // one (chain, chunk) hand-off at most, 1024-byte multiple

struct Params {
    const __nv_bfloat16 *q, *k, *v;
    const float *g, *beta;
    const int32_t *cu;
    int32_t N;
    int64_t T;
    int32_t H;
    const float *s0;
    float scale, lb;
    float *o, *sT;       // o may be NULL (nothing written but the final states)
    int32_t *status;
    unsigned char *ws;
    int32_t C;           // ring consumers (set by launch): chains go to them, tasks are numbered by them
    int32_t CH;          // consumer CTAs per ring consumer (set by launch): 2 when the 128 value
                         // columns of a chain are split over two CTAs, else 1
    int32_t Cws;         // consumers the workspace rings were sized for (>= C)
    uint32_t debug;      // KDA_DEBUG_* flags (0 in normal calls)
    int32_t raw;         // 1: g and beta are raw (activated in the producer), see kda_chunk_fwd_raw_gates
    const float *A_log;  // [H] or NULL (raw mode)
    const float *dt_bias;  // [H][128] or NULL (raw mode)
    long long spin;      // polls before a wait gives up
    const int32_t *seq_bos;  // [N] first token of each sequence, or NULL (cu[n]); with it, cu gives
                             // only the lengths and sequences may cover the same tokens
    int64_t Ttok;            // tokens in q, k, v, g, beta (bounds seq_bos ranges)
    const __nv_bfloat16 *ngate;  // [T][H][128] gate of the fused gated RMSNorm of o, or NULL (plain o)
    const float *nweight;        // [128] its per-channel weight
    float neps;                  // its epsilon
    // set by launch: a tiled tensor map of o as [Ttok][H][128] fp32 (box 32
    // channels x 1 head x 64 tokens, 128-byte swizzle), valid when o_tma is 1
    // (a plain o: given, without the gated norm)
    int32_t o_tma;
    CUtensorMap tm_o;
};

// workspace: [64-byte header][ready C*RING][freed C*RING][freed by the second column half
// C*RING] padded to 1024, then the slots
__host__ __device__ constexpr size_t ring_offset(int C) {
    return ((64 + 12 * static_cast<size_t>(C) * RING) + 1023) / 1024 * 1024;
}

int max_consumers(int64_t chains, int grid);
int consumers_for(int64_t chains, int64_t tokens, int64_t seqs, int grid);
bool wy_for(int64_t chains, int64_t tokens, int64_t seqs, int C, int grid);
bool split_for(int64_t chains, int64_t tokens, int64_t seqs, int C, int grid);
size_t workspace_bytes(int64_t chains);
cudaError_t launch(Params p, size_t ws_bytes, cudaStream_t stream);

}  // namespace pers
}  // namespace kda
