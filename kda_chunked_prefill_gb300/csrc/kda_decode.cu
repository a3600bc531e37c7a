// kda_decode_fwd: the KDA recurrence for a few tokens per sequence (decode /
// recurrent step), state in and out. The recurrence is the token form of "在 TPU
// 上加速 Kimi K3 KDA" (junyi.dev tpu-kda report) §1-§2, applied one token after
// the other; the decode step itself, with the state kept on chip for the whole
// call, is the one of "Kimi K3 на графических процессорах AMD Instinct" §1.2-§1.3
// (fused decode; the convolution and norm fused there are outside this call):
//     S <- Diag(e^{g_t}) S ;  S <- S + beta_t k_t (v_t^T - k_t^T S) ;  o_t = scale S^T q_t
//
// One CTA per (sequence, head, quarter of the value columns): 128 threads,
// warp w holding key rows 32w..32w+31 and lane l value column 32*quarter + l of
// the fp32 state in registers, so that state loads and stores are coalesced
// 128-byte rows. The two contractions over the key channel (k^T S and q^T S)
// are per-thread sums over 32 rows plus a 4-way sum across the warps. The
// state is read once and written once per call; everything runs in fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
namespace dec {

constexpr int THREADS = 128;

__global__ void __launch_bounds__(THREADS) kda_decode_kernel(const __nv_bfloat16 *__restrict__ q,
                                                             const __nv_bfloat16 *__restrict__ k,
                                                             const __nv_bfloat16 *__restrict__ v,
                                                             const float *__restrict__ g, const float *__restrict__ beta,
                                                             int32_t tokens_per_seq, int32_t H, const float *s0,
                                                             float *sT, float *__restrict__ o, float scale, float lb,
                                                             int32_t *status) {
    __shared__ float sk[DK], sq[DK], sd[DK], sv[32], part[4][32];
    __shared__ float sbeta;
    const int quarter = blockIdx.x & 3;
    const int chain = blockIdx.x >> 2;  // n * H + h
    const int n = chain / H, h = chain % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int col = 32 * quarter + lane;
    const size_t sbase = static_cast<size_t>(chain) * (DK * DV);

    float S[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) S[r] = s0 ? s0[sbase + static_cast<size_t>(32 * warp + r) * DV + col] : 0.f;

    bool gate_bad = false;
    for (int t = 0; t < tokens_per_seq; ++t) {
        const size_t tok = static_cast<size_t>(n) * tokens_per_seq + t;
        const size_t row = (tok * H + h) * DK;
        {  // this token's key-channel vectors (thread tid = channel tid) and value slice
            const float gg = g[row + tid];
            gate_bad |= !(gg >= lb && gg <= 0.f);
            sd[tid] = __expf(gg);
            sk[tid] = __bfloat162float(k[row + tid]);
            sq[tid] = __bfloat162float(q[row + tid]);
            if (tid < 32) sv[tid] = __bfloat162float(v[row + 32 * quarter + tid]);
            if (tid == 0) sbeta = beta[tok * H + h];
        }
        __syncthreads();
        // decay, then a = k^T S (over this thread's 32 rows, then across warps)
        float a = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            S[r] *= sd[32 * warp + r];
            a = fmaf(sk[32 * warp + r], S[r], a);
        }
        part[warp][lane] = a;
        __syncthreads();
        a = part[0][lane] + part[1][lane] + part[2][lane] + part[3][lane];
        const float coef = sbeta * (sv[lane] - a);
        float oc = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            S[r] = fmaf(sk[32 * warp + r], coef, S[r]);
            oc = fmaf(sq[32 * warp + r], S[r], oc);
        }
        __syncthreads();  // every thread has read part[] for a
        part[warp][lane] = oc;
        __syncthreads();
        if (warp == 0) o[row + col] = scale * (part[0][lane] + part[1][lane] + part[2][lane] + part[3][lane]);
        __syncthreads();  // the next token rewrites the shared vectors
    }
    if (sT) {
#pragma unroll
        for (int r = 0; r < 32; ++r) sT[sbase + static_cast<size_t>(32 * warp + r) * DV + col] = S[r];
    }
    if (gate_bad) set_status(status, KDA_ERR_GATE_RANGE);
}

}  // namespace dec
}  // namespace kda

namespace {
bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
}  // namespace

extern "C" kda_status_t kda_decode_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                       int32_t num_seqs, int32_t tokens_per_seq, int32_t num_heads,
                                       int32_t head_dim_k, int32_t head_dim_v, const float *initial_state,
                                       float scale, float lower_bound, float *o, float *final_state,
                                       int32_t *status_dev, kda_stream_t stream) {
    if (head_dim_k != KDA_HEAD_DIM || head_dim_v != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads < 1 || tokens_per_seq < 0 || tokens_per_seq > KDA_DECODE_MAX_TOKENS)
        return KDA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(num_seqs) * num_heads * 4 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    if (!(scale == scale) || !(lower_bound >= -10.0f && lower_bound < 0.0f)) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0) return KDA_OK;
    if (tokens_per_seq > 0) {
        if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
        if (!aligned_to(q, 16) || !aligned_to(k, 16) || !aligned_to(v, 16) || !aligned_to(g, 16) ||
            !aligned_to(o, 16) || !aligned_to(beta, 4))
            return KDA_ERR_INVALID_ARG;
    }
    if ((initial_state && !aligned_to(initial_state, 16)) || (final_state && !aligned_to(final_state, 16)) ||
        (status_dev && !aligned_to(status_dev, 4)))
        return KDA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    const int grid = num_seqs * num_heads * 4;
    kda::dec::kda_decode_kernel<<<grid, kda::dec::THREADS, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, tokens_per_seq, num_heads, initial_state, final_state, o,
        scale, lower_bound, status_dev);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
