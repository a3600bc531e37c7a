// Split-sequence scan: kda_chunk_fwd for calls whose few, long (sequence, head)
// chains would otherwise run one chunk after another on a handful of SMs.
//
// A segment of a sequence maps its entry state to its exit state affinely,
// S_out = Phi S_in + N (the chunk recurrence of "在 TPU 上加速 Kimi K3 KDA" §6.2
// is affine in S, so a run of chunks is too). By linearity N is the exit state
// from a zero entry state and Phi + N the exit state from the identity. So:
//   pass 1  one launch of the chunked kernel over the segments except each
//           split sequence's last: segment 0 from the sequence's own entry
//           state, the others twice (from I and from 0), states only (no o);
//   combine S_1 = exit of segment 0, S_{s+1} = (F_s - N_s) S_s + N_s, per
//           (sequence, head, 16-column block) in fp32;
//   pass 3  one launch over every segment as a sequence of its own, with entry
//           states S_s, writing o and the segments' exit states;
//   gather  each sequence's last exit state into final_state.
// Pass 1 lists its segments through a token-offset map (a segment appears twice
// over the same tokens); pass 3 partitions the tokens in order.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "kda.h"

#include "kda_checks.h"
#include "kda_persistent.h"

namespace kda {
namespace split {

constexpr int BT = 64, DK = 128, DV = 128;
constexpr size_t STATE = static_cast<size_t>(DK) * DV;  // floats per (sequence, head) state
constexpr int MAX_SEGMENTS = 64;                        // per sequence
using checks::kMaxTokens;

// Measured paces of the chunked kernel on GB300 (the same model picks its
// consumer count): a busy consumer finishes a chunk every 3.5 us, a producer
// every 7.0 us; a launch and its ramp cost about 15 us.
constexpr double T_CONS = 3.5, T_PROD = 7.0, T_LAUNCH = 15.0, T_COMBINE_STEP = 1.0;

int64_t chunks_of(int64_t len) { return (len + BT - 1) / BT; }

// segments of a sequence of n chunks at segment length L (0: no split)
int segments_of(int64_t n, int L) {
    if (L <= 0 || n <= L) return 1;
    const int64_t p = (n + L - 1) / L;
    return static_cast<int>(p > MAX_SEGMENTS ? MAX_SEGMENTS : p);
}
// chunks of segment s of a sequence of n chunks split into P segments of L
int64_t seg_chunks(int64_t n, int L, int P, int s) {
    if (P == 1) return n;
    return s < P - 1 ? L : n - static_cast<int64_t>(L) * (P - 1);
}

// time of one launch of the chunked kernel over `chains` chains of at most
// `longest` chunks, `chunks` chunks in all, on `sms` SMs: the consumers' share
// (the kernel's longest-first schedule balances their chunk counts, bounded
// below by the longest chain) or the producers' share, whichever is larger
double launch_us(int64_t chains, int64_t longest, int64_t chunks, int sms) {
    if (chains < 1) return 0.0;
    const int64_t c = std::min<int64_t>(chains, sms / 2);
    const double per_consumer = std::max(static_cast<double>(longest), static_cast<double>(chunks) / static_cast<double>(c));
    const double cons = per_consumer * T_CONS;
    const double prod = static_cast<double>(chunks) * T_PROD / static_cast<double>(sms - c);
    return std::max(cons, prod) + T_LAUNCH;
}

struct Sizes {
    int64_t n1 = 0, t1 = 0, n3 = 0;  // pass-1 sequences and tokens, pass-3 sequences
    int nsplit = 0, pmax = 1;
};

Sizes sizes_for(const int32_t *cu, int N, int L) {
    Sizes z;
    for (int n = 0; n < N; ++n) {
        const int64_t len = static_cast<int64_t>(cu[n + 1]) - cu[n];
        const int64_t nc = chunks_of(len);
        const int P = segments_of(nc, L);
        z.n3 += P;
        if (P > 1) {
            ++z.nsplit;
            z.pmax = std::max(z.pmax, P);
            z.n1 += 2 * P - 3;  // segment 0 once, segments 1 .. P-2 twice
            z.t1 += static_cast<int64_t>(2 * P - 3) * L * BT;
        }
    }
    return z;
}

// Segment length (chunks) that the estimate prefers, or 0 when no split beats
// the plain launch by 20 %.
int plan(const int32_t *cu, int N, int H, int sms) {
    if (N < 1 || H < 1 || sms < 4) return 0;
    int64_t maxc = 0, totc = 0;
    for (int n = 0; n < N; ++n) {
        const int64_t nc = chunks_of(static_cast<int64_t>(cu[n + 1]) - cu[n]);
        maxc = std::max(maxc, nc);
        totc += nc;
    }
    const double plain = launch_us(static_cast<int64_t>(N) * H, maxc, totc * H, sms);
    int best_L = 0;
    double best = 0.8 * plain;
    for (int P = 2; P <= MAX_SEGMENTS; P *= 2) {
        const int L = static_cast<int>((maxc + P - 1) / P);
        if (L < 4) break;
        const Sizes z = sizes_for(cu, N, L);
        if (z.nsplit == 0 || z.t1 > kMaxTokens) continue;
        const double pass1 = launch_us(z.n1 * H, L, (z.t1 / BT) * H, sms);
        const double pass3 = launch_us(z.n3 * H, L, totc * H, sms);
        const double t = pass1 + pass3 + T_COMBINE_STEP * (z.pmax - 1) + 3 * 5.0;  // + the three small launches
        if (t < best) {
            best = t;
            best_L = L;
        }
    }
    return best_L;
}

// Workspace layout of a split call: the ring of the chunked kernel, the int32
// tables, then the fp32 states E1, F1 (pass 1) and E3, F3 (pass 3).
struct Layout {
    size_t ring = 0, tables = 0, e1 = 0, f1 = 0, e3 = 0, f3 = 0, total = 0;
    // int32 table offsets (elements from `tables`)
    size_t cu1 = 0, bos1 = 0, meta1 = 0, cu3 = 0, segp = 0, base1 = 0, base3 = 0, count = 0;
};

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

Layout layout_for(const Sizes &z, int N, int H) {
    Layout l;
    l.ring = align256(pers::workspace_bytes(std::max(z.n1, z.n3) * H));
    l.cu1 = 0;
    l.bos1 = l.cu1 + z.n1 + 1;
    l.meta1 = l.bos1 + z.n1;
    l.cu3 = l.meta1 + z.n1;
    l.segp = l.cu3 + z.n3 + 1;
    l.base1 = l.segp + N;
    l.base3 = l.base1 + N;
    l.count = l.base3 + N;
    l.tables = l.ring;
    l.e1 = l.tables + align256(l.count * 4);
    l.f1 = l.e1 + static_cast<size_t>(z.n1) * H * STATE * 4;
    l.e3 = l.f1 + static_cast<size_t>(z.n1) * H * STATE * 4;
    l.f3 = l.e3 + static_cast<size_t>(z.n3) * H * STATE * 4;
    l.total = l.f3 + static_cast<size_t>(z.n3) * H * STATE * 4;
    return l;
}

// ---------------------------------------------------------------- kernels
// meta1 = (sequence << 2) | kind: 0 = the sequence's entry state, 1 = identity, 2 = zero
__global__ void __launch_bounds__(256) fill_entry1(const int32_t *meta1, const float *s0, float *e1, int H) {
    const int i = blockIdx.x, h = blockIdx.y;
    const int m = meta1[i], n = m >> 2, kind = m & 3;
    float *dst = e1 + (static_cast<size_t>(i) * H + h) * STATE;
    const float *src = (kind == 0 && s0) ? s0 + (static_cast<size_t>(n) * H + h) * STATE : nullptr;
    for (int e = threadIdx.x; e < static_cast<int>(STATE / 4); e += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (src) {
            v = reinterpret_cast<const float4 *>(src)[e];
        } else if (kind == 1) {
            const int row = (4 * e) / DV, col = (4 * e) % DV;  // one row, four consecutive columns
            v.x = row == col ? 1.f : 0.f;
            v.y = row == col + 1 ? 1.f : 0.f;
            v.z = row == col + 2 ? 1.f : 0.f;
            v.w = row == col + 3 ? 1.f : 0.f;
        }
        reinterpret_cast<float4 *>(dst)[e] = v;
    }
}

// Entry states of every pass-3 segment, for sequence blockIdx.x, head
// blockIdx.y and value columns 16 * blockIdx.z .. +15; thread i owns key row i.
// For a split sequence (P > 1): S_0 = its entry state, S_1 = F1[base1] (the
// exit of segment 0), S_{s+1} = (F1[I_s] - F1[Z_s]) S_s + F1[Z_s] with
// I_s = base1 + 2s - 1 and Z_s = base1 + 2s.
__global__ void __launch_bounds__(DK) combine(const int32_t *segp, const int32_t *base1, const int32_t *base3,
                                              const float *s0, const float *f1, float *e3, int H) {
    __shared__ float S[DK][17];
    const int n = blockIdx.x, h = blockIdx.y, c0 = 16 * blockIdx.z, i = threadIdx.x;
    const int P = segp[n], b1 = base1[n], b3 = base3[n];
    auto st = [&](auto *base, int64_t idx) { return base + (static_cast<size_t>(idx) * H + h) * STATE; };
    float row[16];
    const float *src0 = s0 ? st(s0, n) : nullptr;
#pragma unroll
    for (int c = 0; c < 16; ++c) row[c] = src0 ? src0[i * DV + c0 + c] : 0.f;
    for (int s = 0; s < P; ++s) {
        if (s == 1) {  // the exit of segment 0, run from the sequence's own entry state
            const float *x = st(f1, b1);
#pragma unroll
            for (int c = 0; c < 16; ++c) row[c] = x[i * DV + c0 + c];
        } else if (s > 1) {  // S_s = (F_I - F_Z) S_{s-1} + F_Z for segment s - 1
            const float *fi = st(f1, b1 + 2 * (s - 1) - 1), *fz = st(f1, b1 + 2 * (s - 1));
            __syncthreads();
#pragma unroll
            for (int c = 0; c < 16; ++c) S[i][c] = row[c];
            __syncthreads();
            float acc[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = fz[i * DV + c0 + c];
            for (int kk = 0; kk < DK; kk += 4) {
                const float4 a = *reinterpret_cast<const float4 *>(fi + i * DV + kk);
                const float4 z = *reinterpret_cast<const float4 *>(fz + i * DV + kk);
                const float phi[4] = {a.x - z.x, a.y - z.y, a.z - z.z, a.w - z.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int c = 0; c < 16; ++c) acc[c] = fmaf(phi[q], S[kk + q][c], acc[c]);
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) row[c] = acc[c];
        }
        float *d = st(e3, b3 + s);
#pragma unroll
        for (int c = 0; c < 16; c += 4)
            *reinterpret_cast<float4 *>(d + i * DV + c0 + c) = make_float4(row[c], row[c + 1], row[c + 2], row[c + 3]);
    }
}

// final_state[n] = the exit state of sequence n's last segment
__global__ void __launch_bounds__(256) gather_final(const int32_t *segp, const int32_t *base3, const float *f3,
                                                    float *final_state, int H) {
    const int n = blockIdx.x, h = blockIdx.y;
    const float4 *src = reinterpret_cast<const float4 *>(f3 + (static_cast<size_t>(base3[n] + segp[n] - 1) * H + h) * STATE);
    float4 *dst = reinterpret_cast<float4 *>(final_state + (static_cast<size_t>(n) * H + h) * STATE);
    for (int e = threadIdx.x; e < static_cast<int>(STATE / 4); e += blockDim.x) dst[e] = src[e];
}

using checks::aligned;
using checks::host_seqlens_ok;

int current_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace split
}  // namespace kda

using namespace kda::split;

extern "C" {

int32_t kda_chunk_fwd_split_plan(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                 int32_t num_sms) {
    if (!cu_seqlens_host || num_seqs < 1 || num_heads < 1) return 0;
    if (!host_seqlens_ok(cu_seqlens_host, num_seqs, cu_seqlens_host[num_seqs])) return 0;
    const int sms = num_sms > 0 ? num_sms : current_sms();
    return plan(cu_seqlens_host, num_seqs, num_heads, sms);
}

size_t kda_chunk_fwd_split_workspace_size(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                          int32_t segment_chunks) {
    if (!cu_seqlens_host || num_seqs < 1 || num_heads < 1 || segment_chunks < 0) return 0;
    if (!host_seqlens_ok(cu_seqlens_host, num_seqs, cu_seqlens_host[num_seqs])) return 0;
    const int L = segment_chunks > 0 ? segment_chunks : plan(cu_seqlens_host, num_seqs, num_heads, current_sms());
    const Sizes z = sizes_for(cu_seqlens_host, num_seqs, L);
    if (z.nsplit == 0) return kda_chunk_fwd_workspace_size(num_seqs, num_heads);
    const Layout l = layout_for(z, num_seqs, num_heads);
    return l.ring == 0 ? 0 : l.total;
}

kda_status_t kda_chunk_fwd_split(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t num_seqs,
                                 int64_t total_tokens, int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                 const float *initial_state, float scale, float lower_bound, int32_t segment_chunks,
                                 float *o, float *final_state, int32_t *status_dev, void *workspace,
                                 size_t workspace_bytes, kda_stream_t stream) {
    if (head_dim_k != KDA_HEAD_DIM || head_dim_v != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 1 || num_heads < 1 || total_tokens < 0 || segment_chunks < 0) return KDA_ERR_INVALID_ARG;
    if (num_heads > 65535) return KDA_ERR_UNSUPPORTED;  // a grid dimension of the small kernels
    if (!host_seqlens_ok(cu_seqlens_host, num_seqs, total_tokens)) return KDA_ERR_INVALID_ARG;
    const int L = segment_chunks > 0 ? segment_chunks : plan(cu_seqlens_host, num_seqs, num_heads, current_sms());
    const Sizes z = sizes_for(cu_seqlens_host, num_seqs, L);
    if (z.nsplit == 0)  // nothing to split: the plain call, on the device copy of cu_seqlens
        return kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, num_seqs, total_tokens, num_heads, head_dim_k,
                             head_dim_v, initial_state, scale, lower_bound, o, final_state, status_dev, workspace,
                             workspace_bytes, stream);
    // the checks kda_chunk_fwd makes, for the pointers the passes use
    if (total_tokens > kMaxTokens || z.t1 > kMaxTokens) return KDA_ERR_UNSUPPORTED;
    if (!kda::checks::scale_ok(scale) || !kda::checks::lower_bound_ok(lower_bound)) return KDA_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !beta || !o || !workspace) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(o, 16) ||
        !aligned(beta, 4) || !aligned(workspace, 256) || (initial_state && !aligned(initial_state, 16)) ||
        (final_state && !aligned(final_state, 16)) || (status_dev && !aligned(status_dev, 4)))
        return KDA_ERR_INVALID_ARG;
    const int N = num_seqs, H = num_heads;
    const Layout l = layout_for(z, N, H);
    if (l.ring == 0) return KDA_ERR_CUDA;
    if (workspace_bytes < l.total) return KDA_ERR_INVALID_ARG;

    // the tables, on the host
    std::vector<int32_t> t(l.count);
    int32_t *cu1 = t.data() + l.cu1, *bos1 = t.data() + l.bos1, *meta1 = t.data() + l.meta1;
    int32_t *cu3 = t.data() + l.cu3, *segp = t.data() + l.segp, *base1 = t.data() + l.base1,
            *base3 = t.data() + l.base3;
    int64_t i1 = 0, i3 = 0;
    cu1[0] = 0;
    cu3[0] = 0;
    for (int n = 0; n < N; ++n) {
        const int64_t bos = cu_seqlens_host[n], len = static_cast<int64_t>(cu_seqlens_host[n + 1]) - bos;
        const int64_t nc = chunks_of(len);
        const int P = segments_of(nc, L);
        segp[n] = P;
        base3[n] = static_cast<int32_t>(i3);
        base1[n] = P > 1 ? static_cast<int32_t>(i1) : -1;
        int64_t tok = bos;
        for (int s = 0; s < P; ++s) {
            const int64_t sl = std::min<int64_t>(seg_chunks(nc, L, P, s) * BT, bos + len - tok);
            if (P > 1 && s < P - 1) {  // pass 1: segment 0 from the entry state; 1 .. P-2 from I and from 0
                const int kinds = s == 0 ? 1 : 2;
                for (int r = 0; r < kinds; ++r) {
                    bos1[i1] = static_cast<int32_t>(tok);
                    meta1[i1] = (n << 2) | (s == 0 ? 0 : 1 + r);
                    cu1[i1 + 1] = static_cast<int32_t>(cu1[i1] + sl);
                    ++i1;
                }
            }
            cu3[i3 + 1] = static_cast<int32_t>(tok + sl);
            ++i3;
            tok += sl;
        }
    }
    if (i1 != z.n1 || i3 != z.n3) return KDA_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    int32_t *dt = reinterpret_cast<int32_t *>(ws + l.tables);
    float *e1 = reinterpret_cast<float *>(ws + l.e1), *f1 = reinterpret_cast<float *>(ws + l.f1);
    float *e3 = reinterpret_cast<float *>(ws + l.e3), *f3 = reinterpret_cast<float *>(ws + l.f3);
    if (status_dev && cudaMemsetAsync(status_dev, 0, sizeof(int32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    // pageable source: the copy is staged before the call returns, so `t` may go
    if (cudaMemcpyAsync(dt, t.data(), l.count * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KDA_ERR_CUDA;

    fill_entry1<<<dim3(static_cast<unsigned>(z.n1), H), 256, 0, s>>>(dt + l.meta1, initial_state, e1, H);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;

    kda::pers::Params p{};
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(k);
    p.v = static_cast<const __nv_bfloat16 *>(v);
    p.g = g;
    p.beta = beta;
    p.H = H;
    p.scale = scale;
    p.lb = lower_bound;
    p.status = status_dev;
    p.ws = ws;
    p.Ttok = total_tokens;
    // pass 1: states only, segments listed through the token map
    p.cu = dt + l.cu1;
    p.seq_bos = dt + l.bos1;
    p.N = static_cast<int32_t>(z.n1);
    p.T = z.t1 > 0 ? cu1[z.n1] : 0;
    p.s0 = e1;
    p.sT = f1;
    p.o = nullptr;
    if (kda::pers::launch(p, l.ring, s) != cudaSuccess) return KDA_ERR_CUDA;

    combine<<<dim3(N, H, DV / 16), DK, 0, s>>>(dt + l.segp, dt + l.base1, dt + l.base3, initial_state, f1, e3, H);
    if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;

    // pass 3: every segment in order, from its entry state
    p.cu = dt + l.cu3;
    p.seq_bos = nullptr;
    p.N = static_cast<int32_t>(z.n3);
    p.T = total_tokens;
    p.s0 = e3;
    p.sT = final_state ? f3 : nullptr;
    p.o = o;
    if (kda::pers::launch(p, l.ring, s) != cudaSuccess) return KDA_ERR_CUDA;

    if (final_state) {
        gather_final<<<dim3(N, H), 256, 0, s>>>(dt + l.segp, dt + l.base3, f3, final_state, H);
        if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"
