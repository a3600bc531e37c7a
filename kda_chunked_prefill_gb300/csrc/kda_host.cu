// kda_chunk_fwd_host: the chunked-prefill forward on inputs and outputs in host
// memory.
//
// When every buffer is page-locked host memory that the device addresses in
// place (cudaHostAlloc memory, or cudaHostRegister'ed memory mapped, under
// unified addressing) and the caller lets the library choose the grouping,
// one launch of the chunked kernel reads the inputs and writes o and the
// final states in host memory directly over the CPU-GPU link: no staging
// copies at all. Otherwise the transfers are overlapped with the computation:
//
// The batch is cut into groups of whole sequences of about equal token counts.
// Group i's inputs go to the device on the H2D stream; the compute stream waits
// for them and runs the chunked kernel on that group alone (its own offsets,
// rebased to 0); the D2H stream waits for that launch and brings the group's o
// and final states back. So the copies of group i + 1 in and of group i - 1 out
// run while group i computes. The compute stream finally waits for the last
// copy out, so synchronising it means the host outputs are complete.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "kda.h"

#include "kda_checks.h"
#include "kda_persistent.h"

namespace kda {
namespace host {

constexpr int DK = 128, DV = 128, MAX_GROUPS = 16;
constexpr size_t STATE = static_cast<size_t>(DK) * DV;
using checks::kMaxTokens;
using checks::host_seqlens_ok;

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Groups of whole sequences, each closed once it holds about T / G tokens:
// first[i] .. first[i + 1] - 1 are group i's sequences.
std::vector<int> group_bounds(const int32_t *cu, int N, int G) {
    std::vector<int> first{0};
    const int64_t T = cu[N];
    for (int n = 0; n < N && static_cast<int>(first.size()) < G; ++n) {
        const int64_t target = T * static_cast<int64_t>(first.size()) / G;
        if (cu[n + 1] >= target && n + 1 < N && cu[n + 1] > cu[first.back()]) first.push_back(n + 1);
    }
    first.push_back(N);
    return first;
}

struct Layout {
    size_t q = 0, k = 0, v = 0, g = 0, beta = 0, s0 = 0, o = 0, fs = 0, cu = 0, ring = 0, total = 0;
};

Layout layout_for(const int32_t *cu, int N, int H, bool with_init, bool with_final, const std::vector<int> &first) {
    const size_t T = static_cast<size_t>(cu[N]);
    int64_t max_chains = 1;
    for (size_t i = 0; i + 1 < first.size(); ++i)
        max_chains = std::max<int64_t>(max_chains, static_cast<int64_t>(first[i + 1] - first[i]) * H);
    Layout l;
    size_t at = 0;
    auto take = [&](size_t bytes) { const size_t o = at; at = align256(at + bytes); return o; };
    l.q = take(T * H * DK * 2);
    l.k = take(T * H * DK * 2);
    l.v = take(T * H * DV * 2);
    l.g = take(T * H * DK * 4);
    l.beta = take(T * H * 4);
    l.s0 = take(with_init ? static_cast<size_t>(N) * H * STATE * 4 : 0);
    l.o = take(T * H * DV * 4);
    l.fs = take(with_final ? static_cast<size_t>(N) * H * STATE * 4 : 0);
    l.cu = take(static_cast<size_t>(N + static_cast<int>(first.size())) * 4);
    // the in-place form runs all N x H chains in one launch
    const size_t ring = pers::workspace_bytes(std::max<int64_t>(max_chains, static_cast<int64_t>(N) * H));
    l.ring = take(ring);
    l.total = ring == 0 ? 0 : at;
    return l;
}

// true for NULL and for page-locked host memory the device addresses at the same pointer
bool addressable_in_place(const void *p) {
    if (!p) return true;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

int groups_for(int N, int32_t groups) {
    const int G = groups > 0 ? groups : 4;
    return std::max(1, std::min({G, N, MAX_GROUPS}));
}

}  // namespace host
}  // namespace kda

using namespace kda::host;

extern "C" {

size_t kda_chunk_fwd_host_buffer_size(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                      int32_t with_initial_state, int32_t with_final_state, int32_t groups) {
    if (!cu_seqlens_host || num_seqs < 1 || num_heads < 1 || groups < 0) return 0;
    if (!host_seqlens_ok(cu_seqlens_host, num_seqs, cu_seqlens_host[num_seqs])) return 0;
    const std::vector<int> first = group_bounds(cu_seqlens_host, num_seqs, groups_for(num_seqs, groups));
    return layout_for(cu_seqlens_host, num_seqs, num_heads, with_initial_state != 0, with_final_state != 0, first)
        .total;
}

kda_status_t kda_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu_seqlens_host, int32_t num_seqs, int64_t total_tokens,
                                int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                const float *initial_state, float scale, float lower_bound, float *o,
                                float *final_state, int32_t *status_dev, void *device_buffer,
                                size_t device_buffer_bytes, int32_t groups, kda_stream_t stream,
                                kda_stream_t h2d_stream, kda_stream_t d2h_stream) {
    if (head_dim_k != KDA_HEAD_DIM || head_dim_v != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
    if (num_seqs < 1 || num_heads < 1 || total_tokens < 0 || groups < 0) return KDA_ERR_INVALID_ARG;
    if (total_tokens > kMaxTokens) return KDA_ERR_UNSUPPORTED;
    if (!host_seqlens_ok(cu_seqlens_host, num_seqs, total_tokens)) return KDA_ERR_INVALID_ARG;
    if (!kda::checks::scale_ok(scale) || !kda::checks::lower_bound_ok(lower_bound)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!device_buffer || !kda::checks::aligned(device_buffer, 256)) return KDA_ERR_INVALID_ARG;
    if (status_dev && !kda::checks::aligned(status_dev, 4)) return KDA_ERR_INVALID_ARG;
    const int N = num_seqs, H = num_heads;
    const std::vector<int> first = group_bounds(cu_seqlens_host, N, groups_for(N, groups));
    const int G = static_cast<int>(first.size()) - 1;
    const Layout l = layout_for(cu_seqlens_host, N, H, initial_state != nullptr, final_state != nullptr, first);
    if (l.total == 0) return KDA_ERR_CUDA;
    if (device_buffer_bytes < l.total) return KDA_ERR_INVALID_ARG;

    // per-group offsets rebased to the group's first token, one table for all groups
    std::vector<int32_t> cut;
    std::vector<size_t> cu_at(G);
    for (int i = 0; i < G; ++i) {
        cu_at[i] = cut.size();
        for (int n = first[i]; n <= first[i + 1]; ++n) cut.push_back(cu_seqlens_host[n] - cu_seqlens_host[first[i]]);
    }

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *buf = static_cast<unsigned char *>(device_buffer);
    if (groups == 0 && total_tokens > 0 && addressable_in_place(q) && addressable_in_place(k) &&
        addressable_in_place(v) && addressable_in_place(g) && addressable_in_place(beta) &&
        addressable_in_place(initial_state) && addressable_in_place(o) && addressable_in_place(final_state)) {
        // in place: one launch on the host buffers (only the offsets and the ring are in device memory)
        bool ok = !status_dev || cudaMemsetAsync(status_dev, 0, sizeof(int32_t), cs) == cudaSuccess;
        // pageable source: staged before the call returns
        ok = ok && cudaMemcpyAsync(buf + l.cu, cu_seqlens_host, static_cast<size_t>(N + 1) * 4, cudaMemcpyHostToDevice,
                                   cs) == cudaSuccess;
        if (!ok) return KDA_ERR_CUDA;
        kda::pers::Params p{};
        p.q = static_cast<const __nv_bfloat16 *>(q);
        p.k = static_cast<const __nv_bfloat16 *>(k);
        p.v = static_cast<const __nv_bfloat16 *>(v);
        p.g = g;
        p.beta = beta;
        p.cu = reinterpret_cast<const int32_t *>(buf + l.cu);
        p.N = N;
        p.T = total_tokens;
        p.Ttok = total_tokens;
        p.H = H;
        p.s0 = initial_state;
        p.scale = scale;
        p.lb = lower_bound;
        p.o = o;
        p.sT = final_state;
        p.status = status_dev;
        p.ws = buf + l.ring;
        return kda::pers::launch(p, l.total - l.ring, cs) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    cudaStream_t in = h2d_stream ? reinterpret_cast<cudaStream_t>(h2d_stream) : cs;
    cudaStream_t out = d2h_stream ? reinterpret_cast<cudaStream_t>(d2h_stream) : cs;
    std::vector<cudaEvent_t> ev(2 * G + 2, nullptr);
    auto release = [&]() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);  // released once its work completes
    };
    for (cudaEvent_t &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            release();
            return KDA_ERR_CUDA;
        }
    cudaEvent_t start = ev[2 * G], done = ev[2 * G + 1];
    bool ok = cudaEventRecord(start, cs) == cudaSuccess && cudaStreamWaitEvent(in, start, 0) == cudaSuccess &&
              cudaStreamWaitEvent(out, start, 0) == cudaSuccess;
    if (ok && status_dev) ok = cudaMemsetAsync(status_dev, 0, sizeof(int32_t), cs) == cudaSuccess;
    // pageable source: staged before the call returns
    ok = ok && cudaMemcpyAsync(buf + l.cu, cut.data(), cut.size() * 4, cudaMemcpyHostToDevice, in) == cudaSuccess;

    const size_t th = static_cast<size_t>(H);
    for (int i = 0; ok && i < G; ++i) {
        const int n0 = first[i], n1 = first[i + 1];
        const size_t t0 = static_cast<size_t>(cu_seqlens_host[n0]);
        const size_t nt = static_cast<size_t>(cu_seqlens_host[n1]) - t0;
        const size_t ns = static_cast<size_t>(n1 - n0);
        auto h2d = [&](size_t off, const void *src, size_t elem_off, size_t bytes) {
            if (bytes == 0) return true;
            return cudaMemcpyAsync(buf + off + elem_off, static_cast<const unsigned char *>(src) + elem_off, bytes,
                                   cudaMemcpyHostToDevice, in) == cudaSuccess;
        };
        ok = h2d(l.q, q, t0 * th * DK * 2, nt * th * DK * 2) && h2d(l.k, k, t0 * th * DK * 2, nt * th * DK * 2) &&
             h2d(l.v, v, t0 * th * DV * 2, nt * th * DV * 2) && h2d(l.g, g, t0 * th * DK * 4, nt * th * DK * 4) &&
             h2d(l.beta, beta, t0 * th * 4, nt * th * 4) &&
             (!initial_state || h2d(l.s0, initial_state, n0 * th * STATE * 4, ns * th * STATE * 4));
        ok = ok && cudaEventRecord(ev[2 * i], in) == cudaSuccess && cudaStreamWaitEvent(cs, ev[2 * i], 0) == cudaSuccess;
        if (!ok) break;
        if (nt > 0) {
            kda::pers::Params p{};
            p.q = reinterpret_cast<const __nv_bfloat16 *>(buf + l.q) + t0 * th * DK;
            p.k = reinterpret_cast<const __nv_bfloat16 *>(buf + l.k) + t0 * th * DK;
            p.v = reinterpret_cast<const __nv_bfloat16 *>(buf + l.v) + t0 * th * DV;
            p.g = reinterpret_cast<const float *>(buf + l.g) + t0 * th * DK;
            p.beta = reinterpret_cast<const float *>(buf + l.beta) + t0 * th;
            p.cu = reinterpret_cast<const int32_t *>(buf + l.cu) + cu_at[i];
            p.N = static_cast<int32_t>(ns);
            p.T = static_cast<int64_t>(nt);
            p.Ttok = static_cast<int64_t>(nt);
            p.H = H;
            p.s0 = initial_state ? reinterpret_cast<const float *>(buf + l.s0) + n0 * th * STATE : nullptr;
            p.scale = scale;
            p.lb = lower_bound;
            p.o = reinterpret_cast<float *>(buf + l.o) + t0 * th * DV;
            p.sT = final_state ? reinterpret_cast<float *>(buf + l.fs) + n0 * th * STATE : nullptr;
            p.status = status_dev;
            p.ws = buf + l.ring;
            ok = kda::pers::launch(p, l.total - l.ring, cs) == cudaSuccess;
        } else if (final_state) {  // only empty sequences: the state passes through
            ok = initial_state ? cudaMemcpyAsync(buf + l.fs + n0 * th * STATE * 4, buf + l.s0 + n0 * th * STATE * 4,
                                                 ns * th * STATE * 4, cudaMemcpyDeviceToDevice, cs) == cudaSuccess
                               : cudaMemsetAsync(buf + l.fs + n0 * th * STATE * 4, 0, ns * th * STATE * 4, cs) ==
                                     cudaSuccess;
        }
        ok = ok && cudaEventRecord(ev[2 * i + 1], cs) == cudaSuccess &&
             cudaStreamWaitEvent(out, ev[2 * i + 1], 0) == cudaSuccess;
        if (ok && nt > 0)
            ok = cudaMemcpyAsync(reinterpret_cast<unsigned char *>(o) + t0 * th * DV * 4, buf + l.o + t0 * th * DV * 4,
                                 nt * th * DV * 4, cudaMemcpyDeviceToHost, out) == cudaSuccess;
        if (ok && final_state)
            ok = cudaMemcpyAsync(reinterpret_cast<unsigned char *>(final_state) + n0 * th * STATE * 4,
                                 buf + l.fs + n0 * th * STATE * 4, ns * th * STATE * 4, cudaMemcpyDeviceToHost,
                                 out) == cudaSuccess;
    }
    ok = ok && cudaEventRecord(done, out) == cudaSuccess && cudaStreamWaitEvent(cs, done, 0) == cudaSuccess;
    release();
    return ok ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
