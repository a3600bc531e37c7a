// KDA chunked prefill forward — persistent cooperative kernel, one CTA per SM,
// in two roles that hand chunks to each other through a small ring in L2.
//
//   producers  pull (chain, chunk) tasks from a global counter and run the
//              intra-chunk steps of "在 TPU 上加速 Kimi K3 KDA" (junyi.dev
//              tpu-kda report): step 1 gate prefix sum (§6.1), step 2 Aqk/Akk
//              as products of sub-block-midpoint-rescaled operands (§4), step 3
//              (I+L)^-1 by 16x16 block forward substitution, step 4 the WY form
//              u, w plus q_hat = scale q e^G and kg = k e^(G_last - G) (§4, §6.3).
//              They write [q_hat; w], kg, u, scale*Aqk and d = e^(G_last) into a
//              ring slot already in the swizzled layouts the consumer's tensor-
//              core operands use, then release the slot's ready flag.
//   consumers  own (sequence, head) chains and run step 5 chunk after chunk
//              (§6.2): v_new = u - w S, o = q_hat S + Aqk v_new,
//              S <- Diag(d) S + kg^T v_new, reading the entry state, with the
//              state on chip for the whole chain; each slot is streamed into
//              shared memory by a bulk copy issued one chunk ahead.
//
// The chunk-to-chunk dependency of a chain is the only serial part; the
// intra-chunk work (most of the arithmetic) is spread over every other SM.
// All waits are bounded: a wait that runs out sets KDA_ERR_TIMEOUT and an abort
// word in the workspace, and every CTA then returns.
#include "kda.h"
#include "kda_common.cuh"
#include "kda_persistent.h"

namespace kda {
namespace pers {

constexpr int NCOMP = 512;            // 16 warps, all computing (<= 128 registers each)
constexpr int NTHREADS = NCOMP;
constexpr int NWARPS = NCOMP / 32;
constexpr long long SPIN_LIMIT = 1ll << 24;

// ---------------------------------------------------------------- slot layout
// A slot holds one (chain, chunk) hand-off; every region is 1024-byte aligned.
//   A1  [q_hat ; w]  fp16, 128 rows x 128 key channels, K-major, 128B swizzle
//   KG  kg           fp16, [token][key] (64 x 128): the transposed operand kg^T
//   U   u            fp16, [token][value] (64 x 128)
//   D   e^(G_last)   fp32, 128
//   AQK scale * Aqk  fp16, [t][s] (64 x 64), causal incl. diagonal
// 128-byte swizzle: row r of a 128-byte-wide atom column keeps its 16-byte
// chunk c at position c ^ (r mod 8); wider tiles are split into 64-element
// atom columns stored one after the other.
constexpr int SL_A1 = 0, SL_KG = 32768, SL_U = 49152, SL_D = 65536, SL_AQK = 66560;
static_assert(SLOT_BYTES == 74752, "slot size");

__device__ __forceinline__ int swz(int r, int chunk) { return (chunk ^ (r & 7)) << 4; }
// byte offset of the 16-byte chunk holding columns [c8, c8+8) of row r of a
// swizzled tile with `rows` rows per atom column
__device__ __forceinline__ int tile_chunk(int rows, int r, int c8) {
    return (c8 >> 6) * rows * 128 + r * 128 + swz(r, (c8 & 63) >> 3);
}
__device__ __forceinline__ int tile_elem(int rows, int r, int c) { return tile_chunk(rows, r, c & ~7) + ((c & 7) << 1); }
// ldmatrix lane addresses (byte offsets) on swizzled tiles
__device__ __forceinline__ int a_addr(int lane, int rows, int row0, int col0) {  // A stored [m][k]
    return tile_chunk(rows, row0 + (lane & 15), col0 + ((lane >> 4) << 3));
}
__device__ __forceinline__ int bk_addr(int lane, int rows, int k0, int n0) {  // B stored [k][n]
    const int mi = lane >> 3, rr = lane & 7;
    return tile_chunk(rows, k0 + ((mi & 1) << 3) + rr, n0 + ((mi >> 1) << 3));
}
__device__ __forceinline__ int at_addr(int lane, int rows, int m0, int k0) {  // A stored [k][m]
    const int mi = lane >> 3, rr = lane & 7;
    return tile_chunk(rows, k0 + ((mi >> 1) << 3) + rr, m0 + ((mi & 1) << 3));
}

__device__ __forceinline__ void sync_compute() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Optional event trace (compiled in only with -DKDA_TRACE): per CTA, up to
// TRACE_EVENTS records {globaltimer ns, tag, value} after the ring in the workspace.
#ifdef KDA_TRACE
constexpr int TRACE_EVENTS = 512;
__device__ __forceinline__ void trace(const Params &p, int tag, int value) {
    if (threadIdx.x != 0) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    unsigned char *base = p.ws + ring_offset(p.C) + static_cast<size_t>(p.C) * RING * SLOT_BYTES;
    unsigned long long *rec = reinterpret_cast<unsigned long long *>(base) + blockIdx.x * (TRACE_EVENTS * 2 + 1);
    const unsigned long long n = rec[0];
    if (n < TRACE_EVENTS) {
        rec[1 + 2 * n] = t;
        rec[2 + 2 * n] = (static_cast<unsigned long long>(tag) << 32) | static_cast<unsigned>(value);
        rec[0] = n + 1;
    }
}
#define KDA_TRACE_EV(p, tag, value) trace(p, tag, value)
#else
#define KDA_TRACE_EV(p, tag, value) ((void)0)
#endif

// ---------------------------------------------------------------- workspace
struct Header {
    int counter;  // next producer task
    int abort;    // set on a timed-out wait
    int pad[14];
};

struct Ring {
    Header *hdr;
    int *ready;  // [C][RING]: chunk index + 1 held by the slot
    int *freed;  // [C][RING]: chunk index + 1 the consumer has copied out
    unsigned char *slots;
};

__device__ __forceinline__ Ring ring_of(const Params &p) {
    Ring r;
    r.hdr = reinterpret_cast<Header *>(p.ws);
    r.ready = reinterpret_cast<int *>(p.ws + sizeof(Header));
    r.freed = r.ready + p.C * RING;
    r.slots = p.ws + ring_offset(p.C);
    return r;
}

__device__ __forceinline__ bool wait_flag_geq(const Ring &R, const int *flag, int target, int32_t *status) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (ld_acquire(flag) >= target) return true;
        if ((it & 127) == 127 && ld_relaxed(&R.hdr->abort)) return false;
        __nanosleep(64);
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

__device__ __forceinline__ bool wait_mbar(const Ring &R, uint64_t *bar, uint32_t parity, int32_t *status) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 127) == 127 && ld_relaxed(&R.hdr->abort)) return false;
        __nanosleep(32);
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

// chunks of chain ch (sequence ch / H), or -1 when its bounds are invalid
__device__ __forceinline__ int chain_info(const Params &p, int ch, int64_t &bos, int64_t &len) {
    const int n = ch / p.H;
    const int64_t b = p.cu[n], e = p.cu[n + 1];
    const bool bad = b < 0 || e < b || e > p.T || (n == 0 && b != 0) || (n == p.N - 1 && e != p.T);
    if (bad) {
        bos = 0;
        len = 0;
        return -1;
    }
    bos = b;
    len = e - b;
    return static_cast<int>((len + BT - 1) / BT);
}

// consumer k owns chains k, k + C, k + 2C, ...; its chunks form one sequence
__device__ __forceinline__ int consumer_total(const Params &p, int k) {
    int tot = 0;
    for (int ch = k; ch < p.N * p.H; ch += p.C) {
        int64_t b, l;
        const int nc = chain_info(p, ch, b, l);
        tot += nc > 0 ? nc : 0;
    }
    return tot;
}

__device__ __forceinline__ bool map_task(const Params &p, int k, int j, int &ch_out, int &c_out) {
    for (int ch = k; ch < p.N * p.H; ch += p.C) {
        int64_t b, l;
        int nc = chain_info(p, ch, b, l);
        if (nc < 0) nc = 0;
        if (j < nc) {
            ch_out = ch;
            c_out = j;
            return true;
        }
        j -= nc;
    }
    return false;
}

// ================================================================== producer
// Steps 1-4 for one (chain, chunk) task at a time, on 256 threads with
// warp-level tensor-core products (m16n8k16) for the 16x16 tiles.
namespace prod {
constexpr int RSB = 136, RSF = 136, RSA = 72, RSI = 24;
constexpr int SZ_T = BT * RSB * 2;        // 17408
constexpr int SZ_F = BT * RSF * 4;        // 34816
constexpr int OFF_Q = 0;                  // q -> q*a (bf16 hi)
constexpr int OFF_QLO = OFF_Q + SZ_T;     // q*a (bf16 lo); v / u of the next task (roles swap per task)
constexpr int OFF_K = OFF_QLO + SZ_T;     // k -> k*a (bf16)
constexpr int OFF_V = OFF_K + SZ_T;       // v -> beta*v -> u (fp16); q*a lo of the next task
constexpr int OFF_RK = OFF_V + SZ_T;      // beta*k*e^G -> w (fp16)
constexpr int OFF_G = OFF_RK + SZ_T;      // g -> G (fp32)
constexpr int OFF_KB = OFF_G + SZ_F;      // k*e^(G_m - G) (fp32)
constexpr int OFF_AQK = OFF_KB + SZ_F;    // scale*Aqk (fp16 [64][RSA])
constexpr int SZ_A = BT * RSA * 2;        // 9216
constexpr int OFF_L = OFF_AQK + SZ_A;     // L (fp16 [64][RSA])
constexpr int OFF_LD = OFF_L + SZ_A;      // diagonal blocks of L, fp32 [4][16][17]
constexpr int OFF_INV = OFF_LD + 4352;    // (I+L_ii)^-1 fp16 [4][16][RSI]
constexpr int OFF_TAB = OFF_INV + 3072;   // per-channel tables, fp32 [20][128]
constexpr int OFF_BETA = OFF_TAB + 10240;
constexpr int OFF_MISC = OFF_BETA + 256;  // flags and the task broadcast
constexpr int SMEM = OFF_MISC + 64;
constexpr int TGM = 0, TGL = 4 * 128, TEM = 5 * 128, TEL = 9 * 128, TF = 13 * 128, TD = 19 * 128;
__device__ __forceinline__ int f_pair(int i, int j) { return i * (i - 1) / 2 + j; }
__device__ __forceinline__ bool f16_ok(float x) { return fabsf(x) < F16_SAFE; }

// One (chain, chunk) task: steps 1-4, results into the global slot.
struct Task {
    int valid, k, j, ch, c;
};

// next valid task (thread 0): tasks are numbered j * C + k so every consumer advances together
__device__ __forceinline__ Task fetch_task(const Params &p, const Ring &R, int jmax) {
    Task t{0, 0, 0, 0, 0};
    while (true) {
        const int task = atomicAdd(&R.hdr->counter, 1);
        t.k = task % p.C;
        t.j = task / p.C;
        if (t.j >= jmax) return t;
        if (map_task(p, t.k, t.j, t.ch, t.c)) {
            t.valid = 1;
            return t;
        }
    }
}

// cp.async of part of one task's inputs (rows >= nv zero-filled):
// part 0: g; part 1: q, k, v (v into vbuf) and beta.
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *smem, const Task &tk, int part, int vbuf) {
    const int tid = threadIdx.x;
    const int h = tk.ch % p.H;
    int64_t bos, len;
    chain_info(p, tk.ch, bos, len);
    const int64_t t0 = bos + static_cast<int64_t>(tk.c) * BT;
    const int nv = static_cast<int>((bos + len - t0) < BT ? (bos + len - t0) : BT);
    const size_t rs = static_cast<size_t>(p.H) * DK;
    const size_t base = (static_cast<size_t>(t0) * p.H + h) * DK;
    if (part == 0) {
        float *sG = reinterpret_cast<float *>(smem + OFF_G);
        for (int idx = tid; idx < BT * 32; idx += NCOMP) {
            const int r = idx >> 5, c4 = (idx & 31) << 2;
            const bool ok = r < nv;
            cp_async16(sG + r * RSF + c4, p.g + base + (ok ? r * rs : 0) + c4, ok ? 16 : 0);
        }
    } else {
        __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_Q);
        __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_K);
        __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(smem + vbuf);
        for (int idx = tid; idx < BT * 16; idx += NCOMP) {
            const int r = idx >> 4, c8 = (idx & 15) << 3;
            const bool ok = r < nv;
            const size_t off = base + (ok ? r * rs : 0) + c8;
            cp_async16(sQ + r * RSB + c8, p.q + off, ok ? 16 : 0);
            cp_async16(sK + r * RSB + c8, p.k + off, ok ? 16 : 0);
            cp_async16(sV + r * RSB + c8, p.v + off, ok ? 16 : 0);
        }
        if (tid < BT) {
            const bool ok = tid < nv;
            cp_async4(smem + OFF_BETA + 4 * tid, p.beta + static_cast<size_t>(t0 + (ok ? tid : 0)) * p.H + h, ok ? 4 : 0);
        }
    }
    cp_async_commit();
}

// One (chain, chunk) task: steps 1-4, results into the global slot. Its inputs
// were loaded by issue_loads; `vbuf` holds v (then u), `qlobuf` receives q*a lo
// and then the next task's v. `nxt` (valid or not) is loaded as buffers free up.
__device__ __forceinline__ void run_task(const Params &p, unsigned char *smem, unsigned char *slot, int ch, int c,
                                         int vbuf, int qlobuf, const Task &nxt, bool &gate_bad, bool &range_bad) {
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_Q);
    __nv_bfloat16 *sQlo = reinterpret_cast<__nv_bfloat16 *>(smem + qlobuf);
    __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_K);
    __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(smem + vbuf);
    __half *sRV = reinterpret_cast<__half *>(smem + vbuf);
    __half *sRK = reinterpret_cast<__half *>(smem + OFF_RK);
    float *sG = reinterpret_cast<float *>(smem + OFF_G);
    float *sKB = reinterpret_cast<float *>(smem + OFF_KB);
    __half *sAqk = reinterpret_cast<__half *>(smem + OFF_AQK);
    __half *sL = reinterpret_cast<__half *>(smem + OFF_L);
    float *sLD = reinterpret_cast<float *>(smem + OFF_LD);
    __half *sInv = reinterpret_cast<__half *>(smem + OFF_INV);
    float *sTab = reinterpret_cast<float *>(smem + OFF_TAB);
    float *sBeta = reinterpret_cast<float *>(smem + OFF_BETA);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, qd = lane & 3;
    const float scale = p.scale;
    (void)ch;
    (void)c;
    // ---- step 1: inclusive prefix sum of g (base 2) per key channel, four
    // 16-row quarters per channel on all 512 threads, then the per-channel tables
    {
        const int chn = tid & 127, rq = tid >> 7;
        float x[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) x[q] = sG[(16 * rq + q) * RSF + chn];
        float acc = 0.f;
        bool gb = false;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            gb |= !(x[q] >= p.lb && x[q] <= 0.f);
            acc += x[q] * LOG2E;
            x[q] = acc;
        }
        gate_bad |= gb;
        sTab[TEM + rq * 128 + chn] = acc;  // quarter totals (the EM rows are rebuilt below)
        sync_compute();
        float cy = 0.f;
        for (int q = 0; q < rq; ++q) cy += sTab[TEM + q * 128 + chn];
#pragma unroll
        for (int q = 0; q < 16; ++q) sG[(16 * rq + q) * RSF + chn] = x[q] + cy;
    }
    sync_compute();
    if (tid < DK) {  // rows >= nv carry g = 0, so row 63 holds the last valid prefix
        const int chn = tid;
        float gm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) gm[i] = sG[(16 * i + 7) * RSF + chn];
        const float gl = sG[63 * RSF + chn];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sTab[TGM + i * 128 + chn] = gm[i];
            sTab[TEM + i * 128 + chn] = ex2(gm[i]);
            sTab[TEL + i * 128 + chn] = ex2(gl - gm[i]);
        }
        sTab[TGL + chn] = gl;
        sTab[TD + chn] = ex2(gl);
#pragma unroll
        for (int i = 1; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < i; ++j) sTab[TF + f_pair(i, j) * 128 + chn] = ex2(gm[i] - gm[j]);
    }
    sync_compute();
    KDA_TRACE_EV(p, 21, 0);

    // ---- steps 2a/4a: elementwise operands; q_hat and kg go straight to the slot
    {
        // thread: channels c8..c8+7 of rows r0 and r0 + 8, both in sub-block i
        const int ew_i = tid >> 7, ew_c8 = (tid & 15) << 3, ew_r0 = 16 * ew_i + ((tid >> 4) & 7);
        float Gv[2][8];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int r = ew_r0 + 8 * it, c8 = ew_c8;
            const float4 a = *reinterpret_cast<const float4 *>(sG + r * RSF + c8);
            const float4 b = *reinterpret_cast<const float4 *>(sG + r * RSF + c8 + 4);
            Gv[it][0] = a.x; Gv[it][1] = a.y; Gv[it][2] = a.z; Gv[it][3] = a.w;
            Gv[it][4] = b.x; Gv[it][5] = b.y; Gv[it][6] = b.z; Gv[it][7] = b.w;
        }
        sync_compute();  // the gate tile is free from here on: stream in the next task's g
        if (nxt.valid) issue_loads(p, smem, nxt, 0, 0);
        float GM[8], EM[8], EL[8];
        {
            const int i = ew_i, c8 = ew_c8;
            const float4 a0 = *reinterpret_cast<const float4 *>(sTab + TGM + i * 128 + c8);
            const float4 a1 = *reinterpret_cast<const float4 *>(sTab + TGM + i * 128 + c8 + 4);
            const float4 b0 = *reinterpret_cast<const float4 *>(sTab + TEM + i * 128 + c8);
            const float4 b1 = *reinterpret_cast<const float4 *>(sTab + TEM + i * 128 + c8 + 4);
            const float4 d0 = *reinterpret_cast<const float4 *>(sTab + TEL + i * 128 + c8);
            const float4 d1 = *reinterpret_cast<const float4 *>(sTab + TEL + i * 128 + c8 + 4);
            GM[0] = a0.x; GM[1] = a0.y; GM[2] = a0.z; GM[3] = a0.w; GM[4] = a1.x; GM[5] = a1.y; GM[6] = a1.z; GM[7] = a1.w;
            EM[0] = b0.x; EM[1] = b0.y; EM[2] = b0.z; EM[3] = b0.w; EM[4] = b1.x; EM[5] = b1.y; EM[6] = b1.z; EM[7] = b1.w;
            EL[0] = d0.x; EL[1] = d0.y; EL[2] = d0.z; EL[3] = d0.w; EL[4] = d1.x; EL[5] = d1.y; EL[6] = d1.z; EL[7] = d1.w;
        }
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int r = ew_r0 + 8 * it, c8 = ew_c8;
            const float bt = sBeta[r];
            const uint4 qv = *reinterpret_cast<const uint4 *>(sQ + r * RSB + c8);
            const uint4 kv = *reinterpret_cast<const uint4 *>(sK + r * RSB + c8);
            const uint4 vv = *reinterpret_cast<const uint4 *>(sV + r * RSB + c8);
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(&qv);
            const uint32_t *kw = reinterpret_cast<const uint32_t *>(&kv);
            const uint32_t *vw = reinterpret_cast<const uint32_t *>(&vv);
            uint32_t oQh[4], oQl[4], oKa[4], oBv[4], oBk[4], oQs[4], oKg[4];
            float kb[8];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                const float2 qf = unpack_bf16(qw[q2]), kf = unpack_bf16(kw[q2]), vf = unpack_bf16(vw[q2]);
                float res[2][6];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ce = 2 * q2 + e;
                    const float qq = e ? qf.y : qf.x, kk = e ? kf.y : kf.x, vv2 = e ? vf.y : vf.x;
                    const float x = Gv[it][ce] - GM[ce];
                    const float a = ex2(x), b = ex2(-x);
                    const float eG = a * EM[ce];
                    res[e][0] = qq * a;            // q e^(G - G_m)
                    res[e][1] = kk * a;            // k e^(G - G_m)
                    res[e][2] = bt * vv2;          // beta v
                    res[e][3] = bt * kk * eG;      // beta k e^G
                    res[e][4] = scale * qq * eG;   // scale q e^G
                    res[e][5] = kk * b * EL[ce];   // k e^(G_last - G)
                    kb[ce] = kk * b;               // k e^(G_m - G)
                }
                split_bf16(res[0][0], res[1][0], oQh[q2], oQl[q2]);
                oKa[q2] = pack_bf16(res[0][1], res[1][1]);
                range_bad |= !(f16_ok(res[0][2]) && f16_ok(res[1][2]));
                oBv[q2] = pack_f16(res[0][2], res[1][2]);
                oBk[q2] = pack_f16(res[0][3], res[1][3]);
                oQs[q2] = pack_f16(res[0][4], res[1][4]);
                oKg[q2] = pack_f16(res[0][5], res[1][5]);
            }
            *reinterpret_cast<uint4 *>(sQ + r * RSB + c8) = *reinterpret_cast<uint4 *>(oQh);
            *reinterpret_cast<uint4 *>(sQlo + r * RSB + c8) = *reinterpret_cast<uint4 *>(oQl);
            *reinterpret_cast<uint4 *>(sK + r * RSB + c8) = *reinterpret_cast<uint4 *>(oKa);
            *reinterpret_cast<uint4 *>(sRV + r * RSB + c8) = *reinterpret_cast<uint4 *>(oBv);
            *reinterpret_cast<uint4 *>(sRK + r * RSB + c8) = *reinterpret_cast<uint4 *>(oBk);
            *reinterpret_cast<float4 *>(sKB + r * RSF + c8) = make_float4(kb[0], kb[1], kb[2], kb[3]);
            *reinterpret_cast<float4 *>(sKB + r * RSF + c8 + 4) = make_float4(kb[4], kb[5], kb[6], kb[7]);
            *reinterpret_cast<uint4 *>(slot + SL_A1 + tile_chunk(128, r, c8)) = *reinterpret_cast<uint4 *>(oQs);
            *reinterpret_cast<uint4 *>(slot + SL_KG + tile_chunk(64, r, c8)) = *reinterpret_cast<uint4 *>(oKg);
        }
    }
    sync_compute();
    KDA_TRACE_EV(p, 22, 0);

    // ---- step 2b: Aqk (split bf16, three products) and Akk (bf16) on the 10
    // lower 16x16 tiles. Tile (i,j) needs k_s e^(G_{m_i} - G_s) for s in
    // sub-block j: the stored k e^(G_{m_j} - G) times e^(G_{m_i} - G_{m_j}) (<= 1).
    for (int pair = warp; pair < 10; pair += NWARPS) {
        int i = 0;
        while ((i + 1) * (i + 2) / 2 <= pair) ++i;
        const int j = pair - i * (i + 1) / 2;
        const float *kbrow0 = sKB + (16 * j + gq) * RSF;      // column s = 16j + gq
        const float *kbrow1 = sKB + (16 * j + 8 + gq) * RSF;  // column s = 16j + 8 + gq
        const float *fr = sTab + TF + (i > j ? f_pair(i, j) : 0) * 128;
        float aq[2][4] = {}, ak[2][4] = {};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t fa[4], fl[4], fk[4];
            ldsm_x4(fa, sQ + (16 * i + (lane & 15)) * RSB + 16 * kk + ((lane >> 4) << 3));
            ldsm_x4(fl, sQlo + (16 * i + (lane & 15)) * RSB + 16 * kk + ((lane >> 4) << 3));
            ldsm_x4(fk, sK + (16 * i + (lane & 15)) * RSB + 16 * kk + ((lane >> 4) << 3));
            const int c0 = 16 * kk + 2 * qd;
            float2 f0 = make_float2(1.f, 1.f), f1 = make_float2(1.f, 1.f);
            if (i > j) {
                f0 = *reinterpret_cast<const float2 *>(fr + c0);
                f1 = *reinterpret_cast<const float2 *>(fr + c0 + 8);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float *row = nt ? kbrow1 : kbrow0;
                const float2 x0 = *reinterpret_cast<const float2 *>(row + c0);
                const float2 x1 = *reinterpret_cast<const float2 *>(row + c0 + 8);
                uint32_t bh0, bl0, bh1, bl1;
                split_bf16(x0.x * f0.x, x0.y * f0.y, bh0, bl0);
                split_bf16(x1.x * f1.x, x1.y * f1.y, bh1, bl1);
                mma16816(aq[nt], fa, bh0, bh1);
                mma16816(aq[nt], fl, bh0, bh1);
                mma16816(aq[nt], fa, bl0, bl1);
                mma16816(ak[nt], fk, bh0, bh1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int tl = gq + 8 * hf, sl = 8 * nt + 2 * qd;
                const int t = 16 * i + tl, s = 16 * j + sl;
                const float bt = sBeta[t];
                float vq[2], vk[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool incl = (i > j) || (sl + e <= tl);
                    const bool strict = (i > j) || (sl + e < tl);
                    vq[e] = incl ? scale * aq[nt][2 * hf + e] : 0.f;
                    vk[e] = strict ? bt * ak[nt][2 * hf + e] : 0.f;
                    if (i == j) sLD[(i * 16 + tl) * 17 + sl + e] = vk[e];
                }
                *reinterpret_cast<uint32_t *>(sAqk + t * RSA + s) = pack_f16(vq[0], vq[1]);
                *reinterpret_cast<uint32_t *>(sL + t * RSA + s) = pack_f16(vk[0], vk[1]);
            }
    }
    // upper tiles of scale*Aqk are zero (the consumer reads the full 64x64)
    for (int idx = tid; idx < 6 * 16 * 8; idx += NCOMP) {
        const int tile = idx >> 7, rr = (idx >> 3) & 15, cc = (idx & 7) << 1;
        const int i = tile < 3 ? 0 : (tile < 5 ? 1 : 2);
        const int j = tile < 3 ? tile + 1 : (tile < 5 ? tile - 1 : 3);
        *reinterpret_cast<uint32_t *>(sAqk + (16 * i + rr) * RSA + 16 * j + cc) = 0u;
    }
    sync_compute();
    // q, k, q*a lo, kb and beta are free: stream in the rest of the next task
    if (nxt.valid) issue_loads(p, smem, nxt, 1, qlobuf);
    KDA_TRACE_EV(p, 23, 0);

    // ---- step 3a: (I + L_ii)^-1 for the four diagonal blocks, fp32 substitution
    if (warp < 4 && lane < 16) {
        const int i = warp, jc = lane;
        const float *Ld = sLD + i * 16 * 17;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = (r == jc) ? 1.f : 0.f;
#pragma unroll
            for (int cc = 0; cc < r; ++cc) s -= Ld[r * 17 + cc] * x[cc];
            x[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sInv[(i * 16 + r) * RSI + jc] = __float2half_rn(x[r]);
    }
    sync_compute();
    KDA_TRACE_EV(p, 24, 0);

    // ---- steps 3b/4: X = (I+L)^-1 [beta v | beta k e^G], in place; warp w owns 16 columns
    {
        __half *R = (warp < 8) ? sRV : sRK;
        const int col0 = 16 * (warp & 7);
        for (int i = 0; i < 4; ++i) {
            float acc[2][4] = {};
            for (int j = 0; j < i; ++j) {
                uint32_t fa[4], fb[4];
                ldsm_x4(fa, sL + (16 * i + (lane & 15)) * RSA + 16 * j + ((lane >> 4) << 3));
                ldsm_x4_t(fb, R + bk_off(lane, 16 * j, col0, RSB));
                mma16816_f16(acc[0], fa, fb[0], fb[1]);
                mma16816_f16(acc[1], fa, fb[2], fb[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t *pp = reinterpret_cast<uint32_t *>(R + (16 * i + gq + 8 * hf) * RSB + col0 + 8 * nt + 2 * qd);
                    const float2 rv = unpack_f16(*pp);
                    const float y0 = rv.x - acc[nt][2 * hf], y1 = rv.y - acc[nt][2 * hf + 1];
                    range_bad |= !(f16_ok(y0) && f16_ok(y1));
                    *pp = pack_f16(y0, y1);
                }
            __syncwarp();
            float xo[2][4] = {};
            {
                uint32_t fa[4], fb[4];
                ldsm_x4(fa, sInv + (16 * i + (lane & 15)) * RSI + ((lane >> 4) << 3));
                ldsm_x4_t(fb, R + bk_off(lane, 16 * i, col0, RSB));
                mma16816_f16(xo[0], fa, fb[0], fb[1]);
                mma16816_f16(xo[1], fa, fb[2], fb[3]);
            }
            __syncwarp();
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int rr = 16 * i + gq + 8 * hf, cc = col0 + 8 * nt + 2 * qd;
                    range_bad |= !(f16_ok(xo[nt][2 * hf]) && f16_ok(xo[nt][2 * hf + 1]));
                    *reinterpret_cast<uint32_t *>(R + rr * RSB + cc) = pack_f16(xo[nt][2 * hf], xo[nt][2 * hf + 1]);
                }
            __syncwarp();
        }
    }
    sync_compute();
    KDA_TRACE_EV(p, 25, 0);

    // ---- hand-off: Aqk, u, w and e^(G_last) into the slot (16-byte stores)
    for (int idx = tid; idx < BT * 8; idx += NCOMP) {
        const int r = idx >> 3, c8 = (idx & 7) << 3;
        *reinterpret_cast<uint4 *>(slot + SL_AQK + tile_chunk(64, r, c8)) =
            *reinterpret_cast<const uint4 *>(sAqk + r * RSA + c8);
    }
    for (int idx = tid; idx < BT * 16; idx += NCOMP) {
        const int r = idx >> 4, c8 = (idx & 15) << 3;
        *reinterpret_cast<uint4 *>(slot + SL_U + tile_chunk(64, r, c8)) =
            *reinterpret_cast<const uint4 *>(sRV + r * RSB + c8);
        *reinterpret_cast<uint4 *>(slot + SL_A1 + tile_chunk(128, 64 + r, c8)) =
            *reinterpret_cast<const uint4 *>(sRK + r * RSB + c8);
    }
    if (tid < 32)
        *reinterpret_cast<float4 *>(slot + SL_D + 16 * tid) = *reinterpret_cast<const float4 *>(sTab + TD + 4 * tid);
}

__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int pid) {
    const int tid = threadIdx.x;
    Ring R = ring_of(p);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);
    // longest consumer sequence: tasks beyond it do not exist
    if (tid == 0) misc[1] = 0;
    sync_compute();
    {
        int mx = 0;
        for (int k = tid; k < p.C; k += NCOMP) mx = max(mx, consumer_total(p, k));
        atomicMax(&misc[1], mx);
    }
    sync_compute();
    const int jmax = misc[1];
    auto fetch = [&]() {  // all threads; thread 0 draws, everyone reads after the barrier
        if (tid == 0) {
            const Task t = fetch_task(p, R, jmax);
            misc[2] = t.valid; misc[3] = t.k; misc[4] = t.j; misc[5] = t.ch; misc[6] = t.c;
        }
        sync_compute();
        const Task t{misc[2], misc[3], misc[4], misc[5], misc[6]};
        sync_compute();
        return t;
    };
    Task cur = fetch();
    int vbuf = OFF_V, qlobuf = OFF_QLO;
    if (cur.valid) {
        issue_loads(p, smem, cur, 0, vbuf);
        issue_loads(p, smem, cur, 1, vbuf);
    }
    bool gate_bad = false, range_bad = false;
    while (cur.valid) {
        const Task nxt = fetch();
        const int s = cur.j % RING;
        KDA_TRACE_EV(p, 1, cur.j * p.C + cur.k);
        if (tid == 0)
            misc[7] = (cur.j < RING) ? 1 : (wait_flag_geq(R, &R.freed[cur.k * RING + s], cur.j - RING + 1, p.status) ? 1 : 0);
        cp_async_wait_all();
        sync_compute();
        if (!misc[7]) break;
        KDA_TRACE_EV(p, 20, 0);
        unsigned char *slot = R.slots + static_cast<size_t>(cur.k * RING + s) * SLOT_BYTES;
        run_task(p, smem, slot, cur.ch, cur.c, vbuf, qlobuf, nxt, gate_bad, range_bad);
        sync_compute();  // every thread's slot stores precede the barrier, hence the release below
        if (tid == 0) st_release(&R.ready[cur.k * RING + s], cur.j + 1);
        KDA_TRACE_EV(p, 3, cur.j * p.C + cur.k);
        cur = nxt;
        const int tmp = vbuf;
        vbuf = qlobuf;
        qlobuf = tmp;
    }
    cp_async_wait_all();
    if (gate_bad) set_status(p.status, KDA_ERR_GATE_RANGE);
    if (range_bad) set_status(p.status, KDA_ERR_VALUE_RANGE);
}
}  // namespace prod

// ================================================================== consumer
// Step 5 on the 5th-generation tensor cores. TMEM holds the fp32 state S
// (columns 0-127, lane = key channel) and the accumulator D = [q_hat S ; w S]
// (columns 128-255, lanes 0-63 = tokens of q_hat S, lanes 64-127 = tokens of
// w S). One thread issues the MMAs; all sixteen warps run the epilogues, warp w
// on TMEM lanes 32*(w%4).. and value columns 32*(w/4)..
//   MMA1  D  = [q_hat ; w] (K-major, 128 x 128) * S16 (fp16 snapshot, MN-major)
//   MMA2  D += [scale*Aqk ; 0] (K-major, 128 x 64) * v_new (MN-major)   (lanes 0-63: o)
//   MMA3  S += kg^T (MN-major, 128 x 64) * v_new, after S <- Diag(d) S in TMEM
namespace cons {
constexpr int BUF_BYTES = SLOT_BYTES + 8192;   // slot + 8 KB of zeros: rows 64-127 of [Aqk; 0]
constexpr int OFF_BUF0 = 0;
constexpr int OFF_BUF1 = BUF_BYTES;             // 82944 (1024-aligned)
constexpr int OFF_S = 2 * BUF_BYTES;            // S16: fp16 [key][value], MN-major swizzled, 32 KB
constexpr int OFF_VN = OFF_S + 32768;           // v_new: fp16 [token][value], MN-major swizzled, 16 KB
constexpr int OFF_BAR = OFF_VN + 16384;         // full[2], mma1, mma23
constexpr int OFF_TMEM = OFF_BAR + 32;          // TMEM base address written by tcgen05.alloc
constexpr int OFF_MISC = OFF_BAR + 64;
constexpr int SMEM = OFF_MISC + 64;
constexpr uint32_t TMEM_COLS = 256;
constexpr int OST = 132;                        // fp32 row stride of the o staging tile (64 x OST spans S16 + v_new)
static_assert(64 * OST * 4 <= 32768 + 16384, "o staging fits in the state and v_new tiles");
__device__ __forceinline__ bool f16_ok(float x) { return fabsf(x) < F16_SAFE; }

__device__ __forceinline__ bool wait_all(const Ring &R, uint64_t *bar, uint32_t parity, int32_t *status) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 1023) == 1023 && ld_relaxed(&R.hdr->abort)) return false;
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, slice = warp >> 2;  // TMEM lane quarter, 32-column value slice
    const int row = 32 * quad + lane;             // this thread's TMEM lane
    Ring R = ring_of(p);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *bar_mma1 = full + 2;
    uint64_t *bar_mma23 = full + 3;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);
    unsigned char *sS = smem + OFF_S;
    unsigned char *sVN = smem + OFF_VN;

    for (int i = tid; i < 2 * 512; i += NCOMP)  // the two zero blocks
        *reinterpret_cast<uint4 *>(smem + (i >> 9) * BUF_BYTES + SLOT_BYTES + (i & 511) * 16) = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma23, 1);
        mbar_fence_init();
        misc[0] = 1;
    }
    if (warp == 0) tmem_alloc(tslot, TMEM_COLS);
    fence_proxy_async_shared();
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem + (static_cast<uint32_t>(32 * quad) << 16) + 32 * slice;  // this thread's S columns
    const uint32_t tD = tS + 128;                                                       // this thread's D columns
    const int total = consumer_total(p, k);

    auto issue = [&](int jj) {  // slot jj -> buffer jj % 2 (thread 0)
        const unsigned char *src = R.slots + static_cast<size_t>(k * RING + jj % RING) * SLOT_BYTES;
        unsigned char *dst = smem + ((jj & 1) ? OFF_BUF1 : OFF_BUF0);
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&full[jj & 1], SLOT_BYTES);
        bulk_g2s(dst, src, 32768, &full[jj & 1]);
        bulk_g2s(dst + 32768, src + 32768, 32768, &full[jj & 1]);
        bulk_g2s(dst + 65536, src + 65536, SLOT_BYTES - 65536, &full[jj & 1]);
    };
    bool issued_next = false;  // thread 0 only
    if (tid == 0 && total > 0) {
        if (wait_flag_geq(R, &R.ready[k * RING], 1, p.status))
            issue(0);
        else
            misc[0] = 0;
    }
    const uint32_t idesc_qw = umma_idesc_f16(false, true, 128, 128);  // [q_hat; w] x S16
    const uint32_t idesc_av = umma_idesc_f16(false, true, 128, 128);  // [Aqk; 0] x v_new
    const uint32_t idesc_kv = umma_idesc_f16(true, true, 128, 128);   // kg^T x v_new

    int j = 0;
    bool range_bad = false, alive = true;
    for (int ch = k; ch < p.N * p.H && alive; ch += p.C) {
        int64_t bos, len;
        const int nc = chain_info(p, ch, bos, len);
        if (nc < 0) {
            if (tid == 0) set_status(p.status, KDA_ERR_BAD_SEQLENS);
            continue;
        }
        const int n = ch / p.H, h = ch % p.H;
        const size_t state_base = (static_cast<size_t>(n) * p.H + h) * (DK * DV);
        // initial state (or zeros) -> TMEM: row `row`, columns 32*slice..+31
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t r[16];
            if (p.s0) {
                const float4 *src = reinterpret_cast<const float4 *>(p.s0 + state_base + row * DV + 32 * slice + 16 * cb);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 f = src[e];
                    r[4 * e] = __float_as_uint(f.x); r[4 * e + 1] = __float_as_uint(f.y);
                    r[4 * e + 2] = __float_as_uint(f.z); r[4 * e + 3] = __float_as_uint(f.w);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = 0u;
            }
            tmem_st16(tS + 16 * cb, r);
        }
        tmem_wait_st();

        for (int c = 0; c < nc; ++c, ++j) {
            const int b = j & 1;
            const int64_t t0 = bos + static_cast<int64_t>(c) * BT;
            const int nv = static_cast<int>((bos + len - t0) < BT ? (bos + len - t0) : BT);
            KDA_TRACE_EV(p, 10, j);
            // (1) slot j has landed: release its ring slot, start fetching slot j + 1
            if (tid == 0) {
                if (misc[0] && wait_mbar(R, &full[b], (j >> 1) & 1, p.status)) {
                    fence_proxy_async_global();
                    st_release(&R.freed[k * RING + j % RING], j + 1);
                    issued_next = false;
                    if (j + 1 < total && ld_acquire(&R.ready[k * RING + (j + 1) % RING]) >= j + 2) {
                        issue(j + 1);
                        issued_next = true;
                    }
                } else {
                    misc[0] = 0;
                }
            }
            sync_compute();
            if (!misc[0]) {
                alive = false;
                break;
            }
            for (int it = 0; !mbar_try_wait(&full[b], (j >> 1) & 1); ++it)
                if (it > (1 << 20)) {
                    set_status(p.status, KDA_ERR_TIMEOUT);
                    break;
                }
            const unsigned char *bb = smem + (b ? OFF_BUF1 : OFF_BUF0);
            KDA_TRACE_EV(p, 11, j);

            // (2) fp16 snapshot of the entry state for MMA1, then S <- Diag(d) S in TMEM
            {
                const float d = reinterpret_cast<const float *>(bb + SL_D)[row];
                uint32_t r0[16], r1[16];
                tmem_ld16(tS, r0);
                tmem_ld16(tS + 16, r1);
                tmem_wait_ld();
                auto snap = [&](uint32_t (&r)[16], int cb) {
                    uint32_t hp[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
                        range_bad |= !(f16_ok(x0) && f16_ok(x1));
                        hp[e] = pack_f16(x0, x1);
                    }
                    const int c8 = 32 * slice + 16 * cb;
                    *reinterpret_cast<uint4 *>(sS + tile_chunk(128, row, c8)) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
                    *reinterpret_cast<uint4 *>(sS + tile_chunk(128, row, c8 + 8)) = make_uint4(hp[4], hp[5], hp[6], hp[7]);
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * d);
                };
                snap(r0, 0);
                snap(r1, 1);
                tmem_st16(tS, r0);
                tmem_st16(tS + 16, r1);
                tmem_wait_st();
            }
            fence_proxy_async_shared();
            tc_fence_before();
            sync_compute();
            KDA_TRACE_EV(p, 13, j);

            // (3) MMA1: D = [q_hat ; w] S16
            if (tid == 0) {
                tc_fence_after();
                const uint32_t a0 = smem_u32(bb + SL_A1), b0 = smem_u32(sS);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_f16(tmem + 128, umma_desc_sw128(a0 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                             umma_desc_sw128(b0 + kk * 2048, 16384, 1024), idesc_qw, kk > 0);
                umma_commit(bar_mma1);
            }

            // (4) v_new = u - w S (TMEM lanes 64-127) -> fp16 [token][value] tile
            wait_all(R, bar_mma1, j & 1, p.status);
            tc_fence_after();
            KDA_TRACE_EV(p, 14, j);
            if (quad >= 2) {
                const int t = row - 64;
                uint32_t r0[16], r1[16];
                tmem_ld16(tD, r0);
                tmem_ld16(tD + 16, r1);
                tmem_wait_ld();
                auto vnew = [&](const uint32_t (&r)[16], int cb) {
                    const int c8 = 32 * slice + 16 * cb;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint4 uu = *reinterpret_cast<const uint4 *>(bb + SL_U + tile_chunk(64, t, c8 + 8 * hh));
                        const uint32_t *uw = reinterpret_cast<const uint32_t *>(&uu);
                        uint32_t vp[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 u2 = unpack_f16(uw[e]);
                            const float y0 = u2.x - __uint_as_float(r[8 * hh + 2 * e]);
                            const float y1 = u2.y - __uint_as_float(r[8 * hh + 2 * e + 1]);
                            range_bad |= !(f16_ok(y0) && f16_ok(y1));
                            vp[e] = pack_f16(y0, y1);
                        }
                        *reinterpret_cast<uint4 *>(sVN + tile_chunk(64, t, c8 + 8 * hh)) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
                    }
                };
                vnew(r0, 0);
                vnew(r1, 1);
            }
            fence_proxy_async_shared();
            tc_fence_before();
            sync_compute();
            KDA_TRACE_EV(p, 15, j);

            // (5) MMA2: D[0:64] += (scale Aqk) v_new ; MMA3: S += kg^T v_new
            if (tid == 0) {
                tc_fence_after();
                const uint32_t aq = smem_u32(bb + SL_AQK), vn = smem_u32(sVN), kg = smem_u32(bb + SL_KG);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f16(tmem + 128, umma_desc_sw128(aq + kk * 32, 16, 1024), umma_desc_sw128(vn + kk * 2048, 8192, 1024),
                             idesc_av, 1);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f16(tmem, umma_desc_sw128(kg + kk * 2048, 8192, 1024), umma_desc_sw128(vn + kk * 2048, 8192, 1024),
                             idesc_kv, 1);
                umma_commit(bar_mma23);
            }

            // (6) o (TMEM lanes 0-63) -> staging in the (now free) state/v_new tiles ->
            // global, one full 512-byte row per warp store
            wait_all(R, bar_mma23, j & 1, p.status);
            tc_fence_after();
            KDA_TRACE_EV(p, 16, j);
            float *stg = reinterpret_cast<float *>(sS);  // [64][OST] fp32, spans the S16 and v_new tiles
            if (quad < 2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tD, r0);
                tmem_ld16(tD + 16, r1);
                tmem_wait_ld();
                float *dst = stg + row * OST + 32 * slice;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    reinterpret_cast<float4 *>(dst)[e] = make_float4(__uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                                                                     __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3]));
                    reinterpret_cast<float4 *>(dst + 16)[e] = make_float4(__uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                                                                          __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3]));
                }
            }
            tc_fence_before();
            sync_compute();
            for (int rr = warp; rr < nv; rr += NCOMP / 32)
                reinterpret_cast<float4 *>(p.o + (static_cast<size_t>(t0 + rr) * p.H + h) * DV)[lane] =
                    *reinterpret_cast<const float4 *>(stg + rr * OST + 4 * lane);
            KDA_TRACE_EV(p, 12, j);
            if (tid == 0 && !issued_next && j + 1 < total) {
                if (wait_flag_geq(R, &R.ready[k * RING + (j + 1) % RING], j + 2, p.status))
                    issue(j + 1);
                else
                    misc[0] = 0;
            }
        }
        if (!alive) break;
        // final state: TMEM -> global
        if (p.sT) {
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t r[16];
                tmem_ld16(tS + 16 * cb, r);
                tmem_wait_ld();
                float4 *dst = reinterpret_cast<float4 *>(p.sT + state_base + row * DV + 32 * slice + 16 * cb);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                         __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
            }
        }
    }
    if (range_bad) set_status(p.status, KDA_ERR_VALUE_RANGE);
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}
}  // namespace cons

constexpr int SMEM_MAX = (prod::SMEM > cons::SMEM ? prod::SMEM : cons::SMEM) + 1024;  // + alignment slack
static_assert(SMEM_MAX <= 232448, "shared memory budget");

__global__ void __launch_bounds__(NTHREADS, 1) kda_persistent_kernel(const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    if (static_cast<int>(blockIdx.x) < p.C)
        cons::run(p, smem, blockIdx.x);
    else
        prod::run(p, smem, blockIdx.x - p.C);
}

// ------------------------------------------------------------------ host side
static int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

int consumers_for(int64_t chains, int grid) {
    int64_t c = grid / 2;
    if (c < 1) c = 1;
    if (chains < c) c = chains;
    return static_cast<int>(c < 1 ? 1 : c);
}

size_t workspace_bytes(int64_t chains) {
    const int sms = num_sms();
    if (sms < 2 || chains < 1) return 0;
    const int C = consumers_for(chains, sms);
    size_t bytes = ring_offset(C) + static_cast<size_t>(C) * RING * SLOT_BYTES;
#ifdef KDA_TRACE
    bytes += static_cast<size_t>(sms) * (TRACE_EVENTS * 2 + 1) * 8;
#endif
    return bytes;
}

cudaError_t launch(Params p, size_t ws_bytes, cudaStream_t stream) {
    const int sms = num_sms();
    if (sms < 2) return cudaErrorInvalidDevice;
    cudaError_t e = cudaFuncSetAttribute(kda_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_persistent_kernel, NTHREADS, SMEM_MAX);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = sms;  // one CTA per SM; all co-resident (cooperative launch)
    p.C = consumers_for(static_cast<int64_t>(p.N) * p.H, grid);
    if (ws_bytes < ring_offset(p.C) + static_cast<size_t>(p.C) * RING * SLOT_BYTES) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(p.ws, 0, ring_offset(p.C), stream);
    if (e != cudaSuccess) return e;
#ifdef KDA_TRACE
    e = cudaMemsetAsync(p.ws + ring_offset(p.C) + static_cast<size_t>(p.C) * RING * SLOT_BYTES, 0,
                        static_cast<size_t>(grid) * (TRACE_EVENTS * 2 + 1) * 8, stream);
    if (e != cudaSuccess) return e;
#endif
    void *args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(kda_persistent_kernel), dim3(grid), dim3(NTHREADS),
                                       args, SMEM_MAX, stream);
}

}  // namespace pers
}  // namespace kda
