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

#include <cmath>
#include "kda.h"
#include "kda_common.cuh"
#include "kda_persistent.h"

namespace kda {
namespace pers {

constexpr int NCOMP = 512;            // 16 warps, all computing (<= 128 registers each)
constexpr int NTHREADS = NCOMP;
constexpr int NWARPS = NCOMP / 32;
constexpr long long SPIN_LIMIT = 1ll << 24;         // polls before a wait gives up (normal calls)
constexpr long long SPIN_LIMIT_DEBUG = 1ll << 14;   // the same under KDA_DEBUG_WITHHOLD_READY
#ifdef KDA_TRACE
constexpr int TRACE_COUNTS_OFFSET = 231424;  // past every role's tiles (checked below), 16 ints
#endif

// ---------------------------------------------------------------- slot layout
// A slot holds one (chain, chunk) hand-off; every region is 1024-byte aligned.
//   A1  [q_hat ; w]  fp16, 128 rows x 128 key channels, K-major, 128B swizzle
//   KG  kg           fp16, [token][key] (64 x 128): the transposed operand kg^T
//   U   u            fp16, [token][value] (64 x 128)
//   D   e^(G_last)   fp32, 128
//   AQK scale * Aqk  fp16, [t][s] (64 x 64), causal incl. diagonal
//   T   T = (I + L)^-1 fp16, [t][s] (64 x 64), lower block triangle: only in
//       the launches where the consumers form the WY product (then A1's rows
//       64-127 hold beta k e^G and U holds beta v instead of w and u), whose
//       ring slots are SLOT_BYTES apart; otherwise slots are SL_T apart
// 128-byte swizzle: row r of a 128-byte-wide atom column keeps its 16-byte
// chunk c at position c ^ (r mod 8); wider tiles are split into 64-element
// atom columns stored one after the other.
constexpr int SL_A1 = 0, SL_KG = 32768, SL_U = 49152, SL_D = 65536, SL_AQK = 66560, SL_T = 74752;
static_assert(SLOT_BYTES == SL_T + 8192, "slot size");
template <bool WY> constexpr int SLOT_STRIDE = WY ? SLOT_BYTES : SL_T;  // WY: the consumers form the WY product

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

// Optional event trace (compiled in only with -DKDA_TRACE): per CTA and warp,
// up to TRACE_EVENTS records {globaltimer ns, tag << 32 | value} after the ring
// in the workspace, written by lane 0 of the warp; per-warp counts live in
// shared memory (past the roles' tiles) and are mirrored to the workspace.
#ifdef KDA_TRACE
constexpr int TRACE_EVENTS = 512;
constexpr size_t TRACE_CTA_WORDS = 16 + 16 * TRACE_EVENTS * 2;
__device__ __forceinline__ void trace_any(const Params &p, int tag, int value) {
    extern __shared__ unsigned char smem_raw[];
    int *cnt = reinterpret_cast<int *>(smem_raw + TRACE_COUNTS_OFFSET);
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    const int w = threadIdx.x >> 5;
    unsigned char *base = p.ws + ring_offset(p.Cws) + static_cast<size_t>(p.Cws) * RING * SLOT_BYTES;
    unsigned long long *rec = reinterpret_cast<unsigned long long *>(base) + blockIdx.x * TRACE_CTA_WORDS;
    const int n = cnt[w];
    if (n < TRACE_EVENTS) {
        unsigned long long *r = rec + 16 + (static_cast<size_t>(w) * TRACE_EVENTS + n) * 2;
        r[0] = t;
        r[1] = (static_cast<unsigned long long>(tag) << 32) | static_cast<unsigned>(value);
        cnt[w] = n + 1;
        rec[w] = n + 1;
    }
}
__device__ __forceinline__ void trace(const Params &p, int tag, int value) {
    if (threadIdx.x != 0) return;
    trace_any(p, tag, value);
}
#define KDA_TRACE_EV(p, tag, value) trace(p, tag, value)
#define KDA_TRACE_ANY(p, tag, value) trace_any(p, tag, value)
#else
#define KDA_TRACE_EV(p, tag, value) ((void)0)
#define KDA_TRACE_ANY(p, tag, value) ((void)0)
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
    int *freed2; // [C][RING]: the same for the second CTA of a consumer whose columns are split
    unsigned char *slots;
    long long spin;  // polls before a wait gives up
};

__device__ __forceinline__ Ring ring_of(const Params &p) {
    Ring r;
    r.hdr = reinterpret_cast<Header *>(p.ws);
    r.ready = reinterpret_cast<int *>(p.ws + sizeof(Header));
    r.freed = r.ready + p.C * RING;
    r.freed2 = r.freed + p.C * RING;
    r.slots = p.ws + ring_offset(p.C);
    r.spin = p.spin;
    return r;
}

__device__ __forceinline__ bool wait_flag_geq(const Ring &R, const int *flag, int target, int32_t *status) {
    for (long long it = 0; it < R.spin; ++it) {
        if (ld_acquire(flag) >= target) return true;
        if ((it & 127) == 127 && ld_relaxed(&R.hdr->abort)) return false;
        __nanosleep(64);
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

__device__ __forceinline__ bool wait_mbar(const Ring &R, uint64_t *bar, uint32_t parity, int32_t *status) {
    for (long long it = 0; it < R.spin; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 127) == 127 && ld_relaxed(&R.hdr->abort)) return false;
        __nanosleep(32);
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

// After an abort: wait (bounded, ignoring the abort word) for this CTA's own
// bulk copies on `bar` to land before it leaves.
__device__ __forceinline__ void drain_mbar(uint64_t *bar, uint32_t parity) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return;
        __nanosleep(64);
    }
}

// chunks of chain ch (sequence ch / H), or -1 when its bounds are invalid;
// `cu` is p.cu or a copy of it in shared memory. The sequence's first token is
// cu[n], or seq_bos[n] when that map is given.
__device__ __forceinline__ int chain_info(const Params &p, const int32_t *cu, int ch, int64_t &bos, int64_t &len) {
    const int n = ch / p.H;
    const int64_t b = cu[n], e = cu[n + 1];
    const int64_t s = p.seq_bos ? static_cast<int64_t>(p.seq_bos[n]) : b;
    const bool bad = b < 0 || e < b || e > p.T || (n == 0 && b != 0) || (n == p.N - 1 && e != p.T) || s < 0 ||
                     s + (e - b) > p.Ttok;
    if (bad) {
        bos = 0;
        len = 0;
        return -1;
    }
    bos = s;
    len = e - b;
    return static_cast<int>((len + BT - 1) / BT);
}

// ------------------------------------------------------------ chain schedule
// Which chains each consumer runs, in order. When every sequence has the same
// number of chunks, consumer k takes chains k, k + C, k + 2C, ... (no table).
// Otherwise, for at most SCHED_MAX_CHAINS chains and when its cost (about
// 150 ns per sequence) is small against the run, every CTA builds the same
// table at start-up (deterministically, in shared memory): sequences in
// decreasing order of their chunk count hand their H chains to the H consumers
// with the least work so far (ties to the lower index), the longest-first
// greedy rule, so that unequal lengths do not leave one consumer with most of
// the work. order[cstart[k] .. cstart[k + 1]) lists consumer k's chains.
// The same region keeps a copy of cu_seqlens (when it has at most CU_CACHE
// entries) for both roles: the ring's acquire loads invalidate L1, so global
// reads of it would go to L2 on every task.
constexpr int SCHED_MAX_CHAINS = 1024, SCHED_MAX_C = 160, CU_CACHE = 1024;
constexpr int SCHED_CU = 16 + 4 * (SCHED_MAX_C + 1) + 4 * SCHED_MAX_CHAINS;  // byte offset of the cu copy
constexpr int SCHED_BYTES = SCHED_CU + 4 * CU_CACHE;
// The schedule sits at OFF_SCHED of every CTA's shared memory, past both roles'
// tiles: int flags[4] (table present, cu copy present), cstart, order, cu copy.
constexpr int OFF_SCHED = 215168;  // = the consumer's tiles, the larger role (checked below)
__device__ __forceinline__ const int *sched_flags(const unsigned char *smem) {
    return reinterpret_cast<const int *>(smem + OFF_SCHED);
}
// cu_seqlens: the shared-memory copy, or p.cu
__device__ __forceinline__ const int32_t *sched_cu(const Params &p, const unsigned char *smem) {
    return sched_flags(smem)[1] ? reinterpret_cast<const int32_t *>(smem + OFF_SCHED + SCHED_CU) : p.cu;
}
// number of chains of consumer k, and its r-th chain
__device__ __forceinline__ int sched_count(const Params &p, const unsigned char *smem, int k) {
    const int *f = sched_flags(smem);
    return f[0] ? f[4 + k + 1] - f[4 + k] : (p.N * p.H - k + p.C - 1) / p.C;
}
__device__ __forceinline__ int sched_chain(const Params &p, const unsigned char *smem, int k, int r) {
    const int *f = sched_flags(smem);
    return f[0] ? f[4 + SCHED_MAX_C + 1 + f[4 + k] + r] : k + r * p.C;
}

// Builds the schedule into `sched` on all threads of the CTA; `scratch` (at
// least 8 KB + 8 * SCHED_MAX_CHAINS bytes) is free shared memory for the duration.
__device__ void build_sched(const Params &p, unsigned char *sched, unsigned char *scratch) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int N = p.N, H = p.H, C = p.C, chains = N * H;
    int *flag = reinterpret_cast<int *>(sched);
    int *cstart = flag + 4, *order = cstart + SCHED_MAX_C + 1;
    const bool cache_cu = N + 1 <= CU_CACHE;
    int32_t *cuc = reinterpret_cast<int32_t *>(sched + SCHED_CU);
    int *nchk = reinterpret_cast<int *>(scratch);          // chunks per sequence
    int *sorted = nchk + SCHED_MAX_CHAINS;                   // sequences by decreasing chunks
    int *load = sorted + SCHED_MAX_CHAINS;                   // chunks given to each consumer
    int *cnt = load + SCHED_MAX_C;                           // chains given to each consumer
    int *asg = cnt + SCHED_MAX_C;                            // per chain: consumer << 16 | position
    const bool fits = chains <= SCHED_MAX_CHAINS && C <= SCHED_MAX_C && N > 0;
    // warp 0: copy cu_seqlens and find whether the sequences differ in chunk count
    if (tid < 32) {
        bool uneq = false;
        int first = 0;
        long long chunks = 0;  // chunks of all sequences (one head)
        for (int n0 = 0; n0 <= N; n0 += 32) {
            const int n = n0 + tid;
            int32_t b = 0, e = 0;
            if (n <= N) {
                b = p.cu[n];
                if (cache_cu) cuc[n] = b;
            }
            if (n < N) e = p.cu[n + 1];
            const int nc = (n < N && e > b && b >= 0) ? static_cast<int>((static_cast<int64_t>(e) - b + BT - 1) / BT) : 0;
            if (n0 == 0) first = __shfl_sync(0xffffffffu, nc, 0);
            if (fits && n < N) nchk[n] = nc;
            uneq |= __any_sync(0xffffffffu, n < N && nc != first);
            chunks += nc;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) chunks += __shfl_xor_sync(0xffffffffu, chunks, o);
        // the table costs about 150 ns per sequence in every CTA; build it only
        // when that is under 2 % of the producers' expected time (~7 us per chunk)
        const long long prod_ns = chunks * H * 7000 / (static_cast<int>(gridDim.x) - C > 0 ? static_cast<int>(gridDim.x) - C : 1);
        const bool worth = N <= 256 && static_cast<long long>(N) * 150 * 50 <= prod_ns;
        if (tid == 0) {
            flag[0] = (fits && uneq && worth) ? 1 : 0;
            flag[1] = cache_cu ? 1 : 0;
        }
    }
    __syncthreads();
    if (!flag[0]) return;
    for (int n = tid; n < N; n += nthr) {
        int r = 0;
        for (int m = 0; m < N; ++m) r += (nchk[m] > nchk[n]) || (nchk[m] == nchk[n] && m < n);
        sorted[r] = n;
    }
    for (int k = tid; k < C; k += nthr) {
        load[k] = 0;
        cnt[k] = 0;
    }
    __syncthreads();
    for (int i = 0; i < N; ++i) {
        const int n = sorted[i], w = nchk[n];
        for (int h0 = 0; h0 < H; h0 += C) {  // the sequence's chains, at most C at a time
            const int take = H - h0 < C ? H - h0 : C;
            int rk = C;
            if (tid < C) {
                const int lk = load[tid];
                rk = 0;
                for (int m = 0; m < C; ++m) rk += (load[m] < lk) || (load[m] == lk && m < tid);
            }
            __syncthreads();
            if (tid < C && rk < take) {
                asg[n * H + h0 + rk] = (tid << 16) | cnt[tid];
                ++cnt[tid];
                load[tid] += w;
            }
            __syncthreads();
        }
    }
    if (tid == 0) {
        int acc = 0;
        for (int k = 0; k < C; ++k) {
            cstart[k] = acc;
            acc += cnt[k];
        }
        cstart[C] = acc;
    }
    __syncthreads();
    for (int ch = tid; ch < chains; ch += nthr) order[cstart[asg[ch] >> 16] + (asg[ch] & 0xffff)] = ch;
    __syncthreads();
}

// total chunks of consumer k (its chains' chunks form one sequence)
__device__ __forceinline__ int consumer_total(const Params &p, const unsigned char *sc, const int32_t *cu, int k) {
    int tot = 0;
    int64_t b, l;
    if (!sched_flags(sc)[0]) {
        for (int ch = k; ch < p.N * p.H; ch += p.C) {
            const int nc = chain_info(p, cu, ch, b, l);
            tot += nc > 0 ? nc : 0;
        }
        return tot;
    }
    const int nchains = sched_count(p, sc, k);
    for (int r = 0; r < nchains; ++r) {
        const int nc = chain_info(p, cu, sched_chain(p, sc, k, r), b, l);
        tot += nc > 0 ? nc : 0;
    }
    return tot;
}

// chunk j of consumer k: its chain, the chunk's index in the chain and the chain's bounds
__device__ __forceinline__ bool map_task(const Params &p, const unsigned char *sc, const int32_t *cu, int k, int j, int &ch_out,
                                         int &c_out, int64_t &bos, int64_t &len) {
    const bool table = sched_flags(sc)[0] != 0;
    const int *row = sched_flags(sc) + 4 + SCHED_MAX_C + 1 + (table ? sched_flags(sc)[4 + k] : 0);
    const int nchains = table ? sched_count(p, sc, k) : 0;
    for (int r = 0, ch = k;; ++r, ch += p.C) {
        if (table) {
            if (r >= nchains) return false;
            ch = row[r];
        } else if (ch >= p.N * p.H) {
            return false;
        }
        int64_t b, l;
        int nc = chain_info(p, cu, ch, b, l);
        if (nc < 0) nc = 0;
        if (j < nc) {
            ch_out = ch;
            c_out = j;
            bos = b;
            len = l;
            return true;
        }
        j -= nc;
    }
}

// ================================================================== producer
// Steps 1-4 for one (chain, chunk) task at a time on all sixteen warps, with
// warp-level tensor-core products (m16n8k16) for the 16x16 tiles. The task's
// ring slot is assembled in shared memory (the slot image) and leaves with one
// bulk store; while warps 0-9 compute the strips, one thread of the idle last
// warp publishes the previous slot, draws the next task and waits for this
// task's slot to be free, so none of that memory traffic stalls the warps.
// Round an fp32 value to tf32 (nearest, ties away from zero) for a tf32 MMA
// operand: adding half a tf32 unit in the last place to the sign-magnitude bit
// pattern carries into bit 13 exactly when the dropped 13 bits are at least
// half of it, and the MMA reads only the upper 19 bits. Finite inputs only.
__device__ __forceinline__ uint32_t tf32_rna(float x) { return __float_as_uint(x) + 0x1000u; }

namespace prod {
// q, k, v and their derived tiles are [64 tokens][128 channels] 16-bit tiles
// and g is a [64][128] fp32 tile, all in the 128-byte-swizzled layout the
// input copies write (16 KB and 32 KB; 1024-byte aligned).
constexpr int RSF = 136, RSA = 72;
constexpr int SZ_T = BT * DK * 2;             // 16384
constexpr int SZ_F = BT * RSF * 4;            // 34816 (kb keeps a padded row stride)
constexpr int OFF_IMG = 0;                    // slot image: a ring slot up to T (T has its own tile, OFF_T)
constexpr int OFF_Q = OFF_IMG + SL_T;         // q; then q*a as tf32 (fp32 [64][128], spans OFF_Q and OFF_QLO)
constexpr int OFF_QLO = OFF_Q + SZ_T;
constexpr int OFF_K = OFF_QLO + SZ_T;         // k -> k*a (bf16)
constexpr int OFF_V = OFF_K + SZ_T;           // v (bf16)
constexpr int OFF_GKB = OFF_V + SZ_T;         // g -> G (fp32, swizzled), then k*e^(G_m - G) (fp32, padded)
constexpr int SZ_A = BT * RSA * 2;            // 9216
constexpr int OFF_L = OFF_GKB + SZ_F;         // L (fp16 [64][RSA])
constexpr int OFF_LD = OFF_L + SZ_A;          // diagonal blocks of L, fp32 [4][16][17]
constexpr int OFF_T = OFF_LD + 4352;          // T = (I+L)^-1, fp16 [64][RSA] (lower blocks); with WY
                                              // the swizzled [64][64] tile the consumer reads
constexpr int OFF_TAB = OFF_T + SZ_A;         // per-channel tables, fp32 [20][128]
constexpr int OFF_BETA = OFF_TAB + 10240;
constexpr int OFF_MISC = OFF_BETA + 256;      // flags and the task broadcast (32 ints)
constexpr int OFF_GPAR = OFF_MISC + 128;      // raw gates: the task head's dt_bias row (128 fp32) and A_log
constexpr int SMEM = OFF_GPAR + 528;
static_assert(OFF_GPAR % 16 == 0, "cp.async destinations are 16-byte aligned");
// Warp w runs on sub-partition w % 4. During the strips, warps 0-9 hold the
// ten tiles (three on partitions 0 and 1, two on 2 and 3); the diagonal
// inverses run on warps 10, 11, 14, 15 (partitions 2 and 3) and the ring work,
// mostly waiting, on warps 12 and 13 (partitions 0 and 1).
constexpr int BAR_TB = 6;                     // WY: named barrier of warps 0-2 building T's block diagonals
constexpr int SYNC_TID = 13 * 32;             // lane 0 of warp 13: draws tasks
constexpr int REL_TID = 12 * 32;              // lane 0 of warp 12: waits for free slots, stores and publishes images
constexpr int TGM = 0, TGL = 4 * 128, TEM = 5 * 128, TEL = 9 * 128, TF = 13 * 128, TD = 19 * 128;
static_assert(OFF_Q % 1024 == 0 && OFF_GKB % 1024 == 0, "swizzled tiles are 1024-byte aligned");
// byte offset of the 16-byte chunk holding channels [c4, c4+4) of row r of the g tile
__device__ __forceinline__ int g_chunk(int r, int c4) {
    return (c4 >> 5) * (BT * 128) + r * 128 + ((((c4 >> 2) & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ int g_elem(int r, int c) { return g_chunk(r, c & ~3) + ((c & 3) << 2); }
// q*a tile, fp32 [64][128]: channel pair c/2 of row r is stored at pair
// (c/2) ^ 4(r mod 4), so the strip loads (8 bytes at rows g, channels 2q + 16k)
// are free of bank conflicts and a group of 4 pairs stays 32 contiguous bytes
__device__ __forceinline__ int qa_pair(int r, int c) { return r * 512 + ((((c >> 1) ^ ((r & 3) << 2))) << 3); }
__device__ __forceinline__ int f_pair(int i, int j) { return i * (i - 1) / 2 + j; }
// The image leaves in two bulk stores: q_hat (rows 0-63 of A1) and kg as soon
// as the elementwise step has written them, the rest after the solve.
__device__ __forceinline__ void store_early(unsigned char *dst, const unsigned char *img) {
    fence_proxy_async_global();  // after the acquire that found the slot free
    bulk_s2g(dst + SL_A1, img + SL_A1, 8192);                  // q_hat, channels 0-63
    bulk_s2g(dst + SL_A1 + 16384, img + SL_A1 + 16384, 8192);  // q_hat, channels 64-127
    bulk_s2g(dst + SL_KG, img + SL_KG, SL_U - SL_KG);          // kg
    bulk_commit();
}
// (With WY, w and u are beta k e^G and beta v, and T follows from its own tile.)
template <bool WY>
__device__ __forceinline__ void store_late(unsigned char *dst, const unsigned char *img) {
    bulk_s2g(dst + SL_A1 + 8192, img + SL_A1 + 8192, 8192);    // w, channels 0-63
    bulk_s2g(dst + SL_A1 + 24576, img + SL_A1 + 24576, 8192);  // w, channels 64-127
    bulk_s2g(dst + SL_U, img + SL_U, SL_T - SL_U);             // u, e^(G_last), scale*Aqk
    if constexpr (WY) bulk_s2g(dst + SL_T, img + (OFF_T - OFF_IMG), 8192);  // T
    bulk_commit();
}
static_assert(SL_KG == 32768 && SL_U == 49152 && SL_D == 65536 && SL_AQK > SL_D, "slot layout used by the stores");

// slot-image byte offsets of u (token rows of U) and w (rows 64-127 of A1)
__device__ __forceinline__ int uw_chunk(bool isw, int r, int c8) {
    return isw ? SL_A1 + tile_chunk(128, 64 + r, c8) : SL_U + tile_chunk(64, r, c8);
}
__device__ __forceinline__ int uw_elem(bool isw, int r, int c) { return uw_chunk(isw, r, c & ~7) + ((c & 7) << 1); }
__device__ __forceinline__ int uw_bk(bool isw, int lane, int k0, int n0) {  // ldmatrix.trans lane address, B [k][n]
    return isw ? SL_A1 + bk_addr(lane, 128, 64 + k0, n0) : SL_U + bk_addr(lane, 64, k0, n0);
}

// A task and where its tokens are: t0 = first token of the chunk, nv = its
// valid rows, h = its head (computed once when the task is drawn).
struct Task {
    int valid, k, j, ch, c, t0, nv, h;
};
__device__ __forceinline__ void put_task(int *m, const Task &t) {
    m[0] = t.valid; m[1] = t.k; m[2] = t.j; m[3] = t.ch; m[4] = t.c; m[5] = t.t0; m[6] = t.nv; m[7] = t.h;
}
__device__ __forceinline__ Task get_task(const int *m) { return Task{m[0], m[1], m[2], m[3], m[4], m[5], m[6], m[7]}; }

// Tasks are numbered j * C + k (chunk j of consumer k), so every consumer
// advances together; producer pid takes the numbers pid, pid + P, pid + 2P,
// ... in order. The cursor holds the next number as (k, j) and the stride P
// as (P mod C, P div C), so that drawing divides nothing.
struct Cursor {
    int k, j, dk, dj;
};
__device__ __forceinline__ Cursor make_cursor(int pid, int P, int C) { return Cursor{pid % C, pid / C, P % C, P / C}; }

// next valid task of the cursor (numbers whose consumer has fewer chunks are skipped)
__device__ __forceinline__ Task fetch_task(const Params &p, const unsigned char *sc, const int32_t *cu, int jmax, Cursor &cs) {
    Task t{0, 0, 0, 0, 0, 0, 0, 0};
    while (cs.j < jmax) {
        t.k = cs.k;
        t.j = cs.j;
        cs.k += cs.dk;
        cs.j += cs.dj;
        if (cs.k >= p.C) {
            cs.k -= p.C;
            ++cs.j;
        }
        int64_t bos, len;
        if (map_task(p, sc, cu, t.k, t.j, t.ch, t.c, bos, len)) {
            const int64_t t0 = bos + static_cast<int64_t>(t.c) * BT;
            t.t0 = static_cast<int>(t0);
            t.nv = static_cast<int>((bos + len - t0) < BT ? (bos + len - t0) : BT);
            t.h = t.ch % p.H;
            t.valid = 1;
            return t;
        }
    }
    return t;
}

// One task's inputs into shared memory, called by all threads once the
// buffers are free: 16-byte cp.async copies into the 128-byte-swizzled tile
// layouts, g (fp32) in a first commit group, q, k, v (bf16) and beta in a
// second, so the prefix sum can start before q, k and v land. Rows past the
// sequence end are zero-filled (g = 0 keeps row 63 of G at the last valid
// prefix; k = v = beta = 0 rows are inert in every product).
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *smem, const Task &tk) {
    const int tid = threadIdx.x;
    // rows [t0, t0 + nv) of head h; a failed index check zero-fills the task's tiles
    const bool inb = checked(tk.t0 >= 0 && tk.nv >= 0 && tk.nv <= BT && static_cast<int64_t>(tk.t0) + tk.nv <= p.Ttok &&
                                 tk.h >= 0 && tk.h < p.H,
                             p.status);
    const int t0 = inb ? tk.t0 : 0, nv = inb ? tk.nv : 0, h = inb ? tk.h : 0;
    const size_t rs = static_cast<size_t>(p.H) * DK;  // token stride, elements
    const size_t hb = static_cast<size_t>(h) * DK;
    KDA_TRACE_EV(p, 30, 0);
#pragma unroll
    for (int it = 0; it < BT * 32 / NCOMP; ++it) {  // g: 64 rows x 32 chunks of 4 channels
        const int idx = tid + it * NCOMP, r = idx >> 5, c4 = (idx & 31) << 2;
        const bool ok = r < nv;
        cp_async16(smem + OFF_GKB + g_chunk(r, c4), p.g + static_cast<size_t>(t0 + (ok ? r : 0)) * rs + hb + c4,
                   ok ? 16 : 0);
    }
    if (p.raw && tid < 33) {  // the gate activation's per-head parameters (zeros when not given)
        if (tid < 32)
            cp_async16(smem + OFF_GPAR + 16 * tid, p.dt_bias ? p.dt_bias + hb + 4 * tid : p.g, p.dt_bias ? 16 : 0);
        else
            cp_async4(smem + OFF_GPAR + 512, p.A_log ? p.A_log + h : p.g, p.A_log ? 4 : 0);
    }
    cp_async_commit();
#pragma unroll
    for (int it = 0; it < BT * 16 / NCOMP; ++it) {  // q, k, v: 64 rows x 16 chunks of 8 channels
        const int idx = tid + it * NCOMP, r = idx >> 4, c8 = (idx & 15) << 3;
        const bool ok = r < nv;
        const size_t off = static_cast<size_t>(t0 + (ok ? r : 0)) * rs + hb + c8;
        const int d = tile_chunk(64, r, c8);
        cp_async16(smem + OFF_Q + d, p.q + off, ok ? 16 : 0);
        cp_async16(smem + OFF_K + d, p.k + off, ok ? 16 : 0);
        cp_async16(smem + OFF_V + d, p.v + off, ok ? 16 : 0);
    }
    if (tid >= NCOMP - BT) {  // warps 14 and 15
        const int r = tid - (NCOMP - BT);
        const bool ok = r < nv;
        cp_async4(smem + OFF_BETA + 4 * r, p.beta + static_cast<size_t>(t0 + (ok ? r : 0)) * p.H + h, ok ? 4 : 0);
    }
    cp_async_commit();
}

// One (chain, chunk) task: steps 1-4 into the slot image, then the bulk store
// of the image into the task's slot. Its inputs were loaded by issue_loads.
// `nxt` is the next task (drawn one task earlier); its input copies start
// right after the strips.
// During the strips, REL_TID completes and publishes the previous task's slot
// (`pending` = its ready-flag index or -1, `pending_val` the value) while
// SYNC_TID draws the task after `nxt` into `nxt2` and waits for this task's
// slot to be free. The publication waits only for this CTA's own bulk store,
// never for a consumer, so a producer never waits on a consumer while its
// finished chunk stays unpublished (and tasks drawn but not started wait on
// nothing: the lowest-numbered unpublished task can always proceed).
// Returns false when the slot wait gave up (timeout or abort).
template <bool WY, bool HALF>  // the consumers form the WY product; each consumer is two CTAs (column halves)
__device__ __forceinline__ bool run_task(const Params &p, const Ring &Rg, unsigned char *smem, const Task &cur,
                                         const int32_t *cu_s, int jmax, const Task &nxt, Task &nxt2, Cursor &cs, int &pending,
                                         int pending_val, bool &gate_bad, float &vmax) {
    unsigned char *img = smem + OFF_IMG;
    unsigned char *sQ = smem + OFF_Q, *sK = smem + OFF_K, *sV = smem + OFF_V;
    unsigned char *sGb = smem + OFF_GKB;  // G, swizzled (g_chunk / g_elem)
    float *sKB = reinterpret_cast<float *>(smem + OFF_GKB);
    __half *sL = reinterpret_cast<__half *>(smem + OFF_L);
    float *sLD = reinterpret_cast<float *>(smem + OFF_LD);
    __half *sT = reinterpret_cast<__half *>(smem + OFF_T);
    float *sTab = reinterpret_cast<float *>(smem + OFF_TAB);
    float *sBeta = reinterpret_cast<float *>(smem + OFF_BETA);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, qd = lane & 3;
    const float scale = p.scale;
    // ---- step 1: inclusive prefix sum of g (base 2) per key channel, four
    // 16-row quarters per channel on all 512 threads, then the per-channel tables
    {
        const int chn = tid & 127, rq = tid >> 7;
        float x[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) x[q] = *reinterpret_cast<const float *>(sGb + g_elem(16 * rq + q, chn));
        if (p.raw) {  // g = lower_bound * sigmoid(e^A_log (g_raw + dt_bias)); rows past the sequence end stay 0
            const float *gp = reinterpret_cast<const float *>(smem + OFF_GPAR);
            const float a = __expf(gp[128]), db = gp[chn];
#pragma unroll
            for (int q = 0; q < 16; ++q)
                x[q] = (16 * rq + q < cur.nv) ? __fdividef(p.lb, 1.f + __expf(-a * (x[q] + db))) : 0.f;
        }
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
        for (int q = 0; q < 16; ++q) *reinterpret_cast<float *>(sGb + g_elem(16 * rq + q, chn)) = x[q] + cy;
    }
    sync_compute();
    if (tid < DK) {  // rows >= nv carry g = 0, so row 63 holds the last valid prefix
        const int chn = tid;
        float gm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) gm[i] = *reinterpret_cast<const float *>(sGb + g_elem(16 * i + 7, chn));
        const float gl = *reinterpret_cast<const float *>(sGb + g_elem(63, chn));
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
    if (tid == REL_TID) bulk_wait_read();  // the previous image has been read out and may be rewritten
    cp_async_wait_all();  // q, k, v and beta
    sync_compute();
    if (p.raw) {  // beta = sigmoid(beta_raw); rows past the sequence end stay 0
        if (tid < BT) sBeta[tid] = tid < cur.nv ? __fdividef(1.f, 1.f + __expf(-sBeta[tid])) : 0.f;
        sync_compute();
    }
    KDA_TRACE_EV(p, 21, 0);

    // ---- steps 2a/4a: elementwise operands; q_hat, kg, beta*v and
    // beta*k*e^G go straight into the slot image
    {
        // warp w: rows 4w .. 4w+3 (all in sub-block w / 4); lane: channels
        // 4 lane .. 4 lane + 3, so that every fp32 access of a warp is one
        // contiguous 512-byte row and every 16-bit one a 256-byte row
        const int ew_i = warp >> 2, c4 = lane << 2, r0 = warp << 2;
        const int h8 = (c4 & 4) << 1;  // byte offset of these 4 channels in their 16-byte chunk
        float4 Gv[4];
        uint2 qv[4], kv[4], vv[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = r0 + it;
            Gv[it] = *reinterpret_cast<const float4 *>(sGb + g_chunk(r, c4));
            const int tc = tile_chunk(64, r, c4 & ~7) + h8;
            qv[it] = *reinterpret_cast<const uint2 *>(sQ + tc);
            kv[it] = *reinterpret_cast<const uint2 *>(sK + tc);
            vv[it] = *reinterpret_cast<const uint2 *>(sV + tc);
        }
        sync_compute();  // G and q are read: kb and q*a overwrite them below
        const float4 GM = *reinterpret_cast<const float4 *>(sTab + TGM + ew_i * 128 + c4);
        const float4 EM = *reinterpret_cast<const float4 *>(sTab + TEM + ew_i * 128 + c4);
        const float4 EL = *reinterpret_cast<const float4 *>(sTab + TEL + ew_i * 128 + c4);
        const float gm[4] = {GM.x, GM.y, GM.z, GM.w}, em[4] = {EM.x, EM.y, EM.z, EM.w}, el[4] = {EL.x, EL.y, EL.z, EL.w};
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int r = r0 + it;
            const float bt = sBeta[r];
            const float gv[4] = {Gv[it].x, Gv[it].y, Gv[it].z, Gv[it].w};
            const uint32_t qw[2] = {qv[it].x, qv[it].y}, kw[2] = {kv[it].x, kv[it].y}, vw[2] = {vv[it].x, vv[it].y};
            uint32_t oQa[4], oKa[2], oBv[2], oBk[2], oQs[2], oKg[2];
            float kb[4];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                const float2 qf = unpack_bf16(qw[q2]), kf = unpack_bf16(kw[q2]), vf = unpack_bf16(vw[q2]);
                float res[2][6];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ce = 2 * q2 + e;
                    const float qq = e ? qf.y : qf.x, kk = e ? kf.y : kf.x, vv2 = e ? vf.y : vf.x;
                    const float x = gv[ce] - gm[ce];
                    const float a = ex2(x), b = ex2(-x);
                    const float eG = a * em[ce];
                    res[e][0] = qq * a;            // q e^(G - G_m)
                    res[e][1] = kk * a;            // k e^(G - G_m)
                    res[e][2] = bt * vv2;          // beta v
                    res[e][3] = bt * kk * eG;      // beta k e^G
                    res[e][4] = scale * qq * eG;   // scale q e^G
                    res[e][5] = kk * b * el[ce];   // k e^(G_last - G)
                    kb[ce] = kk * b;               // k e^(G_m - G)
                }
                oQa[2 * q2] = tf32_rna(res[0][0]);
                oQa[2 * q2 + 1] = tf32_rna(res[1][0]);
                oKa[q2] = pack_bf16(res[0][1], res[1][1]);
#pragma unroll
                for (int e = 0; e < 2; ++e)
#pragma unroll
                    for (int o = 2; o < 6; ++o) vmax = max_abs_nan(vmax, res[e][o]);
                oBv[q2] = pack_f16(res[0][2], res[1][2]);
                oBk[q2] = pack_f16(res[0][3], res[1][3]);
                oQs[q2] = pack_f16(res[0][4], res[1][4]);
                oKg[q2] = pack_f16(res[0][5], res[1][5]);
            }
            const int tc = tile_chunk(64, r, c4 & ~7) + h8;
            *reinterpret_cast<uint4 *>(sQ + qa_pair(r, c4)) = make_uint4(oQa[0], oQa[1], oQa[2], oQa[3]);
            *reinterpret_cast<uint2 *>(sK + tc) = make_uint2(oKa[0], oKa[1]);
            *reinterpret_cast<float4 *>(sKB + r * RSF + c4) = make_float4(kb[0], kb[1], kb[2], kb[3]);
            *reinterpret_cast<uint2 *>(img + uw_chunk(false, r, c4 & ~7) + h8) = make_uint2(oBv[0], oBv[1]);
            *reinterpret_cast<uint2 *>(img + uw_chunk(true, r, c4 & ~7) + h8) = make_uint2(oBk[0], oBk[1]);
            *reinterpret_cast<uint2 *>(img + SL_A1 + tile_chunk(128, r, c4 & ~7) + h8) = make_uint2(oQs[0], oQs[1]);
            *reinterpret_cast<uint2 *>(img + SL_KG + tile_chunk(64, r, c4 & ~7) + h8) = make_uint2(oKg[0], oKg[1]);
        }
        if (tid < 32)
            *reinterpret_cast<float4 *>(img + SL_D + 16 * tid) = *reinterpret_cast<const float4 *>(sTab + TD + 4 * tid);
    }
    // the image parts just written are read by the early bulk store, and the
    // input tiles just written (q*a, k*a, kb) are rewritten by the next tensor
    // copies: order these generic writes before both
    fence_proxy_async_shared();
    sync_compute();
    KDA_TRACE_EV(p, 22, 0);

    // ---- ring work, on warps 12 and 13 (no strip pair, no diagonal block).
    // REL_TID: publish the previous slot, then wait for this task's slot and
    // send the part of the image that is final already. SYNC_TID: draw.
    const bool slot_inb = checked(cur.k >= 0 && cur.k < p.C && cur.j >= 0, p.status);
    unsigned char *dst = Rg.slots + static_cast<size_t>(slot_inb ? cur.k * RING + cur.j % RING : 0) * SLOT_STRIDE<WY>;
    if (tid == REL_TID) {
        if (pending >= 0) {
            bulk_wait_all();
            fence_proxy_async_global();
            if (!(p.debug & KDA_DEBUG_WITHHOLD_READY)) st_release(&Rg.ready[pending], pending_val);
            pending = -1;
        }
        KDA_TRACE_ANY(p, 31, 0);
        const int s = cur.j % RING;
        const bool free_ok =
            slot_inb && ((cur.j < RING) || (wait_flag_geq(Rg, &Rg.freed[cur.k * RING + s], cur.j - RING + 1, p.status) &&
                                            (!HALF || wait_flag_geq(Rg, &Rg.freed2[cur.k * RING + s], cur.j - RING + 1, p.status))));
        misc[20] = free_ok ? 1 : 0;
        if (free_ok) store_early(dst, img);
        KDA_TRACE_ANY(p, 33, 0);
    }
    if (tid == SYNC_TID) {
        const Task t = fetch_task(p, smem, cu_s, jmax, cs);
        put_task(misc + 2, t);
        KDA_TRACE_ANY(p, 35, 0);
    }
    // ---- step 2b: Aqk (tf32) and Akk (bf16) on the 10
    // lower 16x16 tiles, one tile per warp. Tile (i,j) needs k_s e^(G_{m_i} - G_s)
    // for s in sub-block j: the stored k e^(G_{m_j} - G) times e^(G_{m_i} - G_{m_j}) (<= 1).
    static_assert(NWARPS == 16, "warps 0-9 strips, 10, 11, 14, 15 diagonal inverses, 12-13 ring work");
    // Warp w runs on sub-partition w % 4, so warps 0-9 leave partitions 0 and 1
    // with three tiles and 2 and 3 with two: the diagonal tiles (pairs 0, 2, 5,
    // 9), whose L_ii feed the inverses, go to warps 2, 3, 6, 7 on the lighter ones.
    if (warp < 10) {
        const int pair = (0x8795642031ull >> (4 * warp)) & 15;  // warp -> pair: 1 3 0 2 4 6 5 9 7 8
        int i = 0;
        while ((i + 1) * (i + 2) / 2 <= pair) ++i;
        const int j = pair - i * (i + 1) / 2;
        const float *kbrow0 = sKB + (16 * j + gq) * RSF;      // column s = 16j + gq
        const float *kbrow1 = sKB + (16 * j + 8 + gq) * RSF;  // column s = 16j + 8 + gq
        const float *fr = sTab + TF + (i > j ? f_pair(i, j) : 0) * 128;
        float aq[2][4] = {}, ak[2][4] = {};
        // Aqk on tf32 (m16n8k8), Akk on bf16 (m16n8k16). Within each 16-channel
        // step the tf32 k slots are permuted (slot q <-> channel 2q, slot q+4 <->
        // channel 2q+1, for each half) so that one 8-byte load of the scaled
        // k row feeds both the tf32 and the bf16 B fragments.
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int c0 = 16 * kk + 2 * qd;
            uint32_t fa0[4], fa1[4], fk[4];
            {
                const uint2 u00 = *reinterpret_cast<const uint2 *>(sQ + qa_pair(16 * i + gq, c0));
                const uint2 u10 = *reinterpret_cast<const uint2 *>(sQ + qa_pair(16 * i + gq + 8, c0));
                const uint2 u01 = *reinterpret_cast<const uint2 *>(sQ + qa_pair(16 * i + gq, c0 + 8));
                const uint2 u11 = *reinterpret_cast<const uint2 *>(sQ + qa_pair(16 * i + gq + 8, c0 + 8));
                fa0[0] = u00.x; fa0[1] = u10.x; fa0[2] = u00.y; fa0[3] = u10.y;
                fa1[0] = u01.x; fa1[1] = u11.x; fa1[2] = u01.y; fa1[3] = u11.y;
            }
            ldsm_x4(fk, sK + a_addr(lane, 64, 16 * i, 16 * kk));
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
                const float b00 = x0.x * f0.x, b01 = x0.y * f0.y, b10 = x1.x * f1.x, b11 = x1.y * f1.y;
                mma1688_tf32(aq[nt], fa0, tf32_rna(b00), tf32_rna(b01));
                mma1688_tf32(aq[nt], fa1, tf32_rna(b10), tf32_rna(b11));
                mma16816(ak[nt], fk, pack_bf16(b00, b01), pack_bf16(b10, b11));
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
                    vmax = max_abs_nan(max_abs_nan(vmax, vq[e]), vk[e]);
                }
                *reinterpret_cast<uint32_t *>(img + SL_AQK + tile_elem(64, t, s)) = pack_f16(vq[0], vq[1]);
                *reinterpret_cast<uint32_t *>(sL + t * RSA + s) = pack_f16(vk[0], vk[1]);
            }
        if (i == j) {  // L_ii is in place: hand it to the inverse warp of block i
            __syncwarp();
            named_bar_arrive(2 + i, 64);
        }
        if (lane == 0) KDA_TRACE_ANY(p, 40 + warp, 0);
    }
    // ---- step 3a, on warps 10, 11, 14, 15 (blocks 0-3) while the strips run:
    // T_ii = (I + L_ii)^-1 by fp32 forward substitution, once the warp with
    // tile (i, i) has written L_ii
    if (warp == 10 || warp == 11 || warp == 14 || warp == 15) {
        const int i = (warp & 1) | ((warp & 4) >> 1);
        named_bar_sync(2 + i, 64);
        if (lane < 16) {
            const int jc = lane;
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
            for (int r = 0; r < 16; ++r) {
                vmax = max_abs_nan(vmax, x[r]);
                if constexpr (WY)
                    *reinterpret_cast<__half *>(smem + OFF_T + tile_elem(64, 16 * i + r, 16 * i + jc)) = __float2half_rn(x[r]);
                else
                    sT[(16 * i + r) * RSA + 16 * i + jc] = __float2half_rn(x[r]);
            }
        }
        if (lane == 0) KDA_TRACE_ANY(p, 50 + i, 0);
    }
    sync_compute();  // the strips only read the input tiles: their values are in registers by now
    nxt2 = get_task(misc + 2);
    const bool slot_ok = misc[20] != 0;
    // q, k, v, q*a lo, kb and beta are free: stream in the next task
    if (nxt.valid) issue_loads(p, smem, nxt);
    if (!slot_ok) return false;
    KDA_TRACE_EV(p, 23, 0);

    if constexpr (WY) {
        // ---- step 3b alone (the consumers form the WY product): block
        // diagonal d of T on warps 0 .. 3-d, block (w + d, w) on warp w,
        // T_ij = -T_ii * sum_{k=j}^{i-1} L_ik T_kj, in the swizzled tile the
        // late store sends
        unsigned char *sTw = smem + OFF_T;
        if (warp < 3) {
#pragma unroll
            for (int d = 1; d < 4; ++d) {
                if (warp < 4 - d) {
                    const int j = warp, i = warp + d;
                    float m[2][4] = {};
                    for (int kb = j; kb < i; ++kb) {
                        uint32_t fa[4], fb[4];
                        ldsm_x4(fa, sL + (16 * i + (lane & 15)) * RSA + 16 * kb + ((lane >> 4) << 3));
                        ldsm_x4_t(fb, sTw + bk_addr(lane, 64, 16 * kb, 16 * j));
                        mma16816_f16(m[0], fa, fb[0], fb[1]);
                        mma16816_f16(m[1], fa, fb[2], fb[3]);
                    }
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            vmax = max_abs_nan(max_abs_nan(vmax, m[nt][2 * hf]), m[nt][2 * hf + 1]);
                            *reinterpret_cast<uint32_t *>(sTw + tile_elem(64, 16 * i + gq + 8 * hf, 16 * j + 8 * nt + 2 * qd)) =
                                pack_f16(m[nt][2 * hf], m[nt][2 * hf + 1]);
                        }
                    __syncwarp();
                    float t[2][4] = {};
                    {
                        uint32_t fa[4], fb[4];
                        ldsm_x4(fa, sTw + a_addr(lane, 64, 16 * i, 16 * i));
                        ldsm_x4_t(fb, sTw + bk_addr(lane, 64, 16 * i, 16 * j));
                        mma16816_f16(t[0], fa, fb[0], fb[1]);
                        mma16816_f16(t[1], fa, fb[2], fb[3]);
                    }
                    __syncwarp();
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            vmax = max_abs_nan(max_abs_nan(vmax, t[nt][2 * hf]), t[nt][2 * hf + 1]);
                            *reinterpret_cast<uint32_t *>(sTw + tile_elem(64, 16 * i + gq + 8 * hf, 16 * j + 8 * nt + 2 * qd)) =
                                pack_f16(-t[nt][2 * hf], -t[nt][2 * hf + 1]);
                        }
                }
                if (d < 3) named_bar_sync(BAR_TB, 96);  // block diagonal d is complete
            }
        }
    } else {
    // ---- steps 3b and 4, interleaved. Block row i of X = [u | w] =
    // T [beta v | beta k e^G] needs block rows 0..i of T = (I + L)^-1 only, so
    // while all warps compute X_i, warps 0 .. 2-i build block diagonal i+1 of T:
    // T_ij = -T_ii * sum_{k=j}^{i-1} L_ik T_kj. X is written in place in the
    // slot image (u in U, w in rows 64-127 of A1); warp w owns 16 columns and
    // holds all four row blocks of them in registers before it writes any.
    {
        const bool isw = warp >= 8;
        const int col0 = 16 * (warp & 7);
        uint32_t rb[4][4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) ldsm_x4_t(rb[kb], img + uw_bk(isw, lane, 16 * kb, col0));
#pragma unroll
        for (int xi = 0; xi < 4; ++xi) {
            const int d = xi + 1;
            if (d < 4 && warp < 4 - d) {
                const int j = warp, i = warp + d;
                float m[2][4] = {};
                for (int kb = j; kb < i; ++kb) {
                    uint32_t fa[4], fb[4];
                    ldsm_x4(fa, sL + (16 * i + (lane & 15)) * RSA + 16 * kb + ((lane >> 4) << 3));
                    ldsm_x4_t(fb, sT + bk_off(lane, 16 * kb, 16 * j, RSA));
                    mma16816_f16(m[0], fa, fb[0], fb[1]);
                    mma16816_f16(m[1], fa, fb[2], fb[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        vmax = max_abs_nan(max_abs_nan(vmax, m[nt][2 * hf]), m[nt][2 * hf + 1]);
                        *reinterpret_cast<uint32_t *>(sT + (16 * i + gq + 8 * hf) * RSA + 16 * j + 8 * nt + 2 * qd) =
                            pack_f16(m[nt][2 * hf], m[nt][2 * hf + 1]);
                    }
                __syncwarp();
                float t[2][4] = {};
                {
                    uint32_t fa[4], fb[4];
                    ldsm_x4(fa, sT + (16 * i + (lane & 15)) * RSA + 16 * i + ((lane >> 4) << 3));
                    ldsm_x4_t(fb, sT + bk_off(lane, 16 * i, 16 * j, RSA));
                    mma16816_f16(t[0], fa, fb[0], fb[1]);
                    mma16816_f16(t[1], fa, fb[2], fb[3]);
                }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        vmax = max_abs_nan(max_abs_nan(vmax, t[nt][2 * hf]), t[nt][2 * hf + 1]);
                        *reinterpret_cast<uint32_t *>(sT + (16 * i + gq + 8 * hf) * RSA + 16 * j + 8 * nt + 2 * qd) =
                            pack_f16(-t[nt][2 * hf], -t[nt][2 * hf + 1]);
                    }
            }
            float acc[2][4] = {};
#pragma unroll
            for (int kb = 0; kb <= xi; ++kb) {
                uint32_t fa[4];
                ldsm_x4(fa, sT + (16 * xi + (lane & 15)) * RSA + 16 * kb + ((lane >> 4) << 3));
                mma16816_f16(acc[0], fa, rb[kb][0], rb[kb][1]);
                mma16816_f16(acc[1], fa, rb[kb][2], rb[kb][3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int rr = 16 * xi + gq + 8 * hf, cc = col0 + 8 * nt + 2 * qd;
                    vmax = max_abs_nan(max_abs_nan(vmax, acc[nt][2 * hf]), acc[nt][2 * hf + 1]);
                    *reinterpret_cast<uint32_t *>(img + uw_elem(isw, rr, cc)) = pack_f16(acc[nt][2 * hf], acc[nt][2 * hf + 1]);
                }
            if (xi < 3) sync_compute();  // block diagonal d of T is complete
        }
    }
    }
    KDA_TRACE_EV(p, 24, 0);
    fence_proxy_async_shared();  // this thread's image writes, before the bulk store reads them
    sync_compute();
    KDA_TRACE_EV(p, 25, 0);

    // ---- hand-off: the rest of the image (published by REL_TID during the
    // next task's strips, or after the last task)
    if (tid == REL_TID) store_late<WY>(dst, img);
    return true;
}

template <bool WY, bool HALF>
__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int pid) {
    const int tid = threadIdx.x;
    Ring R = ring_of(p);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);
    const int32_t *cu_s = sched_cu(p, smem);  // sequence bounds (in shared memory when small enough)
    // longest consumer sequence: tasks beyond it do not exist
    if (tid == 0) misc[1] = 0;
    sync_compute();
    {
        int mx = 0;
        for (int k = tid; k < p.C; k += NCOMP) mx = max(mx, consumer_total(p, smem, cu_s, k));
        atomicMax(&misc[1], mx);
    }
    // the upper 16x16 tiles of scale*Aqk are never written: zero them once
    for (int idx = tid; idx < 6 * 16 * 8; idx += NCOMP) {
        const int tile = idx >> 7, rr = (idx >> 3) & 15, cc = (idx & 7) << 1;
        const int i = tile < 3 ? 0 : (tile < 5 ? 1 : 2);
        const int j = tile < 3 ? tile + 1 : (tile < 5 ? tile - 1 : 3);
        *reinterpret_cast<uint32_t *>(smem + OFF_IMG + SL_AQK + tile_elem(64, 16 * i + rr, 16 * j + cc)) = 0u;
        if constexpr (WY) *reinterpret_cast<uint32_t *>(smem + OFF_T + tile_elem(64, 16 * i + rr, 16 * j + cc)) = 0u;  // and of T
    }
    sync_compute();
    const int jmax = misc[1];
    Cursor cs = make_cursor(pid, static_cast<int>(gridDim.x) - (HALF ? 2 : 1) * p.C, p.C);  // used by SYNC_TID
    if (tid == SYNC_TID) {
        const Task t = fetch_task(p, smem, cu_s, jmax, cs);
        put_task(misc + 2, t);
        const Task u = fetch_task(p, smem, cu_s, jmax, cs);
        put_task(misc + 10, u);
    }
    sync_compute();
    Task cur = get_task(misc + 2);
    Task nxt = get_task(misc + 10);
    sync_compute();
    if (cur.valid) issue_loads(p, smem, cur);
    bool gate_bad = false;
    float vmax = 0.f;  // largest magnitude packed into an fp16 operand (NaN if any was NaN)
    int pending = -1, pending_val = 0;  // REL_TID: the last slot stored but not yet published
    while (cur.valid) {
        KDA_TRACE_EV(p, 1, cur.j * p.C + cur.k);
        cp_async_wait_group1();  // g (q, k, v and beta may still be in flight)
        sync_compute();
        KDA_TRACE_EV(p, 20, 0);
        Task nxt2{0, 0, 0, 0, 0, 0, 0, 0};
        if (!run_task<WY, HALF>(p, R, smem, cur, cu_s, jmax, nxt, nxt2, cs, pending, pending_val, gate_bad, vmax))
            break;
        if (tid == REL_TID) {
            pending = cur.k * RING + cur.j % RING;
            pending_val = cur.j + 1;
        }
        KDA_TRACE_EV(p, 3, cur.j * p.C + cur.k);
        cur = nxt;
        nxt = nxt2;
    }
    if (tid == REL_TID) {
        bulk_wait_all();
        if (pending >= 0) {
            fence_proxy_async_global();
            if (!(p.debug & KDA_DEBUG_WITHHOLD_READY)) st_release(&R.ready[pending], pending_val);
        }
    }
    cp_async_wait_all();
    if (gate_bad) set_status(p.status, KDA_ERR_GATE_RANGE);
    if (!(vmax < F16_SAFE)) set_status(p.status, KDA_ERR_VALUE_RANGE);
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
// When the consumers form the WY product (WY), A1 holds [q_hat ; beta k e^G]
// and U holds beta v, so the v_new step yields Z = beta v - beta k e^G S, and
//   MMAT  V  = [scale*Aqk ; T] (K-major, 128 x 64) * Z (MN-major)   (lanes 64-127: v_new = T Z)
// goes into TMEM columns 256-383 before MMA2 and MMA3; the T tile then takes
// the place of the zeros in MMA2, whose rows 64-127 land in the consumed
// lanes 64-127 of D.
namespace cons {
constexpr int BUF_BYTES = SL_T + 8192;          // slot + 8 KB of zeros (or T): rows 64-127 of [Aqk; 0]
constexpr int OFF_BUF0 = 0;
constexpr int OFF_BUF1 = BUF_BYTES;             // 82944 (1024-aligned)
constexpr int OFF_S = 2 * BUF_BYTES;            // S16: fp16 [key][value], MN-major swizzled, 32 KB
constexpr int OFF_VN = OFF_S + 32768;           // v_new: fp16 [token][value], MN-major swizzled, 16 KB
constexpr int OFF_BAR = OFF_VN + 16384;         // full[2], mma1, mma23
constexpr int OFF_TMEM = OFF_BAR + 32;          // TMEM base address written by tcgen05.alloc
constexpr int OFF_BAR_T = OFF_BAR + 40;         // WY: MMAT's barrier
constexpr int OFF_MISC = OFF_BAR + 64;
constexpr int SMEM = OFF_MISC + 64;
constexpr uint32_t TMEM_COLS = 256;
constexpr int OST = 132;  // fp32 row stride of the o staging tile (64 x OST spans S16 + v_new); columns
                          // 128-131 hold the row's four slice sums of squares for the gated norm
static_assert(64 * OST * 4 <= 32768 + 16384, "o staging fits in the state and v_new tiles");

// one 128-byte line of global memory towards L2 (no register result)
__device__ __forceinline__ void prefetch_l2(const void *ptr) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}
// logistic function of a bf16 pair, as an fp16 pair: 1/2 + tanh(x/2)/2 with the
// packed fp16 hardware tanh (one special-function operation per pair; absolute
// error about 1e-3)
__device__ __forceinline__ uint32_t sigmoid_bf16x2_to_f16x2(uint32_t g2) {
    const float2 g = unpack_bf16(g2);
    const uint32_t hx = pack_f16(0.5f * g.x, 0.5f * g.y);
    uint32_t t, r;
    asm("tanh.approx.f16x2 %0, %1;" : "=r"(t) : "r"(hx));
    asm("fma.rn.f16x2 %0, %1, %2, %2;" : "=r"(r) : "r"(t), "r"(0x38003800u));  // t * 1/2 + 1/2
    return r;
}

// 3-D tiled tensor store shared memory -> global (coordinates innermost
// first), tracked by the issuing thread's bulk async-groups
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}

// completion of this CTA's own MMAs: depends on no other CTA, so only a
// (bounded) timeout ends it early, never the abort word
__device__ __forceinline__ bool wait_all(const Ring &R, uint64_t *bar, uint32_t parity, int32_t *status) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

template <bool WY, bool HALF>  // the consumers form the WY product; this CTA is one column half
__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int k, int half) {
    // value columns of this CTA: all 128, or with HALF the half [v0, v0 + 64)
    // (column j of v_new, o and S depends on column j of S alone)
    constexpr int NV = HALF ? 64 : 128, NCT = NV / 4;  // columns of the CTA; of a thread's slice
    const int v0 = HALF ? 64 * half : 0;
    const __nv_bfloat16 *ngate = HALF ? nullptr : p.ngate;  // (a split consumer has no whole rows to norm)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, slice = warp >> 2;  // TMEM lane quarter, NCT-column value slice
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
        *reinterpret_cast<uint4 *>(smem + (i >> 9) * BUF_BYTES + SL_T + (i & 511) * 16) = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma23, 1);
        if constexpr (WY) mbar_init(reinterpret_cast<uint64_t *>(smem + OFF_BAR_T), 1);
        mbar_fence_init();
        misc[0] = 1;
    }
    if (warp == 0) tmem_alloc(tslot, WY ? 2 * TMEM_COLS : TMEM_COLS);  // WY: + V
    fence_proxy_async_shared();
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem + (static_cast<uint32_t>(32 * quad) << 16) + NCT * slice;  // this thread's S columns
    const uint32_t tD = tS + 128;                                                       // this thread's D columns
    const int32_t *cu_s = sched_cu(p, smem);
    const int total = consumer_total(p, smem, cu_s, k);

    // slot jj -> buffer jj % 2 (thread 0). The buffer last staged the o of
    // chunk jj - 2 for its tensor stores: they must have read it first.
    // `newest_elsewhere`: this thread's newest store group staged in the
    // other buffer and may go on.
    auto issue = [&](int jj, bool newest_elsewhere) {
        const unsigned char *src = R.slots + static_cast<size_t>(k * RING + jj % RING) * SLOT_STRIDE<WY>;
        unsigned char *dst = smem + ((jj & 1) ? OFF_BUF1 : OFF_BUF0);
        if (newest_elsewhere)
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        else
            bulk_wait_read();
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&full[jj & 1], SLOT_STRIDE<WY>);
        bulk_g2s(dst, src, SLOT_STRIDE<WY>, &full[jj & 1]);
    };
    bool issued_next = false;  // thread 0 only
    if (tid == 0 && total > 0) {
        if (wait_flag_geq(R, &R.ready[k * RING], 1, p.status))
            issue(0, false);
        else
            misc[0] = 0;
    }
    const uint32_t idesc_qw = umma_idesc_f16(false, true, 128, NV);  // [q_hat; w] x S16
    const uint32_t idesc_av = umma_idesc_f16(false, true, 128, NV);  // [Aqk; 0] x v_new
    const uint32_t idesc_kv = umma_idesc_f16(true, true, 128, NV);   // kg^T x v_new

    int j = 0;
    bool alive = true;
    float vmax = 0.f;  // largest magnitude packed into an fp16 operand (NaN if any was NaN)
    const int nchains = sched_count(p, smem, k);
    for (int r = 0; r < nchains && alive; ++r) {
        const int ch = sched_chain(p, smem, k, r);
        int64_t bos, len;
        const int nc = chain_info(p, cu_s, ch, bos, len);
        if (nc < 0) {
            if (tid == 0) set_status(p.status, KDA_ERR_BAD_SEQLENS);
            continue;
        }
        const int n = ch / p.H, h = ch % p.H;
        const bool st_inb = checked(ch >= 0 && n < p.N, p.status);  // a failed check skips the state accesses
        const size_t state_base = st_inb ? (static_cast<size_t>(n) * p.H + h) * (DK * DV) : 0;
        // initial state (or zeros) -> TMEM: row `row`, columns v0 + NCT*slice .. +NCT-1
#pragma unroll
        for (int cb = 0; cb < NCT / 16; ++cb) {
            uint32_t r[16];
            if (p.s0 && st_inb) {
                const float4 *src = reinterpret_cast<const float4 *>(p.s0 + state_base + row * DV + v0 + NCT * slice + 16 * cb);
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
            const int nv_c = static_cast<int>((bos + len - t0) < BT ? (bos + len - t0) : BT);
            // output rows [t0, t0 + nv); a failed index check writes none of them
            const int nv = checked(t0 >= 0 && nv_c >= 0 && t0 + nv_c <= p.Ttok, p.status) ? nv_c : 0;
            KDA_TRACE_EV(p, 10, j);
            // (1) slot j has landed: release its ring slot, start fetching slot j + 1
            if (tid == 0) {
                const bool was_alive = misc[0] != 0;  // then slot j's copy has been issued
                if (was_alive && wait_mbar(R, &full[b], (j >> 1) & 1, p.status)) {
                    // the copy of slot j has completed (its reads are done): free the
                    // slot without ordering this thread's pending o stores before it
                    st_relaxed(&((HALF && half) ? R.freed2 : R.freed)[k * RING + j % RING], j + 1);
                    issued_next = false;
                    // with tensor stores of o, the copy goes after MMA1 instead (the
                    // previous chunk's o stores then have had time to read its buffer;
                    // a part copied earlier shares the copy unit with them and lands later)
                    if (!p.o_tma && j + 1 < total && ld_acquire(&R.ready[k * RING + (j + 1) % RING]) >= j + 2) {
                        issue(j + 1, false);
                        issued_next = true;
                        KDA_TRACE_ANY(p, 17, j + 1);
                    }
                } else {
                    if (was_alive) drain_mbar(&full[b], (j >> 1) & 1);  // let it land before leaving
                    misc[0] = 0;
                }
            }
            sync_compute();
            if (!misc[0]) {
                alive = false;
                break;
            }
            if (ngate && tid < 2 * BT && (tid >> 1) < nv)  // this chunk's gate rows (two lines each) -> L2
                prefetch_l2(ngate + (static_cast<size_t>(t0 + (tid >> 1)) * p.H + h) * DV + 64 * (tid & 1));
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
                if constexpr (NCT > 16) tmem_ld16(tS + 16, r1);
                tmem_wait_ld();
                auto snap = [&](uint32_t (&r)[16], int cb) {
                    uint32_t hp[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
                        vmax = max_abs_nan(max_abs_nan(vmax, x0), x1);
                        hp[e] = pack_f16(x0, x1);
                    }
                    const int c8 = NCT * slice + 16 * cb;
                    *reinterpret_cast<uint4 *>(sS + tile_chunk(128, row, c8)) = make_uint4(hp[0], hp[1], hp[2], hp[3]);
                    *reinterpret_cast<uint4 *>(sS + tile_chunk(128, row, c8 + 8)) = make_uint4(hp[4], hp[5], hp[6], hp[7]);
#pragma unroll
                    for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * d);
                };
                snap(r0, 0);
                if constexpr (NCT > 16) snap(r1, 1);
                tmem_st16(tS, r0);
                if constexpr (NCT > 16) tmem_st16(tS + 16, r1);
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
                if (p.o_tma && j + 1 < total && ld_acquire(&R.ready[k * RING + (j + 1) % RING]) >= j + 2) {
                    issue(j + 1, false);
                    issued_next = true;
                    KDA_TRACE_ANY(p, 17, j + 1);
                }
            }

            // (4) v_new = u - w S (TMEM lanes 64-127) -> fp16 [token][value] tile
            // (WY: Z = beta v - beta k e^G S, the same arithmetic)
            wait_all(R, bar_mma1, j & 1, p.status);
            tc_fence_after();
            KDA_TRACE_EV(p, 14, j);
            if (quad >= 2) {
                const int t = row - 64;
                uint32_t r0[16], r1[16];
                tmem_ld16(tD, r0);
                if constexpr (NCT > 16) tmem_ld16(tD + 16, r1);
                tmem_wait_ld();
                auto vnew = [&](const uint32_t (&r)[16], int cb) {
                    const int c8 = NCT * slice + 16 * cb;  // this CTA's column (u's is v0 + c8)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint4 uu = *reinterpret_cast<const uint4 *>(bb + SL_U + tile_chunk(64, t, v0 + c8 + 8 * hh));
                        const uint32_t *uw = reinterpret_cast<const uint32_t *>(&uu);
                        uint32_t vp[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 u2 = unpack_f16(uw[e]);
                            const float y0 = u2.x - __uint_as_float(r[8 * hh + 2 * e]);
                            const float y1 = u2.y - __uint_as_float(r[8 * hh + 2 * e + 1]);
                            vmax = max_abs_nan(max_abs_nan(vmax, y0), y1);
                            vp[e] = pack_f16(y0, y1);
                        }
                        *reinterpret_cast<uint4 *>(sVN + tile_chunk(64, t, c8 + 8 * hh)) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
                    }
                };
                vnew(r0, 0);
                if constexpr (NCT > 16) vnew(r1, 1);
            }
            fence_proxy_async_shared();
            tc_fence_before();
            sync_compute();
            if constexpr (WY) {
                // (4b) MMAT: V = [scale*Aqk ; T] Z; v_new = V (lanes 64-127) -> the v_new tile
                uint64_t *bar_t = reinterpret_cast<uint64_t *>(smem + OFF_BAR_T);
                if (tid == 0) {
                    tc_fence_after();
                    const uint32_t aq = smem_u32(bb + SL_AQK), vn = smem_u32(sVN);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f16(tmem + 256, umma_desc_sw128(aq + kk * 32, 16, 1024), umma_desc_sw128(vn + kk * 2048, 8192, 1024),
                                 idesc_av, kk > 0);
                    umma_commit(bar_t);
                }
                wait_all(R, bar_t, j & 1, p.status);
                tc_fence_after();
                if (quad >= 2) {
                    const int t = row - 64;
#pragma unroll
                    for (int cb = 0; cb < 2; ++cb) {  // 16 columns at a time
                        uint32_t r[16];
                        tmem_ld16(tS + 256 + 16 * cb, r);
                        tmem_wait_ld();
                        const int c8 = 32 * slice + 16 * cb;
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t vp[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float y0 = __uint_as_float(r[8 * hh + 2 * e]), y1 = __uint_as_float(r[8 * hh + 2 * e + 1]);
                                vmax = max_abs_nan(max_abs_nan(vmax, y0), y1);
                                vp[e] = pack_f16(y0, y1);
                            }
                            *reinterpret_cast<uint4 *>(sVN + tile_chunk(64, t, c8 + 8 * hh)) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
                        }
                    }
                }
                fence_proxy_async_shared();
                tc_fence_before();
                sync_compute();
            }
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
            // global, one full 512-byte row per warp store. With the fused gated
            // RMSNorm, warp w stores rows w, w+16, w+32, w+48: their gate values
            // (this lane's four channels) are loaded before the wait, so that
            // the loads land while MMA2/MMA3 run and o is staged.
            static_assert(NCOMP / 32 * 4 == BT, "four output rows per warp");
            uint2 gv[4];
            if (ngate) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int rr = warp + 16 * q4;
                    gv[q4] = rr < nv ? __ldg(reinterpret_cast<const uint2 *>(ngate + (static_cast<size_t>(t0 + rr) * p.H + h) * DV) + lane)
                                     : make_uint2(0u, 0u);
                }
            }
            wait_all(R, bar_mma23, j & 1, p.status);
            tc_fence_after();
            KDA_TRACE_EV(p, 16, j);
            if (p.o_tma && nv == BT) {
                // A full chunk of a plain o: staged in this chunk's slot buffer
                // (every operand in it is consumed) as four 128-byte-swizzled
                // [64][32] fp32 boxes, and written by four tensor stores that
                // run while the next chunk starts (the next copy into this
                // buffer waits for them to read it).
                // (box NCT*slice/32; this thread's first 16-byte chunk in its row: cb0)
                unsigned char *ob = smem + (b ? OFF_BUF1 : OFF_BUF0) + (NCT * slice / 32) * (BT * 128);
                if (quad < 2) {
                    const int cb0 = (NCT * slice % 32) / 4;
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tD, r0);
                    if constexpr (NCT > 16) tmem_ld16(tD + 16, r1);
                    tmem_wait_ld();
#pragma unroll
                    for (int c4 = 0; c4 < NCT / 4; ++c4) {
                        const uint32_t *r = c4 < 4 ? r0 + 4 * c4 : r1 + 4 * (c4 - 4);
                        *reinterpret_cast<uint4 *>(ob + row * 128 + (((cb0 + c4) ^ (row & 7)) << 4)) = make_uint4(r[0], r[1], r[2], r[3]);
                    }
                }
                fence_proxy_async_shared();
                tc_fence_before();
                sync_compute();
                if (tid == 0) {
                    const unsigned char *o0 = smem + (b ? OFF_BUF1 : OFF_BUF0);
#pragma unroll
                    for (int s4 = 0; s4 < NV / 32; ++s4) tma_store_3d(&p.tm_o, o0 + s4 * (BT * 128), v0 + 32 * s4, h, static_cast<int>(t0));
                    bulk_commit();
                }
                KDA_TRACE_EV(p, 12, j);
                if (tid == 0 && !issued_next && j + 1 < total) {
                    if (wait_flag_geq(R, &R.ready[k * RING + (j + 1) % RING], j + 2, p.status)) {
                        issue(j + 1, true);
                        KDA_TRACE_ANY(p, 18, j + 1);
                    } else
                        misc[0] = 0;
                }
                continue;
            }
            float *stg = reinterpret_cast<float *>(sS);  // [64][OST] fp32, spans the S16 and v_new tiles
            if (quad < 2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tD, r0);
                if constexpr (NCT > 16) tmem_ld16(tD + 16, r1);
                tmem_wait_ld();
                float *dst = stg + row * OST + NCT * slice;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    reinterpret_cast<float4 *>(dst)[e] = make_float4(__uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                                                                     __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3]));
                    if constexpr (NCT > 16)
                        reinterpret_cast<float4 *>(dst + 16)[e] = make_float4(__uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                                                                              __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3]));
                }
                if (!HALF && ngate) {  // this slice's sum of squares of the row, into the row's pad column 128 + slice
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float x0 = __uint_as_float(r0[e]), x1 = __uint_as_float(r1[e]);
                        ss = fmaf(x0, x0, ss);
                        ss = fmaf(x1, x1, ss);
                    }
                    stg[row * OST + DV + slice] = ss;
                }
            }
            tc_fence_before();
            sync_compute();
            if (!p.o) {
                // states only: no output rows
            } else if (!HALF && ngate) {
                // y = x / sqrt(mean(x^2) + eps) * weight * sigmoid(gate) over the row's 128 channels
                const float4 w4 = __ldg(reinterpret_cast<const float4 *>(p.nweight) + lane);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int rr = warp + 16 * q4;
                    if (rr < nv) {  // uniform in the warp
                        const float4 x = *reinterpret_cast<const float4 *>(stg + rr * OST + 4 * lane);
                        const float4 ps = *reinterpret_cast<const float4 *>(stg + rr * OST + DV);  // the four slices' sums
                        const float rs = rsqrtf(((ps.x + ps.y) + (ps.z + ps.w)) * (1.f / DV) + p.neps);
                        const float2 sa = unpack_f16(sigmoid_bf16x2_to_f16x2(gv[q4].x));
                        const float2 sb = unpack_f16(sigmoid_bf16x2_to_f16x2(gv[q4].y));
                        reinterpret_cast<float4 *>(p.o + (static_cast<size_t>(t0 + rr) * p.H + h) * DV)[lane] =
                            make_float4(x.x * rs * w4.x * sa.x, x.y * rs * w4.y * sa.y, x.z * rs * w4.z * sb.x,
                                        x.w * rs * w4.w * sb.y);
                    }
                }
            } else {
                for (int rr = warp; rr < nv; rr += NCOMP / 32)
                    if (NV == 128 || lane < NV / 4)
                        reinterpret_cast<float4 *>(p.o + (static_cast<size_t>(t0 + rr) * p.H + h) * DV + v0)[lane] =
                            *reinterpret_cast<const float4 *>(stg + rr * OST + 4 * lane);
            }
            KDA_TRACE_EV(p, 12, j);
            if (tid == 0 && !issued_next && j + 1 < total) {
                if (wait_flag_geq(R, &R.ready[k * RING + (j + 1) % RING], j + 2, p.status)) {
                    issue(j + 1, false);
                    KDA_TRACE_ANY(p, 18, j + 1);
                }
                else
                    misc[0] = 0;
            }
        }
        if (!alive) break;
        // final state: TMEM -> global
        if (p.sT && st_inb) {
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < NCT / 16; ++cb) {
                uint32_t r[16];
                tmem_ld16(tS + 16 * cb, r);
                tmem_wait_ld();
                float4 *dst = reinterpret_cast<float4 *>(p.sT + state_base + row * DV + v0 + NCT * slice + 16 * cb);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                         __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
            }
        }
    }
    if (!(vmax < F16_SAFE)) set_status(p.status, KDA_ERR_VALUE_RANGE);
    if (tid == 0) bulk_wait_all();  // the last o stores
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, WY ? 2 * TMEM_COLS : TMEM_COLS);
}
}  // namespace cons

static_assert(prod::SMEM <= OFF_SCHED && cons::SMEM <= OFF_SCHED, "the chain schedule lies past both roles' tiles");
constexpr int SMEM_TILES = OFF_SCHED + SCHED_BYTES + 1024;  // + alignment slack
static_assert(8192 + 8 * SCHED_MAX_CHAINS + 8 * SCHED_MAX_C <= OFF_SCHED, "schedule scratch fits below the schedule");
#ifdef KDA_TRACE
static_assert(SMEM_TILES <= TRACE_COUNTS_OFFSET, "trace counters past the tiles");
constexpr int SMEM_MAX = TRACE_COUNTS_OFFSET + 64;
#else
constexpr int SMEM_MAX = SMEM_TILES;
#endif
static_assert(SMEM_MAX <= 232448, "shared memory budget");

template <bool WY, bool HALF>  // the consumers form the WY product; consumers are CTA pairs
__global__ void __launch_bounds__(NTHREADS, 1) kda_persistent_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
#ifdef KDA_TRACE
    if (threadIdx.x < 16) reinterpret_cast<int *>(smem_raw + TRACE_COUNTS_OFFSET)[threadIdx.x] = 0;
    __syncthreads();
#endif
    build_sched(p, smem + OFF_SCHED, smem);  // the roles' tiles serve as scratch until it returns
    // consumer CTAs first: with HALF, CTA k and k + C are the two column halves of consumer k
    const int ncons = HALF ? 2 * p.C : p.C;
    if (static_cast<int>(blockIdx.x) < ncons)
        cons::run<WY, HALF>(p, smem, HALF ? static_cast<int>(blockIdx.x) % p.C : static_cast<int>(blockIdx.x),
                            HALF ? static_cast<int>(blockIdx.x) / p.C : 0);
    else
        prod::run<WY, HALF>(p, smem, blockIdx.x - ncons);
}

// ------------------------------------------------------------------ host side
// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the driver library)
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn encode_tiled() {
    static const EncodeTiledFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}
// map of o as [tokens][heads][128] fp32 with a box of 32 channels x 1 head x
// 64 tokens and the 128-byte swizzle; false when the encoder is unavailable
static bool encode_o(CUtensorMap *m, float *o, int64_t tokens, int heads) {
    const EncodeTiledFn fn = encode_tiled();
    if (!fn || tokens < 1) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(DV), static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(DV) * 4, static_cast<cuuint64_t>(DV) * 4 * heads};
    const cuuint32_t box[3] = {32u, 1u, static_cast<cuuint32_t>(BT)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// Most consumer CTAs a launch uses (half the SMs, at most one per chain): the
// workspace is sized for this many rings.
int max_consumers(int64_t chains, int grid) {
    int64_t c = grid / 2;
    if (c < 1) c = 1;
    if (chains < c) c = chains;
    return static_cast<int>(c < 1 ? 1 : c);
}

// Consumer CTAs for one launch, from a cost model of the two roles: a consumer
// that is kept busy completes about one chunk per 3.5 us (2.45 us of its own
// work; the rest is the ring's hand-off latency with four slots), a producer
// about one chunk per 7.0 us, and the launch takes the longer of
//   (chains per consumer) x (chunks per chain) x 3.5 us   and
//   (all chunks) x 7.0 us / (producer CTAs).
// Candidates give every consumer the same number of chains (C = ceil(chains / m)).
// `tokens` sizes the chunk count (each sequence adds at most one partial chunk).
int consumers_for(int64_t chains, int64_t tokens, int64_t seqs, int grid) {
    const int cmax = max_consumers(chains, grid);
    if (chains < 1 || grid < 2) return cmax;
    constexpr double T_CONS = 3.5, T_PROD = 7.0;  // us per chunk, measured on GB300
    const double chunks = static_cast<double>(chains / (seqs > 0 ? seqs : 1)) *
                          (static_cast<double>(tokens) / BT + 0.5 * static_cast<double>(seqs));
    const double per_chain = chunks / static_cast<double>(chains);
    int best = cmax;
    double best_cost = 1e300;
    for (int64_t m = 1;; ++m) {
        const int64_t c = (chains + m - 1) / m;
        if (c <= cmax && c < grid) {
            const double cons = static_cast<double>((chains + c - 1) / c) * per_chain * T_CONS;
            const double prod = chunks * T_PROD / static_cast<double>(grid - c);
            const double cost = cons > prod ? cons : prod;
            if (cost < best_cost) {
                best_cost = cost;
                best = static_cast<int>(c);
            }
        }
        if (c <= 1) break;
    }
    return best;
}

// Whether the consumers form the WY product X = T [beta v | beta k e^G]. Only
// a batch whose sequences can all have one length (tokens divisible by seqs)
// qualifies, judged with that length by the same kind of estimate: a producer
// task takes about 6.8 us (6.5 when the consumers do the WY product) and a
// consumer chunk about 2.5 us (3.05), and the launch about the longer of
// (busiest consumer's chunks) x (chunk time) and (all chunks) x (task time) /
// (producer CTAs); the consumers' time is counted 1.25 times so that they keep
// slack. (A batch of unequal lengths that still passes runs correctly, only
// perhaps slower.)
bool wy_for(int64_t chains, int64_t tokens, int64_t seqs, int C, int grid) {
    if (seqs < 1 || tokens < 1 || tokens % seqs != 0 || C < 1 || C >= grid) return false;
    const double per_chain = static_cast<double>((tokens / seqs + BT - 1) / BT);
    const double busiest = static_cast<double>((chains + C - 1) / C) * per_chain;
    const double per_prod = static_cast<double>(chains) * per_chain / static_cast<double>(grid - C);
    const double t_prod = std::fmax(2.5 * busiest, 6.8 * per_prod);
    const double t_cons = std::fmax(1.25 * 3.05 * busiest, 6.5 * per_prod);
    return t_cons < t_prod;
}

// Whether each chain's 128 value columns go to a pair of consumer CTAs, one
// column half each (the consumer's MMAs, epilogues and state then halve; both
// CTAs copy the whole slot). Only where every chain can have a pair within half
// the SMs, by the estimate of consumers_for with a split consumer chunk at
// about 2.6 us against 3.5, and the producers short of the second CTAs.
bool split_for(int64_t chains, int64_t tokens, int64_t seqs, int C, int grid) {
    if (chains < 1 || seqs < 1 || C < 1 || C >= grid || 2 * chains > grid / 2) return false;
    constexpr double T_CONS = 3.5, T_SPLIT = 2.6, T_PROD = 7.0;
    const double chunks = static_cast<double>(chains / seqs) *
                          (static_cast<double>(tokens) / BT + 0.5 * static_cast<double>(seqs));
    const double per_chain = chunks / static_cast<double>(chains);
    const double whole = std::fmax(static_cast<double>((chains + C - 1) / C) * per_chain * T_CONS,
                                   chunks * T_PROD / static_cast<double>(grid - C));
    const double split = std::fmax(per_chain * T_SPLIT, chunks * T_PROD / static_cast<double>(grid - 2 * chains));
    return split < whole;
}

size_t workspace_bytes(int64_t chains) {
    const int sms = num_sms();
    if (sms < 2 || chains < 1) return 0;
    const int C = max_consumers(chains, sms);
    size_t bytes = ring_offset(C) + static_cast<size_t>(C) * RING * SLOT_BYTES;
#ifdef KDA_TRACE
    bytes += static_cast<size_t>(sms) * TRACE_CTA_WORDS * 8;
#endif
    return bytes;
}

cudaError_t launch(Params p, size_t ws_bytes, cudaStream_t stream) {
    const int sms = num_sms();
    if (sms < 2) return cudaErrorInvalidDevice;
    const int grid = sms;  // one CTA per SM; all co-resident (cooperative launch)
    const int64_t chains = static_cast<int64_t>(p.N) * p.H;
    p.C = consumers_for(chains, p.T, p.N, grid);
    p.CH = 1;
    p.Cws = max_consumers(chains, grid);
    p.spin = (p.debug & KDA_DEBUG_WITHHOLD_READY) ? SPIN_LIMIT_DEBUG : SPIN_LIMIT;
    if (ws_bytes < ring_offset(p.Cws) + static_cast<size_t>(p.Cws) * RING * SLOT_BYTES) return cudaErrorInvalidValue;
    // a plain o in device memory leaves full chunks by tensor stores (else, and
    // for partial chunks, by the warps: an o in mapped host memory, for one)
    bool o_device = false;
    if (p.o) {
        cudaPointerAttributes at{};
        o_device = cudaPointerGetAttributes(&at, p.o) == cudaSuccess && at.type == cudaMemoryTypeDevice;
        (void)cudaGetLastError();  // clear a failed query
    }
    p.o_tma = (o_device && !p.ngate && encode_o(&p.tm_o, p.o, p.Ttok, p.H)) ? 1 : 0;
    // a chain's columns split over two consumer CTAs (not with the gated norm,
    // which needs whole rows of o, nor with the consumers' WY form)
    bool split = !p.ngate && split_for(chains, p.T, p.N, p.C, grid);
    if (p.debug & KDA_DEBUG_SPLIT_COLUMNS) split = !p.ngate && 2 * chains <= grid / 2;
    if (p.debug & (KDA_DEBUG_WHOLE_COLUMNS | KDA_DEBUG_WY_CONSUMER)) split = false;
    if (split) {
        p.C = static_cast<int32_t>(chains);
        p.CH = 2;
    }
    // the consumers take the WY product only with o on tensor stores (the
    // warps' own o stores, and the gated norm, leave them no slack for it)
    bool wy = !split && p.o_tma && wy_for(chains, p.T, p.N, p.C, grid);
    if (p.debug & KDA_DEBUG_WY_PRODUCER) wy = false;
    if (p.debug & KDA_DEBUG_WY_CONSUMER) wy = true;
    const void *kernel = split ? reinterpret_cast<const void *>(kda_persistent_kernel<false, true>)
                         : wy  ? reinterpret_cast<const void *>(kda_persistent_kernel<true, false>)
                               : reinterpret_cast<const void *>(kda_persistent_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, NTHREADS, SMEM_MAX);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    e = cudaMemsetAsync(p.ws, 0, ring_offset(p.C), stream);
    if (e != cudaSuccess) return e;
#ifdef KDA_TRACE
    e = cudaMemsetAsync(p.ws + ring_offset(p.Cws) + static_cast<size_t>(p.Cws) * RING * SLOT_BYTES, 0,
                        static_cast<size_t>(grid) * TRACE_CTA_WORDS * 8, stream);
    if (e != cudaSuccess) return e;
#endif
    void *args[] = {&p};
    return cudaLaunchCooperativeKernel(kernel, dim3(grid), dim3(NTHREADS), args, SMEM_MAX, stream);
}

}  // namespace pers
}  // namespace kda
