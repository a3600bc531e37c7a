// KDA chunked prefill forward — persistent cooperative kernel, one CTA per SM,
// in two roles that hand chunks to each other through a small ring in L2.
//
//   producers  run the intra-chunk steps of "在 TPU 上加速 Kimi K3 KDA" (junyi.dev
//              tpu-kda report) for (chain, chunk) tasks: step 1 gate prefix sum
//              (§6.1), step 2 Aqk/Akk as products of sub-block-midpoint-rescaled
//              operands (§4), step 3 T = (I+L)^-1 by 16x16 blocks, step 4 the WY
//              form [u | w] = T [beta v | beta k e^G] on the 5th-generation tensor
//              cores, plus q_hat = scale q e^G and kg = k e^(G_last - G) (§4,
//              §6.3). One thread owns one key channel of one 16-token sub-block,
//              so the prefix sum runs in registers and every per-channel product
//              leaves as a contiguous row of the ring slot, in the layouts the
//              consumer's tensor-core operands use; then the slot's ready flag is
//              released.
//   consumers  own (sequence, head) chains and run step 5 chunk after chunk
//              (§6.2) on the transposed state S^T (tensor-memory lane = value
//              column): D^T = S^T [q_hat; w]^T, v_new^T = u^T - (w S)^T,
//              S^T <- S^T Diag(d) and [S^T | o^T] += v_new^T [kg | Aqk^T] in one
//              product, reading the entry state; both per-chunk A operands stay in
//              tensor memory, and each o row leaves as coalesced stores.
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
constexpr long long SPIN_LIMIT = 1ll << 24;         // polls before a wait gives up (normal calls)
constexpr long long SPIN_LIMIT_DEBUG = 1ll << 14;   // the same under any KDA_DEBUG_* flag
#ifdef KDA_TRACE
constexpr int TRACE_COUNTS_OFFSET = 231424;  // past every role's tiles (checked below), 16 ints
#endif

// ---------------------------------------------------------------- slot layout
// A slot holds one (chain, chunk) hand-off in the shared-memory layouts of the
// consumer's tensor-core operands; every region is 1024-byte aligned.
//   B1   [q_hat ; w]^T  fp16 [key][token], MN-major: atom column 0 holds the
//                       64 tokens of q_hat, atom column 1 those of w (32 KB)
//   B23  [kg^T ; Aqk]   fp16, K-major rows of 64 tokens: rows 0-127 are key
//                       channels (kg^T[c][s]), rows 128-191 tokens t
//                       (scale * Aqk[t][s], zero above the diagonal) (24 KB)
//   U    u^T            fp16 [value][token] (16 KB)
//   D    e^(G_last)     fp32 [128]
// 128-byte swizzle: row r of a 128-byte-wide atom column keeps its 16-byte
// chunk c at position c ^ (r mod 8); wider tiles are split into 64-element
// atom columns stored one after the other.
constexpr int SL_B1 = 0, SL_B23 = 32768, SL_U = 57344, SL_D = 73728;
static_assert(SLOT_BYTES == 74752 && SL_D + 512 <= SLOT_BYTES, "slot size");

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
    unsigned char *slots;
    long long spin;  // polls before a wait gives up
};

__device__ __forceinline__ Ring ring_of(const Params &p) {
    Ring r;
    r.hdr = reinterpret_cast<Header *>(p.ws);
    r.ready = reinterpret_cast<int *>(p.ws + sizeof(Header));
    r.freed = r.ready + p.C * RING;
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
constexpr int OFF_SCHED = 197632;  // past both roles' tiles (checked below)
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

// completion of this CTA's own tensor-core products: depends on no other CTA,
// so only a (bounded) timeout ends it early, never the abort word
__device__ __forceinline__ bool wait_local(const Ring &R, uint64_t *bar, uint32_t parity, int32_t *status) {
    for (long long it = 0; it < SPIN_LIMIT; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    set_status(status, KDA_ERR_TIMEOUT);
    atomicExch(&R.hdr->abort, 1);
    return false;
}

// ================================================================== producer
// Steps 1-4 for one (chain, chunk) task at a time on all sixteen warps. Warp w
// owns key channels 32 (w % 4) .. 32 (w % 4) + 31 (its tensor-memory lane
// quarter) of sub-block w / 4, one channel per thread, for the prefix sum, the
// elementwise products, the tensor-memory operand R^T and the read-out of the
// WY product. The strips run on warp-level tensor-core products (m16n8k8 tf32,
// m16n8k16 bf16) over the ten lower 16x16 tiles, the WY product on tcgen05
// with its A operand in tensor memory. The WY product of a task is read out
// during the next task (after its elementwise step), and the task's slot is
// published right then, before the producer waits for anything else.
// Round an fp32 value to tf32 (nearest, ties away from zero) for a tf32 MMA
// operand: adding half a tf32 unit in the last place to the sign-magnitude bit
// pattern carries into bit 13 exactly when the dropped 13 bits are at least
// half of it, and the MMA reads only the upper 19 bits. Finite inputs only.
__device__ __forceinline__ uint32_t tf32_rna(float x) { return __float_as_uint(x) + 0x1000u; }

namespace prod {
constexpr int RSF = 136, RSA = 72;
constexpr int SZ_T = BT * DK * 2;                   // 16384: one [64][128] 16-bit tile
constexpr int OFF_Q = 0, OFF_K = SZ_T, OFF_V = 2 * SZ_T;  // q, k, v (bf16, tile layout)
constexpr int OFF_G = 3 * SZ_T;                     // g (fp32, g_chunk layout, 32 KB)
constexpr int OFF_QA = OFF_G + 2 * SZ_T;            // q e^(G - G_m) as tf32 (fp32 words, qa_pair layout, 32 KB)
constexpr int OFF_KA = OFF_QA + 2 * SZ_T;           // k e^(G - G_m) (bf16, tile layout)
constexpr int OFF_KB = OFF_KA + SZ_T;               // k e^(G_m - G) (fp32 [64][RSF])
constexpr int OFF_L = OFF_KB + BT * RSF * 4;        // L = diag(beta) tril(Akk, -1) (fp16 [64][RSA])
constexpr int OFF_LD = OFF_L + BT * RSA * 2;        // diagonal blocks of L (fp32 [4][16][17])
constexpr int OFF_T = (OFF_LD + 4352 + 1023) / 1024 * 1024;  // T = (I+L)^-1 (fp16 [t][s], tile layout, 64 rows)
constexpr int OFF_GM = OFF_T + 8192;                // G at the sub-block midpoints (fp32 [4][128])
constexpr int OFF_TOT = OFF_GM + 2048;              // per-sub-block sums of g, base 2 (fp32 [4][128])
constexpr int OFF_F = OFF_TOT + 2048;               // 2^(G_mi - G_mj) for j < i (fp32 [6][128])
constexpr int OFF_BETA = OFF_F + 3072;              // beta, two buffers of 64 fp32
constexpr int OFF_MISC = OFF_BETA + 512;            // flags and the task broadcast (32 ints)
constexpr int OFF_GPAR = OFF_MISC + 128;            // raw gates: the task head's dt_bias row (128 fp32) and A_log
constexpr int OFF_BAR = OFF_GPAR + 528;             // WY-product mbarrier, then the TMEM base address
constexpr int SMEM = OFF_BAR + 16;
static_assert(OFF_GPAR % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
static_assert(OFF_Q % 1024 == 0 && OFF_G % 1024 == 0 && OFF_KA % 1024 == 0 && OFF_T % 1024 == 0,
              "swizzled tiles are 1024-byte aligned");
// Tensor memory: R^T = [beta v | beta k e^G]^T (fp16, lane = channel, column c
// = tokens 2c and 2c + 1) in two buffers at +32 columns, and the WY product
// X^T = [u | w]^T (fp32, lane = channel, column = token).
constexpr uint32_t TM_RV = 0, TM_RK = 64, TM_XU = 128, TM_XW = 192, TM_COLS = 256;
// Warp w runs on sub-partition w % 4. During the strips, warps 0-9 hold the
// ten tiles (three on partitions 0 and 1, two on 2 and 3); the diagonal
// inverses run on warps 10, 11, 14, 15 (partitions 2 and 3) and the zero tiles
// of Aqk on warps 12 and 13 (partitions 0 and 1).
constexpr int SYNC_TID = 9 * 32;              // lane 0 of warp 9: draws tasks
constexpr int REL_TID = 12 * 32;              // lane 0 of warp 12: publishes slots, waits for free slots
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

// 32 bytes of row r of a 128-byte-swizzled tile with `rows` rows per atom
// column: the 16 16-bit elements at columns c16 .. c16 + 15 (c16 a multiple of
// 16). Their two 16-byte chunks are adjacent in memory (in swapped order when
// the row's swizzle is odd), so one 32-byte store writes a whole sector.
__device__ __forceinline__ void st_row32(unsigned char *tile, int rows, int r, int c16, const uint32_t (&v)[8]) {
    const int a = (c16 & 63) >> 3, sw = r & 7;
    unsigned char *q = tile + (c16 >> 6) * rows * 128 + r * 128 + (((a ^ sw) & ~1) << 4);
    if (sw & 1)
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(q), "r"(v[4]), "r"(v[5]), "r"(v[6]),
                     "r"(v[7]), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3])
                     : "memory");
    else
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(q), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                     "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                     : "memory");
}

__device__ __forceinline__ unsigned char *slot_of(const Ring &R, const Task &t) {
    return R.slots + static_cast<size_t>(t.k * RING + t.j % RING) * SLOT_BYTES;
}

// One task's inputs into shared memory, issued by the `n` threads first ..
// first + n - 1 once the input tiles are free: 16-byte cp.async copies into
// the 128-byte-swizzled tile layouts, g (fp32) in a first commit group, q, k, v
// (bf16) and beta (into buffer bb) in a second, so the prefix sum can start
// before q, k and v land (every thread waits for its own groups, then the CTA
// meets at a barrier). Rows past the sequence end are zero-filled (g = 0 keeps
// row 63 of G at the last valid prefix; k = v = beta = 0 rows are inert in
// every product).
__device__ __forceinline__ void issue_loads(const Params &p, unsigned char *smem, const Task &tk, int bb, int first, int n) {
    const int li = static_cast<int>(threadIdx.x) - first;
    const size_t rs = static_cast<size_t>(p.H) * DK;  // token stride, elements
    const size_t hb = static_cast<size_t>(tk.h) * DK;
    for (int idx = li; idx < BT * 32; idx += n) {  // g: 64 rows x 32 chunks of 4 channels
        const int r = idx >> 5, c4 = (idx & 31) << 2;
        const bool ok = r < tk.nv;
        cp_async16(smem + OFF_G + g_chunk(r, c4), p.g + static_cast<size_t>(tk.t0 + (ok ? r : 0)) * rs + hb + c4,
                   ok ? 16 : 0);
    }
    if (p.raw && li < 33) {  // the gate activation's per-head parameters (zeros when not given)
        if (li < 32)
            cp_async16(smem + OFF_GPAR + 16 * li, p.dt_bias ? p.dt_bias + hb + 4 * li : p.g, p.dt_bias ? 16 : 0);
        else
            cp_async4(smem + OFF_GPAR + 512, p.A_log ? p.A_log + tk.h : p.g, p.A_log ? 4 : 0);
    }
    cp_async_commit();
    for (int idx = li; idx < BT * 16; idx += n) {  // q, k, v: 64 rows x 16 chunks of 8 channels
        const int r = idx >> 4, c8 = (idx & 15) << 3;
        const bool ok = r < tk.nv;
        const size_t off = static_cast<size_t>(tk.t0 + (ok ? r : 0)) * rs + hb + c8;
        const int d = tile_chunk(64, r, c8);
        cp_async16(smem + OFF_Q + d, p.q + off, ok ? 16 : 0);
        cp_async16(smem + OFF_K + d, p.k + off, ok ? 16 : 0);
        cp_async16(smem + OFF_V + d, p.v + off, ok ? 16 : 0);
    }
    if (li >= n - BT) {  // the last 64 threads: beta
        const int r = li - (n - BT);
        const bool ok = r < tk.nv;
        cp_async4(smem + OFF_BETA + 256 * bb + 4 * r, p.beta + static_cast<size_t>(tk.t0 + (ok ? r : 0)) * p.H + tk.h,
                  ok ? 4 : 0);
    }
    cp_async_commit();
}

// The previous task's WY product X^T = [u | w]^T, read out of tensor memory
// into the previous task's slot: u^T rows into U, w^T rows into atom column 1
// of B1 (this thread: channel `chn`, tokens 16 b .. 16 b + 15 for b in [b0, b1)).
__device__ __forceinline__ void read_out_x(uint32_t tl, unsigned char *pd, int chn, int b0, int b1, float &vmax) {
    for (int b = b0; b < b1; ++b) {
        uint32_t xu[16], xw[16];
        tmem_ld16(tl + TM_XU + 16 * b, xu);
        tmem_ld16(tl + TM_XW + 16 * b, xw);
        tmem_wait_ld();
        uint32_t u2[8], w2[8];
        float vm = vmax;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float a0 = __uint_as_float(xu[2 * e]), a1 = __uint_as_float(xu[2 * e + 1]);
            const float c0 = __uint_as_float(xw[2 * e]), c1 = __uint_as_float(xw[2 * e + 1]);
            vm = max_abs_nan(max_abs_nan(vm, a0), a1);
            vm = max_abs_nan(max_abs_nan(vm, c0), c1);
            u2[e] = pack_f16(a0, a1);
            w2[e] = pack_f16(c0, c1);
        }
        vmax = vm;
        st_row32(pd + SL_U, 128, chn, 16 * b, u2);
        st_row32(pd + SL_B1, 128, chn, 64 + 16 * b, w2);
    }
}

// a slot's ready flag, released once the slot's contents have been written
// (all of them ordered before this thread by a preceding barrier)
__device__ __forceinline__ void publish(const Params &p, const Ring &R, const Task &t) {
    fence_acq_rel_gpu();
    if (!(p.debug & KDA_DEBUG_WITHHOLD_READY)) st_release(&R.ready[t.k * RING + t.j % RING], t.j + 1);
}
// whether task t's slot is free (its consumer has copied out the chunk that
// used it RING chunks earlier), polling at most `polls` times
__device__ __forceinline__ bool slot_free(const Ring &R, const Task &t, long long polls) {
    if (t.j < RING) return true;
    const int *f = &R.freed[t.k * RING + t.j % RING];
    for (long long it = 0; it < polls; ++it) {
        if (ld_acquire(f) >= t.j - RING + 1) return true;
        __nanosleep(64);
    }
    return false;
}

// Step 2b for one group of strip tiles on one warp: row blocks R0 and R0 + 1
// against column blocks C0 .. C0 + NC - 1 (the tiles (i, j) with j <= i among
// them), so that each 16-channel step loads the A fragments of a row block and
// the B values of a column block once for all the group's tiles. Aqk on tf32
// (m16n8k8), Akk on bf16 (m16n8k16). Within each 16-channel step the tf32 k
// slots are permuted (slot q <-> channel 2q, slot q+4 <-> channel 2q+1, for each
// half) so that one 8-byte load of a k e^(G_m - G) row feeds both the tf32 and
// the bf16 B fragments. Tile (i, j) needs k_s e^(G_{m_i} - G_s) for s in
// sub-block j: the stored k e^(G_{m_j} - G) times e^(G_{m_i} - G_{m_j}) (<= 1).
// Writes scale*Aqk into the slot and L = diag(beta) tril(Akk, -1) (and its
// diagonal blocks in fp32) into shared memory.
template <int R0, int C0, int NC>
__device__ __forceinline__ void strip_group(const unsigned char *smem, unsigned char *dst, const float *sBeta, float scale,
                                            int lane) {
    const int gq = lane >> 2, qd = lane & 3;
    const float *sKB = reinterpret_cast<const float *>(smem + OFF_KB);
    const float *sF = reinterpret_cast<const float *>(smem + OFF_F);
    __half *sL = reinterpret_cast<__half *>(const_cast<unsigned char *>(smem) + OFF_L);
    float *sLD = reinterpret_cast<float *>(const_cast<unsigned char *>(smem) + OFF_LD);
    float aq[2][NC][2][4], ak[2][NC][2][4];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri)
#pragma unroll
        for (int cj = 0; cj < NC; ++cj)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) aq[ri][cj][nt][e] = ak[ri][cj][nt][e] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < 8; ++kk) {
        const int c0 = 16 * kk + 2 * qd;
        uint32_t fa0[2][4], fa1[2][4], fk[2][4];
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            const int i = R0 + ri;
            const unsigned char *sQA = smem + OFF_QA;
            const uint2 u00 = *reinterpret_cast<const uint2 *>(sQA + qa_pair(16 * i + gq, c0));
            const uint2 u10 = *reinterpret_cast<const uint2 *>(sQA + qa_pair(16 * i + gq + 8, c0));
            const uint2 u01 = *reinterpret_cast<const uint2 *>(sQA + qa_pair(16 * i + gq, c0 + 8));
            const uint2 u11 = *reinterpret_cast<const uint2 *>(sQA + qa_pair(16 * i + gq + 8, c0 + 8));
            fa0[ri][0] = u00.x; fa0[ri][1] = u10.x; fa0[ri][2] = u00.y; fa0[ri][3] = u10.y;
            fa1[ri][0] = u01.x; fa1[ri][1] = u11.x; fa1[ri][2] = u01.y; fa1[ri][3] = u11.y;
            ldsm_x4(fk[ri], smem + OFF_KA + a_addr(lane, 64, 16 * i, 16 * kk));
        }
        float2 x0[NC][2], x1[NC][2];
#pragma unroll
        for (int cj = 0; cj < NC; ++cj)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float *row = sKB + (16 * (C0 + cj) + 8 * nt + gq) * RSF;
                x0[cj][nt] = *reinterpret_cast<const float2 *>(row + c0);
                x1[cj][nt] = *reinterpret_cast<const float2 *>(row + c0 + 8);
            }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri)
#pragma unroll
            for (int cj = 0; cj < NC; ++cj) {
                const int i = R0 + ri, j = C0 + cj;
                if (j > i) continue;
                float2 f0 = make_float2(1.f, 1.f), f1 = make_float2(1.f, 1.f);
                if (i > j) {
                    const float *fr = sF + f_pair(i, j) * 128;
                    f0 = *reinterpret_cast<const float2 *>(fr + c0);
                    f1 = *reinterpret_cast<const float2 *>(fr + c0 + 8);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float b00 = x0[cj][nt].x * f0.x, b01 = x0[cj][nt].y * f0.y;
                    const float b10 = x1[cj][nt].x * f1.x, b11 = x1[cj][nt].y * f1.y;
                    mma1688_tf32(aq[ri][cj][nt], fa0[ri], tf32_rna(b00), tf32_rna(b01));
                    mma1688_tf32(aq[ri][cj][nt], fa1[ri], tf32_rna(b10), tf32_rna(b11));
                    mma16816(ak[ri][cj][nt], fk[ri], pack_bf16(b00, b01), pack_bf16(b10, b11));
                }
            }
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri)
#pragma unroll
        for (int cj = 0; cj < NC; ++cj) {
            const int i = R0 + ri, j = C0 + cj;
            if (j > i) continue;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int tl16 = gq + 8 * hf, sl = 8 * nt + 2 * qd;
                    const int t = 16 * i + tl16, sc = 16 * j + sl;
                    const float btt = sBeta[t];
                    float vq[2], vk[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const bool incl = (i > j) || (sl + e <= tl16);
                        const bool strict = (i > j) || (sl + e < tl16);
                        vq[e] = incl ? scale * aq[ri][cj][nt][2 * hf + e] : 0.f;
                        vk[e] = strict ? btt * ak[ri][cj][nt][2 * hf + e] : 0.f;
                        if (i == j) sLD[(i * 16 + tl16) * 17 + sl + e] = vk[e];
                    }
                    *reinterpret_cast<uint32_t *>(dst + SL_B23 + tile_elem(192, 128 + t, sc)) = pack_f16(vq[0], vq[1]);
                    *reinterpret_cast<uint32_t *>(sL + t * RSA + sc) = pack_f16(vk[0], vk[1]);
                }
        }
}

__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int pid) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, blk = warp >> 2;  // channel group (tensor-memory lane quarter), sub-block
    const int chn = 32 * quad + lane;            // this thread's key channel
    const int gq = lane >> 2, qd = lane & 3;
    const float scale = p.scale;
    Ring R = ring_of(p);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);
    uint64_t *bar_x = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 8);
    float *sTot = reinterpret_cast<float *>(smem + OFF_TOT);
    float *sGm = reinterpret_cast<float *>(smem + OFF_GM);
    float *sF = reinterpret_cast<float *>(smem + OFF_F);
    float *sKB = reinterpret_cast<float *>(smem + OFF_KB);
    __half *sL = reinterpret_cast<__half *>(smem + OFF_L);
    float *sLD = reinterpret_cast<float *>(smem + OFF_LD);
    unsigned char *sT = smem + OFF_T;
    const int32_t *cu_s = sched_cu(p, smem);  // sequence bounds (in shared memory when small enough)

    // the upper blocks of T are never written: zero the tile once
    for (int i = tid; i < 8192 / 16; i += NCOMP) reinterpret_cast<uint4 *>(sT)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        misc[1] = 0;
        mbar_init(bar_x, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(tslot, TM_COLS);
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);  // this warp's lane quarter
    {  // longest consumer sequence: tasks beyond it do not exist
        int mx = 0;
        for (int k = tid; k < p.C; k += NCOMP) mx = max(mx, consumer_total(p, smem, cu_s, k));
        atomicMax(&misc[1], mx);
    }
    sync_compute();
    const int jmax = misc[1];
    Cursor cs = make_cursor(pid, static_cast<int>(gridDim.x) - p.C, p.C);  // used by SYNC_TID
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
    if (cur.valid) issue_loads(p, smem, cur, 0, 0, NCOMP);
    if (tid == REL_TID) misc[21] = cur.valid && slot_free(R, cur, R.spin) ? 1 : 0;  // nothing is unpublished yet
    const uint32_t idesc_x = umma_idesc_f16(false, false, 128, 64);  // R^T (tensor memory) x T^T (K-major)
    bool gate_bad = false;
    float vmax = 0.f;         // largest magnitude sent to an fp16 operand (NaN if any was NaN)
    Task prev{0, 0, 0, 0, 0, 0, 0, 0};
    bool x_pending = false;   // prev's WY product is in flight
    int it = 0;
    while (cur.valid) {
        const int bb = it & 1;  // beta and R^T buffers of this task
        const float *sBeta = reinterpret_cast<const float *>(smem + OFF_BETA + 256 * bb);
        KDA_TRACE_EV(p, 1, cur.j * p.C + cur.k);
        cp_async_wait_group1();  // g (q, k, v and beta may still be in flight)
        sync_compute();
        // ---- step 1: inclusive prefix sum of g (base 2) over the sub-block's 16
        // tokens in registers, then the sub-block carries through shared memory
        float G[16];
        {
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = *reinterpret_cast<const float *>(smem + OFF_G + g_elem(16 * blk + r, chn));
            if (p.raw) {  // g = lower_bound * sigmoid(e^A_log (g_raw + dt_bias)); rows past the sequence end stay 0
                const float *gp = reinterpret_cast<const float *>(smem + OFF_GPAR);
                const float a = __expf(gp[128]), db = gp[chn];
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    x[r] = (16 * blk + r < cur.nv) ? __fdividef(p.lb, 1.f + __expf(-a * (x[r] + db))) : 0.f;
            }
            float acc = 0.f;
            bool gb = false;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                gb |= !(x[r] >= p.lb && x[r] <= 0.f);
                acc += x[r] * LOG2E;
                G[r] = acc;
            }
            gate_bad |= gb;
            sTot[blk * 128 + chn] = acc;
        }
        cp_async_wait_all();  // q, k, v and beta
        sync_compute();
        if (p.raw && tid < BT) {  // beta = sigmoid(beta_raw); rows past the sequence end stay 0
            float *bw = reinterpret_cast<float *>(smem + OFF_BETA + 256 * bb);
            bw[tid] = tid < cur.nv ? __fdividef(1.f, 1.f + __expf(-bw[tid])) : 0.f;
        }
        float Gl = 0.f;
        {
            float carry = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float t = sTot[q * 128 + chn];
                if (q < blk) carry += t;
                Gl += t;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) G[r] += carry;
        }
        const float Gm = G[7];  // the sub-block midpoint (rows past the end carry the last valid prefix)
        sGm[blk * 128 + chn] = Gm;
        sync_compute();
        for (int j = 0; j < blk; ++j) sF[f_pair(blk, j) * 128 + chn] = ex2(Gm - sGm[j * 128 + chn]);
        KDA_TRACE_EV(p, 20, 0);

        // ---- steps 2a/4a: elementwise products of the thread's 16 tokens:
        // strip operands into shared memory, R^T into tensor memory, q_hat and
        // kg into registers (they go to the slot once it is known to be free)
        uint32_t qh[8], kgp[8];
        {
            const float EM = ex2(Gm), EMs = scale * EM, EL = ex2(Gl - Gm);
            float bt[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 b4 = reinterpret_cast<const float4 *>(sBeta)[4 * blk + q];
                bt[4 * q] = b4.x; bt[4 * q + 1] = b4.y; bt[4 * q + 2] = b4.z; bt[4 * q + 3] = b4.w;
            }
            uint32_t rv[8], rk[8];
            float vm = 0.f;
#pragma unroll
            for (int r2 = 0; r2 < 8; ++r2) {
                float oq[2], ok[2], ov[2], orr[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r = 2 * r2 + e, t = 16 * blk + r;
                    const int te = tile_elem(64, t, chn);
                    const float qf = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_Q + te));
                    const float kf = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_K + te));
                    const float vf = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(smem + OFF_V + te));
                    const float x = G[r] - Gm;
                    const float a = ex2(x), b = ex2(-x);
                    const float qa = qf * a, ka = kf * a, kb = kf * b;
                    *reinterpret_cast<uint32_t *>(smem + OFF_QA + qa_pair(t, chn) + 4 * (chn & 1)) = tf32_rna(qa);
                    *reinterpret_cast<__nv_bfloat16 *>(smem + OFF_KA + te) = __float2bfloat16_rn(ka);
                    sKB[t * RSF + chn] = kb;
                    oq[e] = qa * EMs;           // scale q e^G
                    ok[e] = kb * EL;            // k e^(G_last - G)
                    ov[e] = bt[r] * vf;         // beta v
                    orr[e] = bt[r] * (ka * EM); // beta k e^G
                    vm = max_abs_nan(max_abs_nan(vm, oq[e]), ok[e]);
                    vm = max_abs_nan(max_abs_nan(vm, ov[e]), orr[e]);
                }
                qh[r2] = pack_f16(oq[0], oq[1]);
                kgp[r2] = pack_f16(ok[0], ok[1]);
                rv[r2] = pack_f16(ov[0], ov[1]);
                rk[r2] = pack_f16(orr[0], orr[1]);
            }
            vmax = max_abs_nan(vmax, vm);
            tmem_st8(tl + TM_RV + 32 * bb + 8 * blk, rv);
            tmem_st8(tl + TM_RK + 32 * bb + 8 * blk, rk);
            tmem_wait_st();
        }
        const bool fast = misc[21] != 0;  // written during the previous task's strips
        tc_fence_before();
        sync_compute();  // input tiles consumed; strip operands and tables in place
        KDA_TRACE_EV(p, 21, 0);
        // Is this task's slot known to be free (checked during the previous task)?
        // If so, the previous task's WY product is read out and its slot published
        // by warps 10-13 while the strips run. Otherwise every warp reads it out
        // now, the slot is published, and only then is this task's slot awaited,
        // so that no producer waits for a consumer while it holds an unpublished chunk.
        if (!fast) {
            if (x_pending) {
                wait_local(R, bar_x, (it - 1) & 1, p.status);
                tc_fence_after();
                read_out_x(tl, slot_of(R, prev), chn, blk, blk + 1, vmax);
                x_pending = false;
            }
            tc_fence_before();
            sync_compute();  // every write of the previous slot issued; X^T read out
            if (tid == REL_TID) {
                if (prev.valid) publish(p, R, prev);
                const bool ok = slot_free(R, cur, R.spin);
                if (!ok) {
                    set_status(p.status, KDA_ERR_TIMEOUT);
                    atomicExch(&R.hdr->abort, 1);
                }
                misc[20] = ok ? 1 : 0;
            }
            sync_compute();
            if (!misc[20]) break;
            prev.valid = 0;
        }
        KDA_TRACE_EV(p, 22, 0);
        unsigned char *dst = slot_of(R, cur);
        st_row32(dst + SL_B1, 128, chn, 16 * blk, qh);
        st_row32(dst + SL_B23, 192, chn, 16 * blk, kgp);
        if (blk == 0) reinterpret_cast<float *>(dst + SL_D)[chn] = ex2(Gl);

        // ---- step 2b: Aqk and Akk on the 10 lower 16x16 tiles in four groups,
        // warps 0-3 (one per sub-partition): rows {0,1} x columns {0,1},
        // rows {2,3} x column 0, rows {2,3} x column 1, rows {2,3} x columns {2,3}
        static_assert(NWARPS == 16, "warps 0-3 strips, 4-9 next inputs, 10-13 WY read-out, 14-15 diagonal inverses");
        if (warp < 4) {
            if (warp == 0) strip_group<0, 0, 2>(smem, dst, sBeta, scale, lane);
            else if (warp == 1) strip_group<2, 0, 1>(smem, dst, sBeta, scale, lane);
            else if (warp == 2) strip_group<2, 1, 1>(smem, dst, sBeta, scale, lane);
            else strip_group<2, 2, 2>(smem, dst, sBeta, scale, lane);
            if (warp == 0 || warp == 3) {  // the diagonal blocks of L are in place: hand them to the inverse warps
                __syncwarp();
                named_bar_arrive(2, 128);
            }
            if (lane == 0) KDA_TRACE_ANY(p, 40 + warp, 0);
        }
        // ---- warps 4-9: the next task's inputs (the input tiles are free) and its draw
        if (warp >= 4 && warp < 10) {
            if (tid == SYNC_TID) {
                const Task t = fetch_task(p, smem, cu_s, jmax, cs);
                put_task(misc + 2, t);
            }
            if (nxt.valid) issue_loads(p, smem, nxt, bb ^ 1, 4 * 32, 6 * 32);
        }
        // ---- step 3a, on warps 14 and 15 (two blocks each, 16 lanes per block)
        // while the strips run: T_ii = (I + L_ii)^-1 by fp32 forward substitution,
        // once the four warps with the diagonal tiles have written them
        if (warp >= 14) {
            named_bar_sync(2, 128);
            const int i = 2 * (warp - 14) + (lane >> 4), jc = lane & 15;
            const float *Ld = sLD + i * 16 * 17;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float sacc = (r == jc) ? 1.f : 0.f;
#pragma unroll
                for (int cc = 0; cc < r; ++cc) sacc -= Ld[r * 17 + cc] * x[cc];
                x[r] = sacc;
            }
            float vm = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                vm = max_abs_nan(vm, x[r]);
                *reinterpret_cast<__half *>(sT + tile_elem(64, 16 * i + r, 16 * i + jc)) = __float2half_rn(x[r]);
            }
            vmax = max_abs_nan(vmax, vm);
            if (lane == 0) KDA_TRACE_ANY(p, 50 + warp - 14, 0);
        }
        // ---- warps 10-13 (one per lane quarter): the previous task's WY product
        // into its slot, then its publication; and whether the next task's slot
        // is free: one flag load, issued first and completed by the publication's
        // fence (an acquire), so that nothing here waits on a consumer
        if (warp >= 10 && warp < 14) {
            const bool need_check = nxt.valid && nxt.j >= RING;
            int fr = 0;
            if (tid == REL_TID && need_check) fr = ld_relaxed(&R.freed[nxt.k * RING + nxt.j % RING]);
            if (x_pending) {
                wait_local(R, bar_x, (it - 1) & 1, p.status);
                tc_fence_after();
                read_out_x(tl, slot_of(R, prev), chn, 0, 4, vmax);
            }
            if (cur.j < RING) {  // the first use of this slot: the tiles of Aqk above the diagonal are zero
                for (int idx = tid - 10 * 32; idx < 6 * 16 * 2; idx += 128) {
                    const int tile = idx >> 5, rr = (idx >> 1) & 15, half = idx & 1;
                    const int i = tile < 3 ? 0 : (tile < 5 ? 1 : 2);
                    const int j = tile < 3 ? tile + 1 : (tile < 5 ? tile - 1 : 3);
                    *reinterpret_cast<uint4 *>(dst + SL_B23 + tile_chunk(192, 128 + 16 * i + rr, 16 * j + 8 * half)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            named_bar_sync(6, 128);
            if (tid == REL_TID) {
                if (x_pending && prev.valid)
                    publish(p, R, prev);
                else if (need_check)
                    fence_acq_rel_gpu();
                misc[21] = (nxt.valid && (!need_check || fr >= nxt.j - RING + 1)) ? 1 : 0;
                KDA_TRACE_ANY(p, 29, 0);
            }
        }
        sync_compute();
        x_pending = false;
        const Task nxt2 = get_task(misc + 2);  // drawn after the elementwise step
        KDA_TRACE_EV(p, 23, 0);

        // ---- step 3b: the block diagonals d = 1, 2, 3 of T = (I + L)^-1,
        // T_ij = -T_ii * sum_{k=j}^{i-1} L_ik T_kj, one block per warp
#pragma unroll
        for (int d = 1; d < 4; ++d) {
            if (warp < 4 - d) {
                const int j = warp, i = warp + d;
                float m[2][4] = {};
                for (int kb = j; kb < i; ++kb) {
                    uint32_t fa[4], fb[4];
                    ldsm_x4(fa, sL + (16 * i + (lane & 15)) * RSA + 16 * kb + ((lane >> 4) << 3));
                    ldsm_x4_t(fb, sT + bk_addr(lane, 64, 16 * kb, 16 * j));
                    mma16816_f16(m[0], fa, fb[0], fb[1]);
                    mma16816_f16(m[1], fa, fb[2], fb[3]);
                }
                float vm = 0.f;
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        vm = max_abs_nan(max_abs_nan(vm, m[nt][2 * hf]), m[nt][2 * hf + 1]);
                        *reinterpret_cast<uint32_t *>(sT + tile_elem(64, 16 * i + gq + 8 * hf, 16 * j + 8 * nt + 2 * qd)) =
                            pack_f16(m[nt][2 * hf], m[nt][2 * hf + 1]);
                    }
                __syncwarp();
                float t[2][4] = {};
                {
                    uint32_t fa[4], fb[4];
                    ldsm_x4(fa, sT + a_addr(lane, 64, 16 * i, 16 * i));
                    ldsm_x4_t(fb, sT + bk_addr(lane, 64, 16 * i, 16 * j));
                    mma16816_f16(t[0], fa, fb[0], fb[1]);
                    mma16816_f16(t[1], fa, fb[2], fb[3]);
                }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        vm = max_abs_nan(max_abs_nan(vm, t[nt][2 * hf]), t[nt][2 * hf + 1]);
                        *reinterpret_cast<uint32_t *>(sT + tile_elem(64, 16 * i + gq + 8 * hf, 16 * j + 8 * nt + 2 * qd)) =
                            pack_f16(-t[nt][2 * hf], -t[nt][2 * hf + 1]);
                    }
                vmax = max_abs_nan(vmax, vm);
            }
            if (d < 3) sync_compute();
        }
        // ---- step 4b: X^T = R^T T^T = [u | w]^T on the tensor cores (A operands
        // in tensor memory), read out during the next task
        fence_proxy_async_shared();  // T's generic writes, before the tensor core reads it
        tc_fence_before();
        sync_compute();
        KDA_TRACE_EV(p, 24, 0);
        if (tid == 0) {
            tc_fence_after();
            const uint32_t tb = smem_u32(sT);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_f16_ts(tmem + TM_XU, tmem + TM_RV + 32 * bb + 8 * kk, umma_desc_sw128(tb + kk * 32, 16, 1024), idesc_x,
                            kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_f16_ts(tmem + TM_XW, tmem + TM_RK + 32 * bb + 8 * kk, umma_desc_sw128(tb + kk * 32, 16, 1024), idesc_x,
                            kk > 0);
            umma_commit(bar_x);
        }
        x_pending = true;
        prev = cur;
        ++it;
        KDA_TRACE_EV(p, 3, cur.j * p.C + cur.k);
        cur = nxt;
        nxt = nxt2;
    }
    // the last task's WY product: read out, then publish its slot
    if (x_pending) {
        wait_local(R, bar_x, (it - 1) & 1, p.status);
        tc_fence_after();
        read_out_x(tl, slot_of(R, prev), chn, blk, blk + 1, vmax);
        tc_fence_before();
        sync_compute();
        if (tid == REL_TID) publish(p, R, prev);
    }
    cp_async_wait_all();
    if (gate_bad) set_status(p.status, KDA_ERR_GATE_RANGE);
    if (!(vmax < F16_SAFE)) set_status(p.status, KDA_ERR_VALUE_RANGE);
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}
}  // namespace prod

// ================================================================== consumer
// Step 5 on the 5th-generation tensor cores, on the transposed state: tensor
// memory holds S^T (fp32, lane = value column j, column = key channel c), next
// to it D^T = [q_hat S ; w S]^T (columns 128-191: tokens of q_hat S, which
// become o^T; 192-255: tokens of w S), and the two fp16 A operands of the
// chunk, S16^T and v_new^T. One thread issues the products; warp w serves lanes
// 32 (w % 4) .. + 31 (value columns), key columns 32 (w / 4) .. + 31 of S^T and
// tokens 16 (w / 4) .. + 15 of D^T.
//   MMA1   D^T  = S16^T (tensor memory, 128 x 128) * [q_hat ; w]^T (MN-major)
//   MMA23  [S^T | o^T] += v_new^T (tensor memory, 128 x 64) * [kg^T ; Aqk]
//          (K-major, N = 192), after S^T <- S^T Diag(d)
// Only E1 (the fp16 copy of S^T), MMA1, E2 (v_new) and MMA23 are on the chain;
// the decay and the previous chunk's o rows are done while MMA1 runs.
namespace cons {
constexpr int OFF_BUF0 = 0;
constexpr int OFF_BUF1 = SLOT_BYTES;            // 1024-aligned
constexpr int OFF_RED = 2 * SLOT_BYTES;         // gated norm: per-quarter row sums [4][64], then 1/rms [64]
constexpr int OFF_BAR = OFF_RED + 1280;         // full[2], mma1, mma23
constexpr int OFF_TMEM = OFF_BAR + 32;          // TMEM base address written by tcgen05.alloc
constexpr int OFF_MISC = OFF_BAR + 64;
constexpr int SMEM = OFF_MISC + 64;
constexpr uint32_t TM_S = 0, TM_DQ = 128, TM_DW = 192, TM_S16 = 256, TM_VN = 320, TM_COLS = 512;
static_assert(SLOT_BYTES % 1024 == 0, "slot buffers are 1024-byte aligned");

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

// The o rows of one chunk (first token t0, nv valid rows, head h) from this
// thread's slice of o^T: value column jv, tokens 16 cg .. 16 cg + 15. Each warp
// store writes 32 consecutive value columns of one row (128 contiguous bytes).
// With the fused gated RMSNorm, the rows' sums of squares are reduced over the
// warp's 32 columns (a butterfly that leaves lane l with the sum of token
// T(l)), then over the four column quarters in shared memory; called by all
// threads together (it holds two CTA barriers).
__device__ __forceinline__ void store_o(const Params &p, unsigned char *smem, const uint32_t (&ov)[16], int64_t t0, int nv,
                                        int h, int jv, int cg, int lane, int quad, const uint32_t (&gt)[8], float nw,
                                        int e0 = 0, int e1 = 16) {
    const int tid = threadIdx.x;
    float x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(ov[e]);
    if (p.ngate) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = x[e] * x[e];
#pragma unroll
        for (int w = 16, n = 8; w >= 2; w >>= 1, n >>= 1) {  // halve the values held, pairing lanes l and l ^ w
            const bool up = (lane & w) != 0;
#pragma unroll
            for (int e = 0; e < n; ++e) {
                const float send = up ? v[e] : v[e + n];
                const float keep = up ? v[e + n] : v[e];
                v[e] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        const int tok = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
        float *red = reinterpret_cast<float *>(smem + OFF_RED);
        if ((lane & 1) == 0) red[quad * 64 + 16 * cg + tok] = v[0];
        sync_compute();
        if (tid < BT)
            red[256 + tid] = rsqrtf(((red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid])) * (1.f / DV) + p.neps);
        sync_compute();
        float rs[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 r4 = reinterpret_cast<const float4 *>(red + 256 + 16 * cg)[q];
            rs[4 * q] = r4.x; rs[4 * q + 1] = r4.y; rs[4 * q + 2] = r4.z; rs[4 * q + 3] = r4.w;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 sg = unpack_f16(sigmoid_bf16x2_to_f16x2(gt[e]));
            x[2 * e] *= rs[2 * e] * nw * sg.x;
            x[2 * e + 1] *= rs[2 * e + 1] * nw * sg.y;
        }
    }
    if (p.o) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int t = 16 * cg + e;
            if (e >= e0 && e < e1 && t < nv) p.o[(static_cast<size_t>(t0 + t) * p.H + h) * DV + jv] = x[e];
        }
    }
}

// the gate values of this thread's o slice (tokens 16 cg .. + 15 of column jv),
// as bf16 pairs of consecutive tokens (zero past the chunk's valid rows)
__device__ __forceinline__ void load_gate(const Params &p, uint32_t (&gt)[8], int64_t t0, int nv, int h, int jv, int cg) {
    const unsigned short *gp = reinterpret_cast<const unsigned short *>(p.ngate);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int t = 16 * cg + 2 * e;
        const uint32_t lo = t < nv ? __ldg(gp + (static_cast<size_t>(t0 + t) * p.H + h) * DV + jv) : 0u;
        const uint32_t hi = t + 1 < nv ? __ldg(gp + (static_cast<size_t>(t0 + t + 1) * p.H + h) * DV + jv) : 0u;
        gt[e] = lo | (hi << 16);
    }
}

__device__ __forceinline__ void run(const Params &p, unsigned char *smem, int k) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, cg = warp >> 2;  // TMEM lane quarter; key-column / token group
    const int jv = 32 * quad + lane;            // this thread's value column (TMEM lane)
    Ring R = ring_of(p);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *bar_mma1 = full + 2;
    uint64_t *bar_mma23 = full + 3;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + OFF_TMEM);
    int *misc = reinterpret_cast<int *>(smem + OFF_MISC);

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(bar_mma1, 1);
        mbar_init(bar_mma23, 1);
        mbar_fence_init();
        misc[0] = 1;
    }
    if (warp == 0) tmem_alloc(tslot, TM_COLS);
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * quad) << 16);  // this warp's lane quarter
    const int32_t *cu_s = sched_cu(p, smem);
    const int total = consumer_total(p, smem, cu_s, k);

    auto issue = [&](int jj) {  // slot jj -> buffer jj % 2 (thread 0)
        const unsigned char *src = R.slots + static_cast<size_t>(k * RING + jj % RING) * SLOT_BYTES;
        unsigned char *dst = smem + ((jj & 1) ? OFF_BUF1 : OFF_BUF0);
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&full[jj & 1], SLOT_BYTES);
        bulk_g2s(dst, src, SLOT_BYTES, &full[jj & 1]);
    };
    bool issued_next = false;  // thread 0 only
    if (tid == 0 && total > 0) {
        if (wait_flag_geq(R, &R.ready[k * RING], 1, p.status))
            issue(0);
        else
            misc[0] = 0;
    }
    const uint32_t idesc1 = umma_idesc_f16(false, true, 128, 128);    // S16^T x [q_hat; w]^T (MN-major)
    const uint32_t idesc23 = umma_idesc_f16(false, false, 128, 192);  // v_new^T x [kg^T; Aqk] (K-major)
    const float nw = p.ngate ? __ldg(p.nweight + jv) : 0.f;

    int jj = 0, n23 = 0;
    float vmax = 0.f;  // largest magnitude sent to an fp16 operand (NaN if any was NaN)
    bool alive = true;
    bool pend = false;  // o^T of the chunk (pt0, pnv, ph) waits in D^T to be stored
    int64_t pt0 = 0;
    int pnv = 0, ph = 0;
    uint32_t gt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
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
        const size_t state_base = (static_cast<size_t>(n) * p.H + h) * (DK * DV);
        // entry state (or zeros) -> S^T: lane jv, key columns 32 cg .. + 31 (each
        // warp load reads 32 consecutive value columns of one key row)
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
            uint32_t s[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
                s[e] = p.s0 ? __float_as_uint(__ldg(p.s0 + state_base + static_cast<size_t>(32 * cg + 16 * cb + e) * DV + jv))
                            : 0u;
            tmem_st16(tl + TM_S + 32 * cg + 16 * cb, s);
        }
        tmem_wait_st();

        for (int c = 0; c < nc; ++c, ++jj) {
            const int b = jj & 1;
            const int64_t t0 = bos + static_cast<int64_t>(c) * BT;
            const int nv = static_cast<int>((bos + len - t0) < BT ? (bos + len - t0) : BT);
            KDA_TRACE_EV(p, 10, jj);
            if (c > 0) {  // the previous chunk's MMA23: S^T and its o^T are final, its buffer is free
                wait_local(R, bar_mma23, (n23 - 1) & 1, p.status);
                tc_fence_after();
            }
            // (1) slot jj has landed: release its ring slot, start fetching slot jj + 1
            if (tid == 0) {
                const bool was_alive = misc[0] != 0;  // then slot jj's copy has been issued
                if (was_alive && wait_mbar(R, &full[b], (jj >> 1) & 1, p.status)) {
                    // the copy of slot jj has completed (its reads are done): free the
                    // slot without ordering this thread's pending o stores before it
                    st_relaxed(&R.freed[k * RING + jj % RING], jj + 1);
                    issued_next = false;
                    if (jj + 1 < total && ld_acquire(&R.ready[k * RING + (jj + 1) % RING]) >= jj + 2) {
                        issue(jj + 1);
                        issued_next = true;
                    }
                } else {
                    if (was_alive) drain_mbar(&full[b], (jj >> 1) & 1);  // let it land before leaving
                    misc[0] = 0;
                }
            }
            if (pend && p.ngate) load_gate(p, gt, pt0, pnv, ph, jv, cg);
            sync_compute();
            if (!misc[0]) {
                alive = false;
                break;
            }
            for (int it = 0; !mbar_try_wait(&full[b], (jj >> 1) & 1); ++it)
                if (it > (1 << 20)) {
                    set_status(p.status, KDA_ERR_TIMEOUT);
                    break;
                }
            const unsigned char *bb = smem + (b ? OFF_BUF1 : OFF_BUF0);
            KDA_TRACE_EV(p, 11, jj);

            // (2) E1: fp16 copy of S^T for MMA1 (and the previous chunk's o^T into registers)
            uint32_t sa[16], sb[16], ov[16];
            tmem_ld16(tl + TM_S + 32 * cg, sa);
            tmem_ld16(tl + TM_S + 32 * cg + 16, sb);
            if (pend) tmem_ld16(tl + TM_DQ + 16 * cg, ov);
            tmem_wait_ld();
            {
                uint32_t hp[16];
                float vm = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float a0 = __uint_as_float(sa[2 * e]), a1 = __uint_as_float(sa[2 * e + 1]);
                    const float b0 = __uint_as_float(sb[2 * e]), b1 = __uint_as_float(sb[2 * e + 1]);
                    vm = max_abs_nan(max_abs_nan(vm, a0), a1);
                    vm = max_abs_nan(max_abs_nan(vm, b0), b1);
                    hp[e] = pack_f16(a0, a1);
                    hp[8 + e] = pack_f16(b0, b1);
                }
                vmax = max_abs_nan(vmax, vm);
                tmem_st16(tl + TM_S16 + 16 * cg, hp);
            }
            tmem_wait_st();
            tc_fence_before();
            sync_compute();
            // (3) MMA1: D^T = S16^T [q_hat ; w]^T
            if (tid == 0) {
                tc_fence_after();
                const uint32_t b1 = smem_u32(bb + SL_B1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_f16_ts(tmem + TM_DQ, tmem + TM_S16 + 8 * kk, umma_desc_sw128(b1 + kk * 2048, 16384, 1024), idesc1,
                                kk > 0);
                umma_commit(bar_mma1);
            }
            KDA_TRACE_EV(p, 13, jj);
            // (4) off the chain while MMA1 runs: S^T <- S^T Diag(d), and the
            // previous chunk's o rows
            {
                const float4 *dp = reinterpret_cast<const float4 *>(bb + SL_D) + 8 * cg;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 d0 = dp[q], d1 = dp[4 + q];
                    sa[4 * q] = __float_as_uint(__uint_as_float(sa[4 * q]) * d0.x);
                    sa[4 * q + 1] = __float_as_uint(__uint_as_float(sa[4 * q + 1]) * d0.y);
                    sa[4 * q + 2] = __float_as_uint(__uint_as_float(sa[4 * q + 2]) * d0.z);
                    sa[4 * q + 3] = __float_as_uint(__uint_as_float(sa[4 * q + 3]) * d0.w);
                    sb[4 * q] = __float_as_uint(__uint_as_float(sb[4 * q]) * d1.x);
                    sb[4 * q + 1] = __float_as_uint(__uint_as_float(sb[4 * q + 1]) * d1.y);
                    sb[4 * q + 2] = __float_as_uint(__uint_as_float(sb[4 * q + 2]) * d1.z);
                    sb[4 * q + 3] = __float_as_uint(__uint_as_float(sb[4 * q + 3]) * d1.w);
                }
                tmem_st16(tl + TM_S + 32 * cg, sa);
                tmem_st16(tl + TM_S + 32 * cg + 16, sb);
            }
            KDA_TRACE_EV(p, 15, jj);
            // the first half of the previous chunk's o rows (the other half is stored
            // while MMA23 runs; with the gated norm all of them are, then)
            if (pend && !p.ngate) store_o(p, smem, ov, pt0, pnv, ph, jv, cg, lane, quad, gt, nw, 0, 8);
            tmem_wait_st();
            KDA_TRACE_EV(p, 16, jj);

            // (5) E2: v_new^T = u^T - (w S)^T -> fp16 A operand of MMA23
            wait_local(R, bar_mma1, jj & 1, p.status);
            tc_fence_after();
            KDA_TRACE_EV(p, 14, jj);
            {
                uint32_t dw[16];
                tmem_ld16(tl + TM_DW + 16 * cg, dw);
                const uint4 u0 = *reinterpret_cast<const uint4 *>(bb + SL_U + tile_chunk(128, jv, 16 * cg));
                const uint4 u1 = *reinterpret_cast<const uint4 *>(bb + SL_U + tile_chunk(128, jv, 16 * cg + 8));
                const uint32_t uw[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                tmem_wait_ld();
                uint32_t vp[8];
                float vm = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 u2 = unpack_f16(uw[e]);
                    const float y0 = u2.x - __uint_as_float(dw[2 * e]);
                    const float y1 = u2.y - __uint_as_float(dw[2 * e + 1]);
                    vm = max_abs_nan(max_abs_nan(vm, y0), y1);
                    vp[e] = pack_f16(y0, y1);
                }
                vmax = max_abs_nan(vmax, vm);
                tmem_st8(tl + TM_VN + 8 * cg, vp);
            }
            tmem_wait_st();
            tc_fence_before();
            sync_compute();
            // (6) MMA23: [S^T | o^T] += v_new^T [kg^T ; Aqk]
            if (tid == 0) {
                tc_fence_after();
                const uint32_t b23 = smem_u32(bb + SL_B23);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_f16_ts(tmem + TM_S, tmem + TM_VN + 8 * kk, umma_desc_sw128(b23 + kk * 32, 16, 1024), idesc23, 1);
                umma_commit(bar_mma23);
            }
            if (pend) store_o(p, smem, ov, pt0, pnv, ph, jv, cg, lane, quad, gt, nw, p.ngate ? 0 : 8, 16);
            ++n23;
            pend = true;
            pt0 = t0;
            pnv = nv;
            ph = h;
            KDA_TRACE_EV(p, 12, jj);
            if (tid == 0 && !issued_next && jj + 1 < total) {
                if (wait_flag_geq(R, &R.ready[k * RING + (jj + 1) % RING], jj + 2, p.status))
                    issue(jj + 1);
                else
                    misc[0] = 0;
            }
        }
        if (!alive) break;
        if (nc > 0) {  // the chain's last o rows
            wait_local(R, bar_mma23, (n23 - 1) & 1, p.status);
            tc_fence_after();
            if (p.ngate) load_gate(p, gt, pt0, pnv, ph, jv, cg);
            uint32_t ov[16];
            tmem_ld16(tl + TM_DQ + 16 * cg, ov);
            tmem_wait_ld();
            store_o(p, smem, ov, pt0, pnv, ph, jv, cg, lane, quad, gt, nw);
            pend = false;
        }
        // final state: S^T -> global (each warp store writes 32 consecutive value columns)
        if (p.sT) {
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
                uint32_t s[16];
                tmem_ld16(tl + TM_S + 32 * cg + 16 * cb, s);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    p.sT[state_base + static_cast<size_t>(32 * cg + 16 * cb + e) * DV + jv] = __uint_as_float(s[e]);
            }
        }
        tc_fence_before();
        sync_compute();
        tc_fence_after();
    }
    if (!(vmax < F16_SAFE)) set_status(p.status, KDA_ERR_VALUE_RANGE);
    tc_fence_before();
    sync_compute();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
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

__global__ void __launch_bounds__(NTHREADS, 1) kda_persistent_kernel(const __grid_constant__ Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
#ifdef KDA_TRACE
    if (threadIdx.x < 16) reinterpret_cast<int *>(smem_raw + TRACE_COUNTS_OFFSET)[threadIdx.x] = 0;
    __syncthreads();
#endif
    build_sched(p, smem + OFF_SCHED, smem);  // the roles' tiles serve as scratch until it returns
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
    cudaError_t e = cudaFuncSetAttribute(kda_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_MAX);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_persistent_kernel, NTHREADS, SMEM_MAX);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = sms;  // one CTA per SM; all co-resident (cooperative launch)
    const int64_t chains = static_cast<int64_t>(p.N) * p.H;
    p.C = consumers_for(chains, p.T, p.N, grid);
    p.Cws = max_consumers(chains, grid);
    p.spin = p.debug ? SPIN_LIMIT_DEBUG : SPIN_LIMIT;
    if (ws_bytes < ring_offset(p.Cws) + static_cast<size_t>(p.Cws) * RING * SLOT_BYTES) return cudaErrorInvalidValue;
    e = cudaMemsetAsync(p.ws, 0, ring_offset(p.C), stream);
    if (e != cudaSuccess) return e;
#ifdef KDA_TRACE
    e = cudaMemsetAsync(p.ws + ring_offset(p.Cws) + static_cast<size_t>(p.Cws) * RING * SLOT_BYTES, 0,
                        static_cast<size_t>(grid) * TRACE_CTA_WORDS * 8, stream);
    if (e != cudaSuccess) return e;
#endif
    void *args[] = {&p};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(kda_persistent_kernel), dim3(grid), dim3(NTHREADS),
                                       args, SMEM_MAX, stream);
}

}  // namespace pers
}  // namespace kda
