// KDA chunked prefill forward — one CTA per (sequence, head) chain, every
// contraction on warp-level tensor-core MMA (m16n8k16, fp32 accumulate), the
// 128x128 fp32 state held in registers across the chain.
//
// Operand precision (chosen so o and the final state stay within 1.5% of the
// output RMS in max-abs error even for heavy-tailed outputs):
//   Aqk strips      split bf16 (hi + lo, three products): bf16's exponent range
//                   holds the midpoint factors up to 2^57.7, the split keeps
//                   about 16 significant bits on the path into o;
//   Akk strips      bf16 (the solve is insensitive to their rounding);
//   solve, WY form, state recurrence and output products: fp16 operands
//                   (every one of them is bounded well inside fp16's range for
//                   |v| and |state| below 6e4; larger values set
//                   KDA_ERR_VALUE_RANGE);
//   o               written in fp32.
//
// Follows "在 TPU 上加速 Kimi K3 KDA" (junyi.dev tpu-kda report):
//   step 1  gate prefix sum inside the chunk (§6.1), kept in base 2;
//   step 2  Aqk / Akk as 16x16 products of midpoint-rescaled operands (§4):
//           exp(G_t - G_s) = exp(G_t - G_m) * exp(G_m - G_s), with m the
//           midpoint (row 16i+7) of the row's sub-block i, so every factor
//           stays below 2^(8*|lower_bound|/ln 2) (§4, §13);
//   step 3  (I+L)^-1 applied by 16x16 block forward substitution, the four
//           diagonal blocks inverted exactly in fp32;
//   step 4  WY form u = (I+L)^-1 beta v, w = (I+L)^-1 (beta k exp(G)) (§4, §6.3);
//   step 5  v_new = u - w S, o = q exp(G) S + Aqk v_new, then
//           S <- Diag(exp(G_last)) S + (k exp(G_last - G))^T v_new, reading the
//           entry state (§6.2); only o and final_state reach memory (§6.2–§6.3).
// Chunks restart at each sequence start (§6.4–§6.5); rows past the end of a
// partial chunk are zero-filled (k = v = beta = g = 0), which makes them
// inert in every product.
#include "kda_common.cuh"
#include "kda.h"

namespace kda {
namespace chain_mma {

constexpr int NT = 256;   // 8 warps
constexpr int RSB = 136;  // 16-bit row stride of [*][128] tiles (272 B: conflict-free ldmatrix)
constexpr int RSF = 136;  // fp32 row stride of [64][128] fp32 tiles
constexpr int RSA = 72;   // 16-bit row stride of [64][64] tiles
constexpr int RSI = 24;   // 16-bit row stride of the 16x16 inverse blocks

constexpr int SZ_T = BT * RSB * 2;        // 17408: one [64][128] 16-bit tile
constexpr int SZ_F = BT * RSF * 4;        // 34816: one [64][128] fp32 tile
constexpr int OFF_Q = 0;                  // q -> q*a (bf16 hi)
constexpr int OFF_QLO = OFF_Q + SZ_T;     // q*a (bf16 lo)
constexpr int OFF_K = OFF_QLO + SZ_T;     // k -> k*a (bf16) -> v_new (fp16)
constexpr int OFF_V = OFF_K + SZ_T;       // v -> beta*v (fp16) -> u (fp16)
constexpr int OFF_RK = OFF_V + SZ_T;      // beta*k*e^G (fp16) -> w (fp16)
constexpr int OFF_G = OFF_RK + SZ_T;      // g -> G (fp32) -> [q_hat | kg] (fp16)
constexpr int OFF_KB = OFF_G + SZ_F;      // k*e^(G_m - G) (fp32) -> u (fp32)
constexpr int OFF_SB = OFF_KB + SZ_F;     // state in fp16 [128][RSB]
constexpr int SZ_SB = DK * RSB * 2;       // 34816
constexpr int OFF_AQK = OFF_SB + SZ_SB;   // scale * Aqk (fp16, causal incl. diagonal)
constexpr int SZ_A = BT * RSA * 2;        // 9216
constexpr int OFF_L = OFF_AQK + SZ_A;     // L = beta * tril(Akk,-1) (fp16)
constexpr int OFF_LD = OFF_L + SZ_A;      // diagonal blocks of L in fp32 [4][16][17]
constexpr int SZ_LD = 4 * 16 * 17 * 4;    // 4352
constexpr int OFF_INV = OFF_LD + SZ_LD;   // (I+L_ii)^-1 in fp16 [4][16][RSI]
constexpr int SZ_INV = 4 * 16 * RSI * 2;  // 3072
constexpr int OFF_TAB = OFF_INV + SZ_INV; // per-channel tables (fp32)
constexpr int SZ_TAB = 20 * 128 * 4;      // 10240
constexpr int OFF_BETA = OFF_TAB + SZ_TAB;
constexpr int OFF_FLAG = OFF_BETA + BT * 4;
constexpr int SMEM_BYTES = OFF_FLAG + 16;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(2 * SZ_T <= SZ_F, "q_hat and kg fit in the gate region");
// table rows (each 128 floats): GM[4] GL[1] EM[4] EL[4] F[6] D[1]
constexpr int TGM = 0, TGL = 4 * 128, TEM = 5 * 128, TEL = 9 * 128, TF = 13 * 128, TD = 19 * 128;

__device__ __forceinline__ int f_pair(int i, int j) { return i * (i - 1) / 2 + j; }  // i > j

__device__ __forceinline__ bool f16_ok(float x) { return fabsf(x) < F16_SAFE; }  // false for NaN too

__global__ void __launch_bounds__(NT, 1)
kda_chain_mma_kernel(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                     const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
                     const float *__restrict__ beta, const int32_t *__restrict__ cu_seqlens,
                     int32_t num_seqs, int64_t total_tokens, int32_t H,
                     const float *initial_state, float scale, float lower_bound,
                     float *__restrict__ o, float *final_state, int32_t *status) {
    extern __shared__ __align__(128) unsigned char smem[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_Q);
    __nv_bfloat16 *sQlo = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_QLO);
    __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_K);
    __half *sVN = reinterpret_cast<__half *>(smem + OFF_K);
    __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(smem + OFF_V);
    __half *sRV = reinterpret_cast<__half *>(smem + OFF_V);
    __half *sRK = reinterpret_cast<__half *>(smem + OFF_RK);
    float *sG = reinterpret_cast<float *>(smem + OFF_G);
    __half *sQh = reinterpret_cast<__half *>(smem + OFF_G);
    __half *sKg = reinterpret_cast<__half *>(smem + OFF_G + SZ_T);
    float *sKB = reinterpret_cast<float *>(smem + OFF_KB);
    float *sU = reinterpret_cast<float *>(smem + OFF_KB);
    __half *sSB = reinterpret_cast<__half *>(smem + OFF_SB);
    __half *sAqk = reinterpret_cast<__half *>(smem + OFF_AQK);
    __half *sL = reinterpret_cast<__half *>(smem + OFF_L);
    float *sLD = reinterpret_cast<float *>(smem + OFF_LD);
    __half *sInv = reinterpret_cast<__half *>(smem + OFF_INV);
    float *sTab = reinterpret_cast<float *>(smem + OFF_TAB);
    float *sBeta = reinterpret_cast<float *>(smem + OFF_BETA);
    int *sFlag = reinterpret_cast<int *>(smem + OFF_FLAG);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, qd = lane & 3;  // fragment row group / quad position
    const int64_t chain = blockIdx.x;
    const int n = static_cast<int>(chain / H), h = static_cast<int>(chain % H);

    // ---- sequence bounds (device-side validation: never read outside the buffers)
    const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
    bool bad = bos < 0 || eos < bos || eos > total_tokens;
    if (n == 0 && bos != 0) bad = true;
    if (n == num_seqs - 1 && eos != total_tokens) bad = true;
    if (bad) {
        if (tid == 0) set_status(status, KDA_ERR_BAD_SEQLENS);
        return;
    }
    if (tid == 0) sFlag[0] = sFlag[1] = 0;
    bool range_bad = false;

    // ---- state: warp w owns key rows [16w, 16w+16), all 128 value columns
    float S[16][4];
    const size_t state_base = (static_cast<size_t>(n) * H + h) * (DK * DV);
    {
        const int r0 = 16 * warp + gq;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = 8 * nt + 2 * qd;
            if (initial_state) {
                const float2 a = *reinterpret_cast<const float2 *>(initial_state + state_base + r0 * DV + c);
                const float2 b = *reinterpret_cast<const float2 *>(initial_state + state_base + (r0 + 8) * DV + c);
                S[nt][0] = a.x; S[nt][1] = a.y; S[nt][2] = b.x; S[nt][3] = b.y;
            } else {
                S[nt][0] = S[nt][1] = S[nt][2] = S[nt][3] = 0.f;
            }
        }
    }

    const int64_t L = eos - bos;
    const int nchunks = static_cast<int>((L + BT - 1) / BT);
    const size_t row_stride = static_cast<size_t>(H) * DK;  // elements between tokens

    for (int c = 0; c < nchunks; ++c) {
        const int64_t t0 = bos + static_cast<int64_t>(c) * BT;
        const int nv = static_cast<int>((eos - t0) < BT ? (eos - t0) : BT);  // valid rows
        __syncthreads();  // previous chunk fully consumed

        // ---- entry state in fp16 for this chunk's products (§6.2)
        {
            const int r0 = 16 * warp + gq;
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const int cc = 8 * nt + 2 * qd;
                range_bad |= !(f16_ok(S[nt][0]) && f16_ok(S[nt][1]) && f16_ok(S[nt][2]) && f16_ok(S[nt][3]));
                *reinterpret_cast<uint32_t *>(sSB + r0 * RSB + cc) = pack_f16(S[nt][0], S[nt][1]);
                *reinterpret_cast<uint32_t *>(sSB + (r0 + 8) * RSB + cc) = pack_f16(S[nt][2], S[nt][3]);
            }
        }

        // ---- load the chunk (rows >= nv zero-filled)
        {
            const size_t base = (static_cast<size_t>(t0) * H + h) * DK;
            for (int idx = tid; idx < BT * 16; idx += NT) {
                const int r = idx >> 4, c8 = (idx & 15) << 3;
                const bool ok = r < nv;
                const size_t off = base + (ok ? r * row_stride : 0) + c8;
                cp_async16(sQ + r * RSB + c8, q + off, ok ? 16 : 0);
                cp_async16(sK + r * RSB + c8, k + off, ok ? 16 : 0);
                cp_async16(sV + r * RSB + c8, v + off, ok ? 16 : 0);
            }
            for (int idx = tid; idx < BT * 32; idx += NT) {
                const int r = idx >> 5, c4 = (idx & 31) << 2;
                const bool ok = r < nv;
                cp_async16(sG + r * RSF + c4, g + base + (ok ? r * row_stride : 0) + c4, ok ? 16 : 0);
            }
            if (tid < BT) sBeta[tid] = tid < nv ? beta[static_cast<size_t>(t0 + tid) * H + h] : 0.f;
            cp_async_commit();
            cp_async_wait_all();
        }
        __syncthreads();

        // ---- step 1: inclusive prefix sum of g (base 2) per key channel + tables
        if (tid < DK) {
            const int ch = tid;
            float acc = 0.f;
            bool gbad = false;
#pragma unroll
            for (int r0 = 0; r0 < BT; r0 += 16) {
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = sG[(r0 + r) * RSF + ch];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    gbad |= !(x[r] >= lower_bound && x[r] <= 0.f);
                    acc += x[r] * LOG2E;
                    sG[(r0 + r) * RSF + ch] = acc;
                    if (r == 7) sTab[TGM + (r0 >> 4) * 128 + ch] = acc;
                }
            }
            // rows >= nv carry g = 0, so row 63 holds the last valid prefix
            const float gl = acc;
            sTab[TGL + ch] = gl;
            sTab[TD + ch] = ex2(gl);
            float gm[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) gm[i] = sTab[TGM + i * 128 + ch];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                sTab[TEM + i * 128 + ch] = ex2(gm[i]);
                sTab[TEL + i * 128 + ch] = ex2(gl - gm[i]);
            }
#pragma unroll
            for (int i = 1; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < i; ++j) sTab[TF + f_pair(i, j) * 128 + ch] = ex2(gm[i] - gm[j]);
            if (gbad) sFlag[0] = 1;
        }
        __syncthreads();

        // ---- steps 2a/4a: elementwise operands (4 groups of 8 channels per thread)
        {
            float Gv[4][8];
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int grp = tid + it * NT, r = grp >> 4, c8 = (grp & 15) << 3;
                const float4 a = *reinterpret_cast<const float4 *>(sG + r * RSF + c8);
                const float4 b = *reinterpret_cast<const float4 *>(sG + r * RSF + c8 + 4);
                Gv[it][0] = a.x; Gv[it][1] = a.y; Gv[it][2] = a.z; Gv[it][3] = a.w;
                Gv[it][4] = b.x; Gv[it][5] = b.y; Gv[it][6] = b.z; Gv[it][7] = b.w;
            }
            __syncthreads();  // the gate tile is overwritten below
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int grp = tid + it * NT, r = grp >> 4, c8 = (grp & 15) << 3;
                const int i = r >> 4;
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
                for (int p = 0; p < 4; ++p) {
                    const float2 qf = unpack_bf16(qw[p]), kf = unpack_bf16(kw[p]), vf = unpack_bf16(vw[p]);
                    float res[2][7];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int ch = c8 + 2 * p + e;
                        const float qq = e ? qf.y : qf.x, kk = e ? kf.y : kf.x, vv2 = e ? vf.y : vf.x;
                        const float x = Gv[it][2 * p + e] - sTab[TGM + i * 128 + ch];
                        const float a = ex2(x), b = ex2(-x);
                        const float eG = a * sTab[TEM + i * 128 + ch];
                        res[e][0] = qq * a;                              // q e^(G - G_m)
                        res[e][1] = kk * a;                              // k e^(G - G_m)
                        res[e][2] = bt * vv2;                            // beta v
                        res[e][3] = bt * kk * eG;                        // beta k e^G
                        res[e][4] = scale * qq * eG;                     // scale q e^G
                        res[e][5] = kk * b * sTab[TEL + i * 128 + ch];   // k e^(G_last - G)
                        kb[2 * p + e] = kk * b;                          // k e^(G_m - G)
                    }
                    split_bf16(res[0][0], res[1][0], oQh[p], oQl[p]);
                    oKa[p] = pack_bf16(res[0][1], res[1][1]);
                    range_bad |= !(f16_ok(res[0][2]) && f16_ok(res[1][2]));
                    oBv[p] = pack_f16(res[0][2], res[1][2]);
                    oBk[p] = pack_f16(res[0][3], res[1][3]);
                    oQs[p] = pack_f16(res[0][4], res[1][4]);
                    oKg[p] = pack_f16(res[0][5], res[1][5]);
                }
                *reinterpret_cast<uint4 *>(sQ + r * RSB + c8) = *reinterpret_cast<uint4 *>(oQh);
                *reinterpret_cast<uint4 *>(sQlo + r * RSB + c8) = *reinterpret_cast<uint4 *>(oQl);
                *reinterpret_cast<uint4 *>(sK + r * RSB + c8) = *reinterpret_cast<uint4 *>(oKa);
                *reinterpret_cast<uint4 *>(sRV + r * RSB + c8) = *reinterpret_cast<uint4 *>(oBv);
                *reinterpret_cast<uint4 *>(sRK + r * RSB + c8) = *reinterpret_cast<uint4 *>(oBk);
                *reinterpret_cast<uint4 *>(sQh + r * RSB + c8) = *reinterpret_cast<uint4 *>(oQs);
                *reinterpret_cast<uint4 *>(sKg + r * RSB + c8) = *reinterpret_cast<uint4 *>(oKg);
                *reinterpret_cast<float4 *>(sKB + r * RSF + c8) = make_float4(kb[0], kb[1], kb[2], kb[3]);
                *reinterpret_cast<float4 *>(sKB + r * RSF + c8 + 4) = make_float4(kb[4], kb[5], kb[6], kb[7]);
            }
        }
        __syncthreads();

        // ---- step 2b: Aqk and Akk on the 10 lower 16x16 tiles. Tile (i,j) needs
        // k_s e^(G_{m_i} - G_s) for s in sub-block j: the stored k e^(G_{m_j} - G)
        // times e^(G_{m_i} - G_{m_j}) (<= 1), formed in fp32 and split into bf16
        // hi + lo directly in the B fragments.
        for (int pair = warp; pair < 10; pair += 8) {
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
                ldsm_x4(fa, sQ + a_off(lane, 16 * i, 16 * kk, RSB));
                ldsm_x4(fl, sQlo + a_off(lane, 16 * i, 16 * kk, RSB));
                ldsm_x4(fk, sK + a_off(lane, 16 * i, 16 * kk, RSB));
                const int c0 = 16 * kk + 2 * qd;
                float2 f0 = make_float2(1.f, 1.f), f1 = make_float2(1.f, 1.f);
                if (i > j) {
                    f0 = *reinterpret_cast<const float2 *>(fr + c0);
                    f1 = *reinterpret_cast<const float2 *>(fr + c0 + 8);
                }
                uint32_t bh[2][2], bl[2][2];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const float *row = nt ? kbrow1 : kbrow0;
                    const float2 x0 = *reinterpret_cast<const float2 *>(row + c0);
                    const float2 x1 = *reinterpret_cast<const float2 *>(row + c0 + 8);
                    split_bf16(x0.x * f0.x, x0.y * f0.y, bh[nt][0], bl[nt][0]);
                    split_bf16(x1.x * f1.x, x1.y * f1.y, bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    mma16816(aq[nt], fa, bh[nt][0], bh[nt][1]);
                    mma16816(aq[nt], fl, bh[nt][0], bh[nt][1]);
                    mma16816(aq[nt], fa, bl[nt][0], bl[nt][1]);
                    mma16816(ak[nt], fk, bh[nt][0], bh[nt][1]);
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
        __syncthreads();

        // ---- step 3a: (I + L_ii)^-1 for the four diagonal blocks, fp32 substitution
        if (warp < 4 && lane < 16) {
            const int i = warp, jc = lane;  // column jc of the inverse
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
        __syncthreads();

        // ---- steps 3b/4: X = (I+L)^-1 [beta v | beta k e^G], block forward
        // substitution; warp w owns 32 right-hand-side columns
        {
            __half *R = (warp < 4) ? sRV : sRK;
            const int col0 = 32 * (warp & 3);
            for (int i = 0; i < 4; ++i) {
                float acc[4][4] = {};
                for (int j = 0; j < i; ++j) {
                    uint32_t fa[4];
                    ldsm_x4(fa, sL + a_off(lane, 16 * i, 16 * j, RSA));
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        uint32_t fb[4];
                        ldsm_x4_t(fb, R + bk_off(lane, 16 * j, col0 + 16 * nb, RSB));
                        mma16816_f16(acc[2 * nb], fa, fb[0], fb[1]);
                        mma16816_f16(acc[2 * nb + 1], fa, fb[2], fb[3]);
                    }
                }
                // Y_i = R_i - sum_j L_ij X_j, written in place (fp16)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t *p = reinterpret_cast<uint32_t *>(R + (16 * i + gq + 8 * hf) * RSB + col0 + 8 * nt + 2 * qd);
                        const float2 rv = unpack_f16(*p);
                        const float y0 = rv.x - acc[nt][2 * hf], y1 = rv.y - acc[nt][2 * hf + 1];
                        range_bad |= !(f16_ok(y0) && f16_ok(y1));
                        *p = pack_f16(y0, y1);
                    }
                __syncwarp();
                float xo[4][4] = {};
                {
                    uint32_t fa[4];
                    ldsm_x4(fa, sInv + a_off(lane, 16 * i, 0, RSI));
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        uint32_t fb[4];
                        ldsm_x4_t(fb, R + bk_off(lane, 16 * i, col0 + 16 * nb, RSB));
                        mma16816_f16(xo[2 * nb], fa, fb[0], fb[1]);
                        mma16816_f16(xo[2 * nb + 1], fa, fb[2], fb[3]);
                    }
                }
                __syncwarp();
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        const int rr = 16 * i + gq + 8 * hf, cc = col0 + 8 * nt + 2 * qd;
                        range_bad |= !(f16_ok(xo[nt][2 * hf]) && f16_ok(xo[nt][2 * hf + 1]));
                        *reinterpret_cast<uint32_t *>(R + rr * RSB + cc) = pack_f16(xo[nt][2 * hf], xo[nt][2 * hf + 1]);
                        if (warp < 4)
                            *reinterpret_cast<float2 *>(sU + rr * RSF + cc) = make_float2(xo[nt][2 * hf], xo[nt][2 * hf + 1]);
                    }
                __syncwarp();
            }
        }
        __syncthreads();

        // ---- step 5a: [w S ; q_hat S] for a 16-token x 64-value tile per warp
        const int rb = warp & 3, chv = warp >> 2;
        float accW[8][4] = {}, accO[8][4] = {};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t fw[4], fq[4];
            ldsm_x4(fw, sRK + a_off(lane, 16 * rb, 16 * kk, RSB));
            ldsm_x4(fq, sQh + a_off(lane, 16 * rb, 16 * kk, RSB));
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                uint32_t fb[4];
                ldsm_x4_t(fb, sSB + bk_off(lane, 16 * kk, 64 * chv + 16 * nb, RSB));
                mma16816_f16(accW[2 * nb], fw, fb[0], fb[1]);
                mma16816_f16(accW[2 * nb + 1], fw, fb[2], fb[3]);
                mma16816_f16(accO[2 * nb], fq, fb[0], fb[1]);
                mma16816_f16(accO[2 * nb + 1], fq, fb[2], fb[3]);
            }
        }
        // v_new = u - w S  -> fp16 into the (dead) k*a tile
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int rr = 16 * rb + gq + 8 * hf, cc = 64 * chv + 8 * nt + 2 * qd;
                const float2 u = *reinterpret_cast<const float2 *>(sU + rr * RSF + cc);
                const float y0 = u.x - accW[nt][2 * hf], y1 = u.y - accW[nt][2 * hf + 1];
                range_bad |= !(f16_ok(y0) && f16_ok(y1));
                *reinterpret_cast<uint32_t *>(sVN + rr * RSB + cc) = pack_f16(y0, y1);
            }
        __syncthreads();

        // ---- step 5b: o = q_hat S + (scale Aqk) v_new (causal: token blocks <= rb)
        for (int kk = 0; kk <= rb; ++kk) {
            uint32_t fa[4];
            ldsm_x4(fa, sAqk + a_off(lane, 16 * rb, 16 * kk, RSA));
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                uint32_t fb[4];
                ldsm_x4_t(fb, sVN + bk_off(lane, 16 * kk, 64 * chv + 16 * nb, RSB));
                mma16816_f16(accO[2 * nb], fa, fb[0], fb[1]);
                mma16816_f16(accO[2 * nb + 1], fa, fb[2], fb[3]);
            }
        }
        {
            const size_t base = (static_cast<size_t>(t0) * H + h) * DV;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int rr = 16 * rb + gq + 8 * hf;
                if (rr < nv) {
                    float *orow = o + base + rr * row_stride + 64 * chv + 2 * qd;
#pragma unroll
                    for (int nt = 0; nt < 8; ++nt)
                        *reinterpret_cast<float2 *>(orow + 8 * nt) = make_float2(accO[nt][2 * hf], accO[nt][2 * hf + 1]);
                }
            }
        }

        // ---- step 5c: S <- Diag(e^{G_last}) S + kg^T v_new (warp w: key rows 16w..)
        {
            const float d0 = sTab[TD + 16 * warp + gq], d1 = sTab[TD + 16 * warp + gq + 8];
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                S[nt][0] *= d0; S[nt][1] *= d0; S[nt][2] *= d1; S[nt][3] *= d1;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t fa[4];
                ldsm_x4_t(fa, sKg + at_off(lane, 16 * warp, 16 * kk, RSB));
#pragma unroll
                for (int nb = 0; nb < 8; ++nb) {
                    uint32_t fb[4];
                    ldsm_x4_t(fb, sVN + bk_off(lane, 16 * kk, 16 * nb, RSB));
                    mma16816_f16(S[2 * nb], fa, fb[0], fb[1]);
                    mma16816_f16(S[2 * nb + 1], fa, fb[2], fb[3]);
                }
            }
        }
    }

    // ---- final state
    if (final_state) {
        const int r0 = 16 * warp + gq;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int cc = 8 * nt + 2 * qd;
            *reinterpret_cast<float2 *>(final_state + state_base + r0 * DV + cc) = make_float2(S[nt][0], S[nt][1]);
            *reinterpret_cast<float2 *>(final_state + state_base + (r0 + 8) * DV + cc) = make_float2(S[nt][2], S[nt][3]);
        }
    }
    if (range_bad) sFlag[1] = 1;
    __syncthreads();
    if (tid == 0 && sFlag[0]) set_status(status, KDA_ERR_GATE_RANGE);
    if (tid == 0 && sFlag[1]) set_status(status, KDA_ERR_VALUE_RANGE);
}

cudaError_t launch(const void *q, const void *k, const void *v, const float *g, const float *beta,
                   const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t H,
                   const float *initial_state, float scale, float lower_bound, float *o,
                   float *final_state, int32_t *status, cudaStream_t stream) {
    static_assert(SMEM_BYTES > 48 * 1024, "opt-in shared memory");
    cudaError_t e = cudaFuncSetAttribute(kda_chain_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(num_seqs) * H);
    kda_chain_mma_kernel<<<grid, NT, SMEM_BYTES, stream>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<const __nv_bfloat16 *>(v), g, beta, cu_seqlens, num_seqs, total_tokens, H,
        initial_state, scale, lower_bound, o, final_state, status);
    return cudaGetLastError();
}

}  // namespace chain_mma
}  // namespace kda
