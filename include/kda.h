/*
 * kda.h — C ABI of the KDA (Kimi Delta Attention) chunked-prefill forward
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (source: "在 TPU 上加速 Kimi K3 KDA", junyi.dev tpu-kda report,
 * §1–§2 for the recurrence, §4 and §6.2 for the chunked form, §6.5 for the
 * per-sequence state carry):
 *
 *   for every sequence n (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1) and head h,
 *   with S the [K,V] state (row = key channel) starting at initial_state[n,h]:
 *       S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *       o_t = scale * S_t^T q_t
 *   and final_state[n,h] = S after the sequence's last token.
 *
 * The library computes it chunk by chunk (64-token chunks, 16-token
 * sub-blocks): per-chunk gate prefix sum, sub-block-midpoint strip products
 * for the decayed score matrices, a blocked 16x16 solve with (I+L), the WY
 * form, then the inter-chunk state recurrence fused with the output. The
 * sub-block products are safe in bf16 because lower_bound <= g <= 0 bounds
 * every factor by 2^(8*|lower_bound|/ln 2) (= 2^57.7 at lower_bound = -5,
 * §4 and §13).
 *
 * General contract
 *   - Every pointer argument is CUDA device memory owned by the caller
 *     (except where stated). The library allocates nothing: scratch space is a
 *     caller-provided workspace (kda_chunk_fwd_workspace_size). It keeps no
 *     state between calls; calls are thread-safe as long as concurrent calls
 *     use different workspaces.
 *   - Calls are asynchronous on `stream`. Argument errors detected on the host
 *     are returned synchronously and nothing is launched. Data errors detected
 *     on the device are written to *status_dev (when given); the outputs are
 *     then unspecified.
 *   - Results are deterministic: the same inputs give bitwise-equal outputs.
 */
#ifndef KDA_GB300_KDA_H
#define KDA_GB300_KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 (NULL) is the legacy default stream. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null required pointer, bad size, misalignment, bad scalar */
    KDA_ERR_UNSUPPORTED = 2, /* head_dim_k or head_dim_v other than 128, or
                                total_tokens above 2^31 - 65 */
    KDA_ERR_CUDA = 3,        /* a CUDA runtime call or the launch failed */
    KDA_ERR_GATE_RANGE = 4,  /* device: some g outside [lower_bound, 0] or not finite */
    KDA_ERR_BAD_SEQLENS = 5, /* device: cu_seqlens not 0 .. total_tokens nondecreasing */
    KDA_ERR_TIMEOUT = 6,     /* device: a bounded wait inside a kernel gave up */
    KDA_ERR_VALUE_RANGE = 7, /* device: a value entering an fp16 tensor-core operand
                                exceeded 6e4 in magnitude (or was not finite) */
    KDA_ERR_SCRATCH_TOO_SMALL = 8, /* kda_chunk_fwd_static_scratch: the problem needs more
                                      scratch than KDA_STATIC_SCRATCH_BYTES */
    KDA_ERR_BOUNDS = 9 /* device, only in a library compiled with -DKDA_DEBUG_BOUNDS: an
                          index checked before a global-memory access fell outside its
                          buffer; that access was skipped (no trap) */
} kda_status_t;

#define KDA_HEAD_DIM 128
#define KDA_CHUNK 64
#define KDA_SUBBLOCK 16

/*
 * kda_chunk_fwd — KDA chunked prefill forward over varlen-packed sequences.
 *
 * Defined by the recurrence above (report §1–§2, §13) computed in the chunked
 * form of §4 and §6.2, with the state restarting per sequence (§6.5).
 *
 * Inputs (device memory, row-major, contiguous):
 *   q, k          bf16 [total_tokens, num_heads, 128]; k is expected to be
 *                 L2-normalised per (token, head) as in the model (not checked).
 *   v             bf16 [total_tokens, num_heads, 128].
 *                 total_tokens may not exceed 2^31 - 65 (token offsets of the
 *                 per-chunk tasks are 32-bit).
 *   g             fp32 [total_tokens, num_heads, 128]: natural-log decay per
 *                 key channel, already activated; lower_bound <= g <= 0.
 *   beta          fp32 [total_tokens, num_heads].
 *   cu_seqlens    int32 [num_seqs + 1]: cu[0] = 0, nondecreasing,
 *                 cu[num_seqs] = total_tokens. Empty sequences are allowed.
 *   initial_state fp32 [num_seqs, num_heads, 128, 128] (S[i][j], i = key
 *                 channel, j = value channel), or NULL for zeros.
 *   scale         multiplies o only (typically 128^-0.5).
 *   lower_bound   the gate's lower bound; must lie in [-10, 0) so that the
 *                 sub-block factors 2^(8 |lower_bound| / ln 2) stay below 2^126.
 * Outputs:
 *   o             fp32 [total_tokens, num_heads, 128]. (fp32 rather than bf16: a
 *                 bf16 o alone would round the largest outputs by up to 2^-9 of
 *                 their magnitude, several percent of the output RMS for the
 *                 heavy-tailed outputs of this operation.)
 *   final_state   fp32 [num_seqs, num_heads, 128, 128], or NULL (not written).
 *                 It may be the same pointer as initial_state (updated in
 *                 place); any other overlap between outputs and inputs is
 *                 undefined.
 *   status_dev    optional device int32: set to 0 on the stream before the
 *                 launch, then to the first device-detected error code
 *                 (KDA_ERR_GATE_RANGE, KDA_ERR_BAD_SEQLENS, KDA_ERR_TIMEOUT,
 *                 KDA_ERR_VALUE_RANGE).
 *                 A chain whose sequence bounds are invalid is skipped, so no
 *                 access leaves the given buffers.
 * Alignment: q, k, v, g, o, initial_state, final_state 16-byte aligned;
 *   beta, cu_seqlens, status_dev 4-byte aligned.
 * Precision: products run on tensor cores with fp32 accumulation. The Aqk
 *   strip operands are tf32 (fp32's exponent range holds the 2^57.7 factors,
 *   with 11 significant bits); the Akk strips use bf16; the solve, WY form,
 *   state recurrence and output products use fp16 operands. The state stays fp32 across the whole sequence. Inputs must
 *   keep |v|, |initial_state| and the state below ~6e4 (fp16 operand range);
 *   otherwise KDA_ERR_VALUE_RANGE is reported.
 *   workspace     device scratch of at least kda_chunk_fwd_workspace_size(num_seqs,
 *                 num_heads) bytes, 16-byte aligned, used by one call at a time
 *                 (its first bytes are reset on the stream at every call; calls
 *                 that overlap on the GPU must not share it).
 * Execution: one persistent kernel with one CTA per SM, launched cooperatively
 *   (all CTAs resident). Producer CTAs run the intra-chunk steps for
 *   (chain, chunk) tasks and hand the results through a ring in the workspace
 *   to consumer CTAs that own the chains and carry the state; every wait is
 *   bounded and a wait that runs out reports KDA_ERR_TIMEOUT.
 * Returns KDA_OK once the work is queued, or a host-side error code with
 * nothing launched. num_seqs == 0 launches nothing.
 */
kda_status_t kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                           int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                           int32_t head_dim_v, const float *initial_state, float scale,
                           float lower_bound, float *o, float *final_state,
                           int32_t *status_dev, void *workspace, size_t workspace_bytes,
                           kda_stream_t stream);

/*
 * kda_chunk_fwd_raw_gates — kda_chunk_fwd taking the gate and beta before their
 * activations, which run inside the kernel on the tiles it has loaded: the
 * fusion of "在 TPU 上加速 Kimi K3 KDA" §6.1 (activate_gate(g, A_log[head],
 * dt_bias[head]) moves into the intra-chunk kernel ahead of the chunk prefix
 * sum) and of the fused beta sigmoid in the Kimi K3 PP16 prefill notes' flag
 * table. The pages name the gate activation without defining it; this library
 * reads it as
 *     g    = lower_bound * sigmoid(exp(A_log[h]) * (g_raw + dt_bias[h][c]))
 *     beta = sigmoid(beta_raw)
 * which keeps lower_bound <= g <= 0 by construction and, with A_log = 0 and
 * dt_bias = 0, is the g = lower_bound * sigmoid(x) form of the synthetic inputs.
 *   g_raw     fp32 [total_tokens, num_heads, 128], 16-byte aligned
 *   beta_raw  fp32 [total_tokens, num_heads], 4-byte aligned
 *   A_log     fp32 [num_heads], or NULL for zeros
 *   dt_bias   fp32 [num_heads, 128], 16-byte aligned, or NULL for zeros
 * Every other argument, output, limit and error is as for kda_chunk_fwd
 * (KDA_ERR_GATE_RANGE then flags only non-finite activated gates).
 */
kda_status_t kda_chunk_fwd_raw_gates(const void *q, const void *k, const void *v, const float *g_raw,
                                     const float *beta_raw, const float *A_log, const float *dt_bias,
                                     const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                     int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                     const float *initial_state, float scale, float lower_bound, float *o,
                                     float *final_state, int32_t *status_dev, void *workspace,
                                     size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_gated_norm — kda_chunk_fwd with the gated RMSNorm of the
 * output fused into the kernel's output store: the KDA output tail of the
 * Kimi K3 PP16 prefill notes' flag table (the strided o-norm entry, which fuses
 * FusedRMSNormGated with the copy its reshape forced). The page names the
 * operation without writing it out; this library reads it as, per token t and
 * head h over the 128 value channels c,
 *     o[t][h][c] = x[t][h][c] / sqrt(mean_c(x[t][h][:]^2) + norm_eps)
 *                  * norm_weight[c] * sigmoid(gate[t][h][c])
 * where x is the attention output kda_chunk_fwd would write: an RMS
 * normalisation over one head's value channels, a per-channel weight shared by
 * the heads, and a sigmoid output gate.
 *   gate         bf16 [total_tokens, num_heads, 128], 16-byte aligned
 *   norm_weight  fp32 [128], 16-byte aligned
 *   norm_eps     > 0 and finite (1e-5 is usual)
 *   o            receives the normalised, gated output (fp32, as above); x is
 *                not written anywhere
 * final_state and every other argument, limit and error are as for
 * kda_chunk_fwd. The norm runs in fp32 on the fp32 output rows; the sigmoid is
 * evaluated as 1/2 + tanh(x/2)/2 on the packed fp16 hardware tanh (absolute
 * error about 1e-3, below bf16's resolution at 1).
 */
kda_status_t kda_chunk_fwd_gated_norm(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                      int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                                      int32_t head_dim_v, const float *initial_state, float scale,
                                      float lower_bound, const void *gate, const float *norm_weight,
                                      float norm_eps, float *o, float *final_state, int32_t *status_dev,
                                      void *workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_split — kda_chunk_fwd for calls with few, long (sequence, head)
 * chains, where the plain call runs each chain's chunks one after another on a
 * few SMs (for example one long sequence with a few heads per GPU). Long
 * sequences are cut at chunk boundaries into segments of `segment_chunks`
 * chunks. The chunk recurrence of "在 TPU 上加速 Kimi K3 KDA" §6.2 is affine in
 * the state, so a segment maps its entry state to its exit state as
 * S_out = Phi S_in + N, and by linearity N is the exit state from a zero entry
 * state and Phi + N the exit state from the identity. The call runs
 *   1. one chunked launch over the segments except each sequence's last
 *      (segment 0 from the sequence's entry state, the others from I and from
 *      0), keeping only their exit states;
 *   2. a combine kernel: S_1 = exit of segment 0, S_{s+1} = Phi_s S_s + N_s in
 *      fp32;
 *   3. one chunked launch over all segments as sequences of their own, from
 *      their entry states S_s, writing o;
 *   4. a copy of each sequence's last exit state into final_state.
 *   cu_seqlens_host  host copy of cu_seqlens (int32 [num_seqs + 1]); the plan
 *                    and the segment tables are built from it (validated: 0,
 *                    nondecreasing, total_tokens). cu_seqlens (device) is read
 *                    only when nothing is split.
 *   segment_chunks   segment length in 64-token chunks; 0 lets the library
 *                    choose (kda_chunk_fwd_split_plan); a sequence of more
 *                    chunks is cut into segments of that length (at most 64;
 *                    the last takes the rest). With no sequence cut, this is
 *                    exactly kda_chunk_fwd.
 *   workspace        at least kda_chunk_fwd_split_workspace_size(cu_seqlens_host,
 *                    num_seqs, num_heads, segment_chunks) bytes, 256-byte
 *                    aligned: the ring, the segment tables and four state arrays
 *                    (about 4 x 64 KiB per segment and head).
 * Other arguments, outputs and errors as kda_chunk_fwd (num_heads at most
 * 65535). o and final_state agree with kda_chunk_fwd within the parity
 * tolerance, not bitwise (the entry states come through the fp32 combine).
 * Launches: 1 without a cut; otherwise 4, plus 1 when final_state is given,
 * plus one host-to-device copy of the tables (from pageable memory, staged
 * before the call returns).
 */
kda_status_t kda_chunk_fwd_split(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                 const int32_t *cu_seqlens, const int32_t *cu_seqlens_host, int32_t num_seqs,
                                 int64_t total_tokens, int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                 const float *initial_state, float scale, float lower_bound, int32_t segment_chunks,
                                 float *o, float *final_state, int32_t *status_dev, void *workspace,
                                 size_t workspace_bytes, kda_stream_t stream);

/* How kda_chunk_fwd lays out a call of num_seqs sequences, total_tokens tokens
 * and num_heads heads on a GPU with num_sms SMs (0: the current device), with
 * one CTA per SM:
 *   *consumers        the consumers that carry the chains' recurrence (the
 *                     other CTAs run the intra-chunk steps for them);
 *   *wy_on_consumers  1 when those consumers also form the WY product
 *                     X = T [beta v | beta k e^G] (the producers then send T),
 *                     0 when the producers form it;
 *   *split_columns    1 when each consumer is a pair of CTAs taking one half of
 *                     the 128 value columns each (then one chain per consumer),
 *                     0 when it is one CTA.
 * plain_device_o: 1 for an o in device memory without the gated norm (full
 * chunks of o leave by tensor stores), 0 otherwise; the consumers take the WY
 * product only in the first case. (The gated norm never splits columns; this
 * call does not model it.) Host only; nothing is launched. Returns
 * KDA_OK; KDA_ERR_INVALID_ARG for num_seqs or num_heads below 1, a negative
 * total_tokens or num_sms, or a NULL output; KDA_ERR_UNSUPPORTED for fewer than
 * two SMs; KDA_ERR_CUDA when num_sms is 0 and no device answers.
 * (Not part of the method: the pages define no counterpart.)
 */
kda_status_t kda_chunk_fwd_plan(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t num_sms,
                                int32_t plain_device_o, int32_t *consumers, int32_t *wy_on_consumers,
                                int32_t *split_columns);

/* The segment length (chunks) kda_chunk_fwd_split picks for these lengths on a
 * GPU with num_sms SMs (0: the current device), from the measured paces of the
 * chunked kernel (a busy consumer SM finishes a chunk every 3.5 us, a producer
 * SM every 7.0 us, a launch costs about 15 us); 0 when no segment length is
 * estimated to beat the plain call by 20 %, or the arguments are invalid. */
int32_t kda_chunk_fwd_split_plan(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                 int32_t num_sms);

/* Workspace bytes of kda_chunk_fwd_split for these lengths and segment length
 * (0: the planned one) on the current device; 0 on invalid arguments or when no
 * usable device is current. */
size_t kda_chunk_fwd_split_workspace_size(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                          int32_t segment_chunks);

/*
 * kda_chunk_fwd_host — kda_chunk_fwd on inputs and outputs in HOST memory (a
 * deployment convenience of this library; the pages have no counterpart).
 * With groups = 0 and every buffer in page-locked host memory that the device
 * addresses at the same pointer (cudaHostAlloc memory, or cudaHostRegister'ed
 * memory mapped into the device's address space, under unified addressing),
 * one kernel launch reads the inputs and writes o and final_state in host
 * memory directly over the CPU-GPU link, with no staging copy; h2d_stream and
 * d2h_stream are then unused. Otherwise the transfers are overlapped with the
 * computation: the sequences are cut into
 * `groups` groups of whole sequences with about equal token counts (0: 4;
 * at most 16 and num_seqs). Group i's q, k, v, g, beta and initial states are
 * copied to the device on h2d_stream; `stream` waits for them and runs the
 * chunked kernel on that group alone; d2h_stream waits for that launch and
 * copies the group's o and final states back. Copies of neighbouring groups
 * thus run while a group computes. `stream` finally waits for the last copy
 * back: when it is synchronised, o and final_state hold the results.
 *   q .. beta, initial_state, o, final_state  host memory, layouts as in
 *                   kda_chunk_fwd; page-locked memory lets the copies overlap
 *                   (with pageable memory they still complete, but serialise).
 *                   final_state may alias initial_state.
 *   cu_seqlens_host host int32 [num_seqs + 1] (validated: 0, nondecreasing,
 *                   total_tokens).
 *   device_buffer   device memory of at least kda_chunk_fwd_host_buffer_size(...)
 *                   bytes, 256-byte aligned: device copies of every input and
 *                   output, the rebased offsets and the kernel's workspace; not
 *                   to be shared by calls that overlap on the GPU.
 *   h2d_stream, d2h_stream  streams for the copies in and out (NULL: `stream`,
 *                   which serialises the copies with the computation).
 *   status_dev      optional device int32, as for kda_chunk_fwd.
 * Creates and releases 2 x groups + 2 CUDA events per call (no memory).
 * Returns KDA_OK once everything is queued, or a host-side error code.
 */
kda_status_t kda_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *cu_seqlens_host, int32_t num_seqs, int64_t total_tokens,
                                int32_t num_heads, int32_t head_dim_k, int32_t head_dim_v,
                                const float *initial_state, float scale, float lower_bound, float *o,
                                float *final_state, int32_t *status_dev, void *device_buffer,
                                size_t device_buffer_bytes, int32_t groups, kda_stream_t stream,
                                kda_stream_t h2d_stream, kda_stream_t d2h_stream);

/* Device buffer bytes of kda_chunk_fwd_host for these lengths (with or without
 * initial and final states, and `groups` as in the call) on the current device;
 * 0 on invalid arguments or when no usable device is current. */
size_t kda_chunk_fwd_host_buffer_size(const int32_t *cu_seqlens_host, int32_t num_seqs, int32_t num_heads,
                                      int32_t with_initial_state, int32_t with_final_state, int32_t groups);

/* Workspace bytes kda_chunk_fwd needs for these sizes on the current device
 * (0 when num_seqs or num_heads is 0, or no usable device is current). */
size_t kda_chunk_fwd_workspace_size(int32_t num_seqs, int32_t num_heads);

/* Size of the fixed device scratch array behind kda_chunk_fwd_static_scratch
 * (a build may define a different size). */
#ifndef KDA_STATIC_SCRATCH_BYTES
#define KDA_STATIC_SCRATCH_BYTES (26u << 20)
#endif

/*
 * kda_chunk_fwd_static_scratch — kda_chunk_fwd for callers that cannot allocate
 * device memory, not even a workspace: for example a runtime whose device
 * memory is a fixed arena planned before it starts, a real-time host that
 * forbids allocation after start-up, or a plugin that receives its input and
 * output tensors but cannot request memory. (The TPU report has no
 * counterpart: this is a deployment convenience of this library.)
 *
 * Arguments, layouts, results and asynchronous behaviour are those of
 * kda_chunk_fwd, without the workspace pair. The scratch instead comes from
 * one fixed __device__ array of KDA_STATIC_SCRATCH_BYTES (26 MiB) compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits. No call allocates or frees memory.
 *
 * Each call looks up the array's device address with cudaGetSymbolAddress on
 * the current device (so a reset device context is no problem); the first
 * call on a device also loads the library's device code there, so make it
 * before any stream capture. Every call on a device shares the one array and
 * it keeps the previous call's contents (the part that must start at zero is
 * cleared on the stream by each call), so calls whose GPU work may overlap
 * (different streams, or different host threads) race on it and must be
 * serialised by the caller.
 *
 * Returns KDA_ERR_SCRATCH_TOO_SMALL, with nothing launched, when
 * kda_chunk_fwd_workspace_size(num_seqs, num_heads) exceeds
 * KDA_STATIC_SCRATCH_BYTES; otherwise what kda_chunk_fwd returns.
 */
kda_status_t kda_chunk_fwd_static_scratch(const void *q, const void *k, const void *v, const float *g,
                                          const float *beta, const int32_t *cu_seqlens,
                                          int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                          int32_t head_dim_k, int32_t head_dim_v,
                                          const float *initial_state, float scale, float lower_bound,
                                          float *o, float *final_state, int32_t *status_dev,
                                          kda_stream_t stream);

/*
 * kda_chunk_fwd_debug — kda_chunk_fwd with diagnostic flags, for testing the
 * failure detection without a GPU fault. Arguments, layouts, ownership and
 * return codes are those of kda_chunk_fwd; debug_flags is a combination of:
 *
 *   KDA_DEBUG_WITHHOLD_READY  producers compute every chunk but never publish
 *                             it to its consumer, so the consumers' waits for
 *                             their first chunk run out: the device reports
 *                             KDA_ERR_TIMEOUT in status_dev, every CTA leaves
 *                             (after its own copies have landed and its tensor
 *                             memory is freed) and the context stays usable.
 *
 *   KDA_DEBUG_WY_PRODUCER     the producer CTAs form the WY product
 *                             X = T [beta v | beta k e^G] (u and w go to the
 *                             consumers), whatever the launch's own choice.
 *   KDA_DEBUG_WY_CONSUMER     the consumer CTAs form it (they receive T, beta v
 *                             and beta k e^G and compute v_new = T (beta v -
 *                             beta k e^G S)). Both forms compute the same o and
 *                             final_state within the parity bar; a launch
 *                             normally picks one from the batch's shape (the
 *                             consumers' form only where all sequences can be
 *                             of one length, o is a plain device array (no
 *                             gated norm) and the consumers have slack).
 *                             Setting both returns KDA_ERR_INVALID_ARG.
 *   KDA_DEBUG_SPLIT_COLUMNS   each chain's 128 value columns go to a pair of
 *                             consumer CTAs, one half each, where every chain
 *                             can have a pair within half the SMs (else the
 *                             flag is ignored), whatever the launch's choice.
 *   KDA_DEBUG_WHOLE_COLUMNS   one consumer CTA takes all of a chain's columns.
 *                             Setting both, or KDA_DEBUG_SPLIT_COLUMNS with
 *                             KDA_DEBUG_WY_CONSUMER, returns KDA_ERR_INVALID_ARG.
 *
 * With KDA_DEBUG_WITHHOLD_READY set, a wait gives up after 2^14 polls
 * (milliseconds) instead of 2^24; o and final_state are then unspecified.
 * debug_flags = 0 is exactly kda_chunk_fwd. Unknown flags return
 * KDA_ERR_INVALID_ARG.
 * (Not part of the method: the pages define no counterpart.)
 */
#define KDA_DEBUG_WITHHOLD_READY 1u
#define KDA_DEBUG_WY_PRODUCER 2u
#define KDA_DEBUG_WY_CONSUMER 4u
#define KDA_DEBUG_SPLIT_COLUMNS 8u
#define KDA_DEBUG_WHOLE_COLUMNS 16u
kda_status_t kda_chunk_fwd_debug(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                 int64_t total_tokens, int32_t num_heads, int32_t head_dim_k,
                                 int32_t head_dim_v, const float *initial_state, float scale,
                                 float lower_bound, float *o, float *final_state,
                                 int32_t *status_dev, void *workspace, size_t workspace_bytes,
                                 kda_stream_t stream, uint32_t debug_flags);

/*
 * kda_decode_fwd — the KDA recurrence for a few tokens per sequence (decode /
 * recurrent step), with the state carried in and out.
 *
 * Defined by the token recurrence above (report §1–§2), applied token after
 * token:  S <- Diag(e^{g_t}) S;  S <- S + beta_t k_t (v_t^T - k_t^T S);
 * o_t = scale * S^T q_t. It is the same operation kda_chunk_fwd computes, for
 * batches of equally short sequences, where the chunked form has no chunk to
 * work on: every sequence has exactly tokens_per_seq tokens.
 *
 * Inputs (device memory, row-major, contiguous; T = num_seqs * tokens_per_seq,
 * the tokens of sequence n at rows n*tokens_per_seq .. n*tokens_per_seq + tokens_per_seq - 1):
 *   q, k, v       bf16 [T, num_heads, 128]
 *   g             fp32 [T, num_heads, 128] (natural-log decay, lower_bound <= g <= 0)
 *   beta          fp32 [T, num_heads]
 *   initial_state fp32 [num_seqs, num_heads, 128, 128] (key rows) or NULL for zeros
 *   tokens_per_seq  0 .. KDA_DECODE_MAX_TOKENS (0: the state passes through)
 * Outputs:
 *   o             fp32 [T, num_heads, 128]
 *   final_state   fp32 [num_seqs, num_heads, 128, 128] or NULL; may be the same
 *                 pointer as initial_state (the usual in-place decode update)
 *   status_dev    optional device int32, zeroed on the stream, then set to
 *                 KDA_ERR_GATE_RANGE if some g lies outside [lower_bound, 0]
 * Arithmetic is fp32 throughout. One launch; asynchronous on `stream`; nothing
 * is allocated. Alignment: q, k, v, g, o and the states 16-byte aligned, beta
 * and status_dev 4-byte aligned. Returns KDA_OK once queued, or a host-side
 * error code with nothing launched. (The fused decode step of "Kimi K3 на
 * графических процессорах AMD Instinct" §1.2 also folds in the short
 * convolution and the output norm; those steps are outside this call.)
 */
#define KDA_DECODE_MAX_TOKENS 64
kda_status_t kda_decode_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                            int32_t num_seqs, int32_t tokens_per_seq, int32_t num_heads, int32_t head_dim_k,
                            int32_t head_dim_v, const float *initial_state, float scale, float lower_bound,
                            float *o, float *final_state, int32_t *status_dev, kda_stream_t stream);

/* Number of kernel launches one kda_chunk_fwd call makes for these sizes
 * (0 when num_seqs == 0). Host-only, no CUDA call. */
int32_t kda_chunk_fwd_launches(int32_t num_seqs, int64_t total_tokens, int32_t num_heads);

/* Static description of an error code; never NULL. */
const char *kda_status_string(int32_t status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H */
