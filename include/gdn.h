/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) speculative-decoding hot path on GB300 (sm_103a).
 *
 * The operation is the GDN linear-attention core that hybrid Qwen3-Next-style layers run when a
 * speculative (draft + verify) step and ordinary decode/prefill rows share one batch:
 *   (1) a width-W causal depthwise conv1d + SiLU over the packed q|k|v channels, with each
 *       sequence's conv history kept as a rolled ring in a pool slot;
 *   (2) the sigmoid-gated delta rule over an fp32 d_v x d_k state per v-head, with one state
 *       slot per speculative position;
 *   (3) the split of a mixed batch into speculative and non-speculative rows, each read from
 *       and written back to interleaved global token positions through its own token index.
 *
 * Sources (page title, section):
 *   "[GDN] Spec-decoding-aware attention kernel" (vllm-xpu-kernels PR 336) -- Problem: the conv
 *       ring is a rolled history at column 0 of cache_indices, read at offset num_accepted-1;
 *       Changes: the two-pass conv (stage, then a roll pass that is the slot's only writer),
 *       the state load from spec_state_indices[n, num_accepted[n]-1], the per-token store to
 *       spec_state_indices[n, t], slot <= 0 meaning "no prior state", and the rule that
 *       spec_state_indices and num_accepted_tokens come as a pair.
 *   "[XE2] Support MTP of QWEN model" (vllm-xpu-kernels PR 368) -- Copilot overview: the
 *       spec/non-spec split, num_spec_decodes, token_indx remapping of reads and writes, the
 *       chunked prefill path; review notes: every optional tensor is checked before use;
 *       commit message: no rectangular assumption on spec rows, only the conservation check
 *       non_spec_tokens + spec_tokens == num_actual_tokens.
 *   "[Bugfix] Align Qwen GDN gates with speculative tokens" (vllm PR 51812) -- Purpose: the
 *       a/b gates are gathered with the same index as q|k|v.
 *
 * Conventions shared by every entry point.
 *   Pointers are DEVICE pointers unless stated, borrowed for the duration of the stream work;
 *   the caller owns all memory.  Calls only enqueue work on `stream` (a cudaStream_t passed as
 *   void*, NULL = legacy default stream); they never synchronise, never read device memory on
 *   the host, and allocate nothing.
 *   Dense row-major layouts, no strides.  C = 2*Hk*dk + Hv*dv channels, packed as
 *   q (Hk*dk) | k (Hk*dk) | v (Hv*dv), head-major (x may instead arrive per k-head, see
 *   gdn_qkv_layout).  v-head h uses k-head h / (Hv/Hk).
 *   Activations (x, a, b, out, conv pool, conv weight/bias) use gdn_layer_desc.act_dtype.
 *   The SSM pool is fp32 [num_slots, Hv, dv, dk] (dk fastest).  Conv pool [num_slots,
 *   conv_state_len, C].  Slot values <= 0 are NULL: zero prior on load, no write.
 *   Integer metadata is int32.  All activation, pool and weight pointers must be 16-byte
 *   aligned.
 *   Host-detectable problems return a negative gdn_error before anything is enqueued.
 *   Problems only visible in device data (an index out of range, num_accepted outside
 *   [1, spec_cols], a non-monotone query_start_loc, a spec row longer than spec_cols) never
 *   trap: the kernel ORs a GDN_STATUS_* bit into *d_status (if d_status is not NULL), treats
 *   the bad load as zero and skips the bad write (or the whole row, for row-level problems).
 *   Rows of one call must use distinct slots; overlapping slots give undefined results.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_NULL_ARG = -1,     /* a required pointer is NULL                                   */
  GDN_ERR_SPEC_PAIR = -2,    /* spec_state_indices without num_accepted_tokens, or vice versa */
  GDN_ERR_SHAPE = -3,        /* head/conv sizes, spec_cols, row counts or limits unsupported  */
  GDN_ERR_CONSERVATION = -4, /* non-spec tokens + spec tokens != num_actual_tokens            */
  GDN_ERR_WORKSPACE = -5,    /* workspace NULL or smaller than gdn_workspace_bytes()         */
  GDN_ERR_DTYPE = -6,        /* unknown gdn_dtype                                             */
  GDN_ERR_CUDA = -7,         /* a kernel launch failed (cudaGetLastError after the launch)    */
  GDN_ERR_ALIGN = -8         /* a pointer is not 16-byte aligned                              */
} gdn_error;

/* Bits ORed into *d_status by the kernels. */
#define GDN_STATUS_SLOT_RANGE 0x1u   /* a slot index >= num_slots (load read as zero, store skipped) */
#define GDN_STATUS_NUM_ACCEPTED 0x2u /* num_accepted_tokens[n] outside [1, spec_cols] (row skipped)  */
#define GDN_STATUS_TOKEN_RANGE 0x4u  /* token_indx outside [0, num_global_tokens) (read zero, write skipped) */
#define GDN_STATUS_ROW_RANGE 0x8u    /* query_start_loc not monotone / past num_tokens, or a spec row
                                        longer than spec_cols (row skipped)                            */
#define GDN_STATUS_WAIT_TIMEOUT 0x10u /* a bounded wait inside a tensor-core kernel gave up; that
                                         block's results are missing (never expected in practice)  */

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* Channel order of the pre-conv activation x ("[GDN] Spec-decoding-aware attention kernel",
 * Test Plan: reorder_input).  Packed: q (Hk*dk) | k (Hk*dk) | v (Hv*dv), head-major
 * (reorder_input=True).  Per k-head: for each k-head g, q_g (dk) | k_g (dk) | v of its
 * G = Hv/Hk v-heads (G*dv) -- the projection order of production Qwen3-Next traffic
 * (reorder_input=False).  Conv weights, bias, the conv pool and every post-conv tensor use the
 * packed order in both cases. */
typedef enum { GDN_QKV_PACKED = 0, GDN_QKV_PER_KHEAD = 1 } gdn_qkv_layout;

/* How a speculative row keeps its conv history.  Rolled: one rolled history in column 0 of the
 * row's slots, read at offset num_accepted-1 ("[GDN] Spec-decoding-aware attention kernel",
 * Problem; needs conv_state_len >= W-2+spec_cols).  Per slot: after spec token t the last W-1
 * inputs are written to columns 0..W-2 of spec_state_indices[n, t] and the next step reads
 * spec_state_indices[n, num_accepted-1] ("[XE2] Support MTP of QWEN model", review thread).
 * Non-speculative rows behave the same in both. */
typedef enum { GDN_CONV_ROLLED = 0, GDN_CONV_PER_SLOT = 1 } gdn_conv_layout;

typedef struct {
  int32_t num_k_heads;    /* Hk >= 1                                                   */
  int32_t num_v_heads;    /* Hv, a multiple of Hk                                      */
  int32_t head_k_dim;     /* dk in {16, 32, 64, 128}                                    */
  int32_t head_v_dim;     /* dv, a multiple of 16, <= 256                               */
  int32_t conv_width;     /* W in {2, 3, 4}                                             */
  int32_t conv_state_len; /* columns per conv slot, >= W-1 (rolled spec rows: >= W-2+spec_cols) */
  gdn_dtype act_dtype;    /* GDN_BF16 or GDN_F32                                        */
  float scale;            /* multiplies the normalised q; <= 0 selects 1/sqrt(dk)       */
  int32_t qkv_layout;     /* gdn_qkv_layout of x                                        */
  int32_t conv_layout;    /* gdn_conv_layout of speculative rows                        */
} gdn_layer_desc;

typedef struct {
  const void* conv_weight; /* [C, W] act dtype; w[c][W-1] multiplies the current token */
  const void* conv_bias;   /* [C] act dtype, or NULL for no bias                         */
  const float* A_log;      /* [Hv]: g = -exp(A_log[h]) * softplus(a + dt_bias[h])       */
  const float* dt_bias;    /* [Hv]                                                       */
} gdn_layer_params;

typedef struct {
  void* conv_pool;   /* [num_slots, conv_state_len, C] act dtype (read and written) */
  float* ssm_pool;   /* [num_slots, Hv, dv, dk] fp32 (read and written)             */
  int64_t num_slots; /* slot 0 is conventionally reserved as NULL                   */
} gdn_pools;

/*
 * One subset of rows.  spec_state_indices and num_accepted_tokens come as a pair (both, or
 * GDN_ERR_SPEC_PAIR).  A subset is speculative when it has the pair and no state_indices.
 * A non-speculative subset (state_indices given) may also carry the pair: its rows are then
 * acceptance-aware, i.e. each continues from what its previous verify step accepted -- a
 * verify row cut to a prefix by the batch token budget and scheduled as a plain row ("[Bugfix]
 * Align Qwen GDN gates with speculative tokens", the second mechanism in the reachability
 * comment).  Such a row reads its conv history at column offset num_accepted-1 of
 * state_indices[n] (rolled layout) or from spec_state_indices[n, num_accepted-1] (per-slot
 * layout), loads its SSM state from spec_state_indices[n, num_accepted-1], and writes like any
 * non-spec row.  A row that accepted one token with spec_state_indices[n, 0] == state_indices[n]
 * is an ordinary non-spec row.
 * Local tokens are numbered 0..num_tokens-1 in row order; row n owns local tokens
 * [query_start_loc[n], query_start_loc[n+1]).
 */
typedef struct {
  int32_t num_seqs;                   /* N_sub rows (may be 0)                                   */
  int32_t num_tokens;                 /* T_sub local tokens; query_start_loc[N_sub] must equal it */
  const int32_t* query_start_loc;     /* [N_sub+1], query_start_loc[0] == 0                       */
  const int32_t* token_indx;          /* [T_sub] global token of each local token; NULL = identity */
  const int32_t* state_indices;       /* non-spec: [N_sub] conv+SSM slot of each row              */
  const int32_t* has_initial_state;   /* non-spec: [N_sub], 0 = start from zeros; NULL = all 1    */
  const int32_t* spec_state_indices;  /* spec: [N_sub, spec_cols]; column 0 is also the conv slot;
                                         non-spec: the previous verify step's slots, or NULL     */
  const int32_t* num_accepted_tokens; /* spec (and acceptance-aware non-spec): [N_sub], in
                                         [1, spec_cols]                                          */
  int32_t spec_cols;                  /* spec: columns of spec_state_indices, 1..64                */
} gdn_rows;

/*
 * Bytes of device workspace gdn_mixed_batch needs for a batch without prefill rows (non_spec
 * and spec as they will be passed; either may be NULL): the fp32 post-conv q|k|v of every token,
 * spec subset first, each part rounded up to 256 bytes.  The pages stage the conv output of a
 * step in a buffer between the conv and the recurrence ("[GDN] Spec-decoding-aware attention
 * kernel", Changes: causal_conv1d pass 1 writes its outputs for the gated-delta-rule kernel);
 * keeping it in fp32 rather than the activation dtype is this library's reading (a bf16 rounding
 * of the post-conv values moves the state by more than the 1e-4 the path is held to).
 * Depends only on the host-side counts in the descriptors.  Returns 0 for invalid descriptors.
 */
size_t gdn_workspace_bytes(const gdn_layer_desc* layer, const gdn_rows* non_spec, const gdn_rows* spec);

/*
 * Extra workspace the chunked prefill needs when `rows` (a non-spec subset) holds num_prefills
 * prefill rows: one record of 123904 bytes per (64-token chunk, v-head), the chunk count bounded
 * from rows->num_tokens and num_prefills (ceil(num_tokens / 64) + num_prefills).  The pages run
 * prefill rows through a chunked kernel ("[XE2] Support MTP of QWEN model", Copilot overview:
 * chunk gated delta rule); the record holds that chunk form's state-independent terms, which
 * one kernel computes for all chunks at once and the chunk-by-chunk scan reads.  gdn_mixed_batch needs gdn_workspace_bytes() + gdn_prefill_workspace_bytes(
 * layer, non_spec, num_prefills); gdn_chunk_prefill needs gdn_prefill_workspace_bytes(layer,
 * rows, rows->num_seqs).  0 when the layer does not take the tensor-core path (see
 * gdn_chunk_prefill) or num_prefills is 0.
 */
size_t gdn_prefill_workspace_bytes(const gdn_layer_desc* layer, const gdn_rows* rows, int32_t num_prefills);

/*
 * Conv update of one subset (step (1); "[GDN] Spec-decoding-aware attention kernel",
 * Changes, causal_conv1d.hpp bullets; the review thread of "[XE2] Support MTP of QWEN model").
 * For row n with L tokens, history h = conv_pool[slot][a : a+W-1] where
 *   spec:     slot = spec_state_indices[n, 0], a = num_accepted_tokens[n] - 1 (rolled layout;
 *             per-slot layout: slot = spec_state_indices[n, num_accepted-1], a = 0);
 *   non-spec: slot = state_indices[n], a = 0 (acceptance-aware rows: a = num_accepted-1, or
 *             with the per-slot layout the history slot spec_state_indices[n, num_accepted-1]);
 * h is zero when the history slot is <= 0 or has_initial_state[n] == 0.  With H = h ++ x[token_indx[row]]:
 *   y[t][c] = SiLU(bias[c] + sum_i conv_weight[c][i] * H[t+i][c])     (fp32 arithmetic)
 * and, after every read of the slot, the slot's columns are rewritten as bit copies:
 *   spec:     columns 0 .. W-3+L  <- H[1 .. W-2+L]   (column W-2+t holds token t)
 *   non-spec: columns 0 .. W-2    <- H[L .. L+W-2]   (the last W-1 inputs)
 *   per-slot spec: columns 0 .. W-2 of spec_state_indices[n, t] <- H[t+1 .. t+W-1], t < L
 * other columns and slots are untouched; slot <= 0 is not written; L = 0 rows do nothing.
 *   x [num_global_tokens, C] act dtype (global order, gathered through token_indx);
 *   y [rows->num_tokens, C] in y_dtype (local order).
 * Size limit: one launch covers at most 65535 work units (a spec row is one unit; a non-spec
 * subset counts ceil(num_tokens / 16) + num_seqs), else GDN_ERR_SHAPE; gdn_mixed_batch counts
 * both subsets together.
 */
int gdn_conv_update(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                    const void* x, int32_t num_global_tokens, const gdn_rows* rows, void* y,
                    gdn_dtype y_dtype, uint32_t* d_status, void* stream);

/*
 * Gated delta rule over one subset, token by token (step (2); "[GDN] Spec-decoding-aware
 * attention kernel", Changes, gated_delta_rule.hpp bullet).  For v-head h of row n:
 *   load S (dv x dk) from spec_state_indices[n, num_accepted[n]-1] (spec, and acceptance-aware
 *   non-spec rows) or state_indices[n] (other non-spec rows); zeros for a non-spec row with
 *   has_initial_state[n] == 0 and whenever the slot is <= 0;
 *   per token: g = -exp(A_log[h]) softplus(a + dt_bias[h]) (softplus(x) = x for x > 20),
 *   beta = sigmoid(b), q^ = q / sqrt(|q|^2 + 1e-6) * scale, k^ = k / sqrt(|k|^2 + 1e-6),
 *   S <- e^g S (I - beta k^ k^T) + beta v k^T,  out[token_indx[i]][h] = S q^;
 *   spec rows store S after token t to spec_state_indices[n, t]; non-spec rows store S after
 *   their last token to state_indices[n]; slots <= 0 are not written.
 *   qkv [rows->num_tokens, C] post-conv activation in qkv_dtype (local order);
 *   a, b [num_global_tokens, Hv] act dtype, read at token_indx (the same index as qkv);
 *   out [num_global_tokens, Hv, dv] act dtype, written at token_indx.
 */
int gdn_recurrent_step(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                       const void* qkv, gdn_dtype qkv_dtype, const void* a, const void* b,
                       int32_t num_global_tokens, const gdn_rows* rows, void* out, uint32_t* d_status,
                       void* stream);

/*
 * The same result as gdn_recurrent_step for non-speculative rows of any length, computed
 * chunk by chunk (chunk_size tokens; 64 is the supported size) in the WY/UT form of the gated
 * delta rule on tcgen05 tensor cores ("[XE2] Support MTP of QWEN model", Copilot overview: XE2
 * chunk gated delta rule with remapped output writes).  Only the final state of each row is
 * stored.  The tensor-core path covers dk = dv = 128 with bf16 activations; other layers run the
 * token recurrence of gdn_recurrent_step (and need no workspace).
 *   rows must be non-speculative (GDN_ERR_SPEC_PAIR otherwise);
 *   workspace: at least gdn_prefill_workspace_bytes(layer, rows, rows->num_seqs) bytes,
 *   256-byte aligned (may be NULL when that is 0).
 */
int gdn_chunk_prefill(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                      const void* qkv, gdn_dtype qkv_dtype, const void* a, const void* b,
                      int32_t num_global_tokens, const gdn_rows* rows, int32_t chunk_size, void* out,
                      void* workspace, size_t workspace_bytes, uint32_t* d_status, void* stream);

/*
 * The whole path over a mixed batch (step (3); "[XE2] Support MTP of QWEN model", Copilot
 * overview and commit message; "[Bugfix] Align Qwen GDN gates with speculative tokens").
 * x [num_actual_tokens, C], a, b [num_actual_tokens, Hv] and out [num_actual_tokens, Hv, dv]
 * are in global token order.  The non-spec subset lists num_decodes rows first, then
 * num_prefills rows; the spec subset follows its own order.  Each subset gathers x, a and b
 * through its own token_indx and scatters out through it; when both subsets are non-empty
 * both token_indx must be given.  Requires
 *   non_spec->num_tokens + spec->num_tokens == num_actual_tokens (GDN_ERR_CONSERVATION) and
 *   num_decodes + num_prefills == non_spec->num_seqs (GDN_ERR_SHAPE).
 * Results equal gdn_conv_update (y in fp32) followed by gdn_recurrent_step on the spec rows and
 * the decode rows, and gdn_chunk_prefill on the prefill rows.
 * workspace: at least gdn_workspace_bytes(layer, non_spec, spec) +
 * gdn_prefill_workspace_bytes(layer, non_spec, num_prefills) bytes, 256-byte aligned.
 */
int gdn_mixed_batch(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                    const void* x, const void* a, const void* b, int32_t num_actual_tokens,
                    const gdn_rows* non_spec, int32_t num_decodes, int32_t num_prefills, const gdn_rows* spec,
                    void* out, void* workspace, size_t workspace_bytes, uint32_t* d_status, void* stream);

/*
 * gdn_mixed_batch without a workspace argument, for callers that cannot allocate device
 * memory: a plain C host or a plugin whose framework owns every device allocation and offers
 * no hook for scratch, or a serving loop that must not call cudaMalloc/cudaFree because they
 * can synchronise the device and stall other streams.  The scratch is a fixed device array of
 * GDN_STATIC_WORKSPACE_BYTES (16 MiB) inside the library:
 *   - a batch fits when gdn_workspace_bytes(layer, non_spec, spec) +
 *     gdn_prefill_workspace_bytes(layer, non_spec, num_prefills) is at most 16 MiB.  Without
 *     chunked prefill rows that is 512 tokens of an 8192-channel layer; a prefill row on the
 *     tensor-core path also needs one 123904-byte record per (64-token chunk, v-head), about
 *     3.8 MiB per chunk at 32 v-heads, so on that layer a batch holds prefill rows of a few
 *     chunks at most (one 130-token row is already refused);
 *   - it is reserved on every GPU that loads it and stays reserved until the process exits;
 *   - every call on a device shares it, so calls that may overlap on the GPU race on it;
 *   - it keeps the previous call's contents and is never cleared: no scratch element needs to
 *     start at zero, every element a call reads is written earlier by the same call;
 *   - the first call in each CUDA context (the device's primary context, normally) looks up the
 *     array's device address with that device current (cudaGetSymbolAddress); make that first
 *     call before any stream capture, and do not use this entry point across cudaDeviceReset.
 * The caller still passes inputs and outputs exactly as for gdn_mixed_batch.  Returns
 * GDN_ERR_WORKSPACE when the batch does not fit (nothing is enqueued), GDN_ERR_CUDA when the
 * address lookup fails, and otherwise what gdn_mixed_batch returns for the same arguments.
 * The paper has no counterpart to this entry point.
 */
#define GDN_STATIC_WORKSPACE_BYTES (16u << 20)
int gdn_mixed_batch_static_workspace(const gdn_layer_desc* layer, const gdn_layer_params* params,
                                     const gdn_pools* pools, const void* x, const void* a, const void* b,
                                     int32_t num_actual_tokens, const gdn_rows* non_spec, int32_t num_decodes,
                                     int32_t num_prefills, const gdn_rows* spec, void* out, uint32_t* d_status,
                                     void* stream);

/* Static text for a gdn_error value. */
const char* gdn_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
