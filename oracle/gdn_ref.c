/*
 * gdn_ref.c -- CPU oracle for the Gated DeltaNet (GDN) speculative-decoding hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may build, load or call this file.  It shares no code, header,
 * table or helper with the CUDA library, and it never reads a value the CUDA library wrote.
 *
 * What it computes is the plain definition, token by token, in double precision (the type
 * `real` below).  A second build with -DGDN_REF_FLOAT takes the same steps in float; it exists
 * only to measure the rounding noise that an fp32 implementation of the definition carries
 * (the tests compare it with the double build, never with the CUDA library):
 *
 *   1. Split / gather.  Each subset of rows (speculative or not) sees its tokens through
 *      its own token_indx: x, a and b are all read at x[token_indx[i]], a[token_indx[i]],
 *      b[token_indx[i]] -- the same index for all three ("[Bugfix] Align Qwen GDN gates
 *      with speculative tokens", Purpose), and outputs land back at out[token_indx[i]]
 *      ("[XE2] Support MTP of QWEN model", Copilot overview: token-index remapping).
 *
 *   2. Causal conv1d with the speculative column-0 contract ("[GDN] Spec-decoding-aware
 *      attention kernel", Problem and Changes: pass 1 / pass 2; "[XE2] Support MTP", review
 *      thread on FLA's rolled history at slot 0).  The conv slot of a speculative row is
 *      spec_state_indices[n, 0]; its history is read at column offset num_accepted-1;
 *      the slot is rewritten only after every read of it.
 *
 *   3. Gates, norms and the gated delta rule, per (token, v-head):
 *        g    = -exp(A_log[h]) * softplus(a + dt_bias[h])
 *        beta = sigmoid(b)
 *        q^   = q / sqrt(sum q^2 + eps) * scale,   k^ = k / sqrt(sum k^2 + eps)
 *        S_t  = e^g S_{t-1} (I - beta k^ k^T) + beta v k^T,     o_t = S_t q^
 *      with the state loaded from spec_state_indices[n, num_accepted[n]-1] and stored after
 *      every token t to spec_state_indices[n, t]; a slot <= 0 means "no prior state" on
 *      load and "no store" on store ("[GDN] Spec-decoding-aware attention kernel",
 *      Changes, gated_delta_rule.hpp bullet).  Non-speculative rows load from and store
 *      (after their last token) to state_indices[n].
 *
 * Readings of points the pages leave open (each is also listed in the design notes):
 *   - softplus(x) = x for x > 20, else log1p(exp(x)).
 *   - eps = 1e-6 inside the square root of the L2 norm, the same for q and k.
 *   - v-head h uses k-head h / (Hv/Hk).
 *   - The state of one head is stored [dv][dk], dk fastest; the SSM pool is [P, Hv, dv, dk].
 *   - The conv weight w[c][W-1] multiplies the current token; the bias is optional.
 *   - The packed channels are q (Hk*dk) | k (Hk*dk) | v (Hv*dv), head-major.
 *   - Post-conv q|k|v stay in double here (the kernels keep them in fp32); they are never
 *     rounded to the activation type.
 *   - Spec row of L tokens (L <= spec_cols): the new history H[1 : W-1+L] goes to columns
 *     0 .. W-3+L; a non-spec row writes its last W-1 inputs H[L : L+W-1] to columns 0..W-2.
 *     Other columns stay untouched.  A row with L = 0 reads and writes nothing.
 *   - Alternative spec conv layout (conv_layout = 1): history from column 0 of
 *     spec_state_indices[n, num_accepted-1]; after token t the last W-1 inputs go to columns
 *     0..W-2 of spec_state_indices[n, t].
 *   - Alternative x layout (qkv_layout = 1): per k-head groups [q_g | k_g | v of group g];
 *     weights, bias, the conv pool and the post-conv q|k|v stay in packed order.
 *   - A non-spec row given num_accepted_tokens and spec_state_indices continues from its
 *     previous verify step's accepted state (see acceptance_aware below).
 *   - Outputs are rounded to the activation type (fp32: round to nearest; bf16: round to
 *     nearest fp32 first, then round-to-nearest-even to bf16).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef GDN_REF_FLOAT
typedef float real;
#define R_EXP expf
#define R_LOG1P log1pf
#define R_SQRT sqrtf
#else
typedef double real;
#define R_EXP exp
#define R_LOG1P log1p
#define R_SQRT sqrt
#endif

typedef struct {
  int32_t num_k_heads, num_v_heads, head_k_dim, head_v_dim;
  int32_t conv_width, conv_state_len;
  int32_t act_is_bf16; /* 1: x, a, b, out, conv pool/weights are bf16; 0: fp32 */
  double scale;        /* multiplies q^; the caller passes 1/sqrt(dk) by default */
  double norm_eps;     /* epsilon inside the L2-norm square root */
  int32_t qkv_layout;  /* channel order of x: 0 packed q|k|v; 1 per k-head [q_g | k_g | v of group g] */
  int32_t conv_layout; /* spec conv state: 0 rolled history at column 0; 1 one snapshot per spec slot */
} ref_layer;

typedef struct {
  int32_t num_seqs, num_tokens;
  const int32_t* query_start_loc;     /* [num_seqs+1], local token offsets */
  const int32_t* token_indx;          /* [num_tokens] global token of each local one; NULL = identity */
  const int32_t* state_indices;       /* non-spec rows: [num_seqs] */
  const int32_t* has_initial_state;   /* non-spec rows: [num_seqs] or NULL (= all 1) */
  const int32_t* spec_state_indices;  /* spec rows: [num_seqs, spec_cols] */
  const int32_t* num_accepted_tokens; /* spec rows: [num_seqs] */
  /* Non-spec rows may carry spec_state_indices and num_accepted_tokens too: the slots and the
   * acceptance of the row's previous verify step (acceptance-aware rows, below). */
  int32_t spec_cols;
  int32_t is_spec;
} ref_rows;

/* ---------------------------------------------------------------- element access */

static double act_get(const void* base, int64_t i, int bf16) {
  if (bf16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
  }
  return (double)((const float*)base)[i];
}

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u); /* quiet NaN */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb; /* round half to even on the 16 dropped bits */
  return (uint16_t)(u >> 16);
}

static void act_put(void* base, int64_t i, int bf16, double v) {
  float f = (float)v;
  if (bf16)
    ((uint16_t*)base)[i] = f32_to_bf16_rne(f);
  else
    ((float*)base)[i] = f;
}

static void act_copy(void* dst, int64_t di, const void* src, int64_t si, int bf16) {
  if (bf16)
    ((uint16_t*)dst)[di] = ((const uint16_t*)src)[si];
  else
    ((float*)dst)[di] = ((const float*)src)[si];
}

static int32_t global_token(const ref_rows* r, int32_t i) { return r->token_indx ? r->token_indx[i] : i; }

static real softplus(real x) { return x > (real)20 ? x : R_LOG1P(R_EXP(x)); }
static real sigmoid(real x) { return (real)1 / ((real)1 + R_EXP(-x)); }
static real silu(real x) { return x / ((real)1 + R_EXP(-x)); }

/* ----------------------------------------------------------------------- row checks */

/* Returns 0 when the row's metadata is usable, -1 otherwise (the oracle does not guess). */
static int check_row(const ref_rows* r, int32_t n, int64_t num_slots, int32_t num_global) {
  int32_t bos = r->query_start_loc[n], eos = r->query_start_loc[n + 1];
  if (bos < 0 || eos < bos || eos > r->num_tokens) return -1;
  for (int32_t i = bos; i < eos; ++i) {
    int32_t gt = global_token(r, i);
    if (gt < 0 || gt >= num_global) return -1;
  }
  if (r->is_spec) {
    if (eos - bos > r->spec_cols) return -1;
    int32_t na = r->num_accepted_tokens[n];
    if (eos > bos && (na < 1 || na > r->spec_cols)) return -1;
    for (int32_t j = 0; j < r->spec_cols; ++j)
      if (r->spec_state_indices[(int64_t)n * r->spec_cols + j] >= num_slots) return -1;
  } else {
    if (r->state_indices[n] >= num_slots) return -1;
    if (r->num_accepted_tokens) {
      int32_t na = r->num_accepted_tokens[n];
      if (eos > bos && (na < 1 || na > r->spec_cols)) return -1;
      for (int32_t j = 0; j < r->spec_cols; ++j)
        if (r->spec_state_indices[(int64_t)n * r->spec_cols + j] >= num_slots) return -1;
    }
  }
  return 0;
}

/* A non-spec row that carries its previous verify step's acceptance: a verify row cut to a
 * prefix by the batch budget and scheduled as a plain row ("[Bugfix] Align Qwen GDN gates with
 * speculative tokens", the second mechanism in the reachability comment).  Its history and
 * prior state are where that step's accepted tokens left them: conv history at column
 * offset num_accepted-1 of state_indices[n] (rolled layout) or in the snapshot slot
 * spec_state_indices[n, num_accepted-1] (per-slot layout); SSM state from
 * spec_state_indices[n, num_accepted-1].  Writes are those of any non-spec row. */
static int acceptance_aware(const ref_rows* r) { return !r->is_spec && r->num_accepted_tokens != NULL; }

/* ------------------------------------------------------------------ causal conv1d */

/* Position in x of packed channel c (q | k | v blocks, head-major).  With the per-k-head
 * layout ("[GDN] Spec-decoding-aware attention kernel", Test Plan: reorder_input=False, the
 * projection order used in production Qwen3-Next traffic) x holds, for each k-head g in turn,
 * q_g (dk), k_g (dk) and the dv-channel v of the G = Hv/Hk v-heads of group g. */
static int64_t x_channel(const ref_layer* L, int64_t c) {
  if (!L->qkv_layout) return c;
  const int64_t dk = L->head_k_dim, dv = L->head_v_dim, Hk = L->num_k_heads, G = L->num_v_heads / Hk;
  const int64_t group = 2 * dk + G * dv;
  if (c < Hk * dk) return (c / dk) * group + c % dk;                    /* q of k-head c/dk */
  if (c < 2 * Hk * dk) return ((c - Hk * dk) / dk) * group + dk + c % dk; /* k */
  const int64_t vc = c - 2 * Hk * dk, hv = vc / dv;                     /* v of v-head hv */
  return (hv / G) * group + 2 * dk + (hv % G) * dv + vc % dv;
}

/*
 * Conv update of one subset.  conv_pool [P, state_len, C] (act type) is read and written;
 * y [num_tokens, C] (real, local token order) receives SiLU(conv).
 */
int gdn_ref_conv(const ref_layer* L, const void* conv_w, const void* conv_b, void* conv_pool,
                 int64_t num_slots, const void* x, int32_t num_global, const ref_rows* rows, real* y) {
  const int bf = L->act_is_bf16;
  const int32_t W = L->conv_width, SL = L->conv_state_len;
  const int64_t C = 2LL * L->num_k_heads * L->head_k_dim + (int64_t)L->num_v_heads * L->head_v_dim;
  for (int32_t n = 0; n < rows->num_seqs; ++n)
    if (check_row(rows, n, num_slots, num_global)) return -1;

  for (int32_t n = 0; n < rows->num_seqs; ++n) {
    const int32_t bos = rows->query_start_loc[n], len = rows->query_start_loc[n + 1] - bos;
    if (len == 0) continue;
    /* slot: the row's own conv slot (read and rolled back); rd: where the history is read */
    int32_t slot, rd, anchor, read_prior;
    const int per_slot = rows->is_spec && L->conv_layout == 1;
    const int aware = acceptance_aware(rows);
    if (per_slot) {
      /* one snapshot per spec slot ("[XE2] Support MTP of QWEN model", review thread): the
       * history is the snapshot taken after the last accepted token */
      slot = rd = rows->spec_state_indices[(int64_t)n * rows->spec_cols + rows->num_accepted_tokens[n] - 1];
      anchor = 0;
      read_prior = rd > 0;
    } else if (rows->is_spec) {
      slot = rd = rows->spec_state_indices[(int64_t)n * rows->spec_cols]; /* column 0 of the row */
      anchor = rows->num_accepted_tokens[n] - 1;
      read_prior = rd > 0;
    } else {
      slot = rd = rows->state_indices[n];
      anchor = 0;
      if (aware) {
        const int32_t a = rows->num_accepted_tokens[n] - 1;
        if (L->conv_layout == 1) rd = rows->spec_state_indices[(int64_t)n * rows->spec_cols + a];
        else anchor = a;
      }
      read_prior = rd > 0 && (rows->has_initial_state ? rows->has_initial_state[n] != 0 : 1);
    }
    /* H = (W-1 history columns) ++ (the row's len inputs), kept both as exact values and as
     * the raw stored elements so that the slot write is a bit copy. */
    const int32_t hl = W - 1 + len;
    real* H = (real*)malloc(sizeof(real) * (size_t)hl * (size_t)C);
    void* Hraw = malloc((size_t)hl * (size_t)C * (bf ? 2 : 4));
    if (!H || !Hraw) { free(H); free(Hraw); return -2; }
    for (int32_t i = 0; i < W - 1; ++i)
      for (int64_t c = 0; c < C; ++c) {
        if (read_prior) {
          int64_t src = ((int64_t)rd * SL + anchor + i) * C + c;
          H[i * C + c] = (real)act_get(conv_pool, src, bf);
          act_copy(Hraw, i * C + c, conv_pool, src, bf);
        } else {
          H[i * C + c] = (real)0;
          act_put(Hraw, i * C + c, bf, 0.0);
        }
      }
    for (int32_t t = 0; t < len; ++t) {
      int64_t gt = global_token(rows, bos + t);
      for (int64_t c = 0; c < C; ++c) {
        H[(W - 1 + t) * C + c] = (real)act_get(x, gt * C + x_channel(L, c), bf);
        act_copy(Hraw, (W - 1 + t) * C + c, x, gt * C + x_channel(L, c), bf);
      }
    }
    /* y_t[c] = SiLU(bias[c] + sum_i w[c][i] * H[t+i][c]) */
    for (int32_t t = 0; t < len; ++t)
      for (int64_t c = 0; c < C; ++c) {
        real acc = conv_b ? (real)act_get(conv_b, c, bf) : (real)0;
        for (int32_t i = 0; i < W; ++i) acc += (real)act_get(conv_w, c * W + i, bf) * H[(t + i) * C + c];
        y[(int64_t)(bos + t) * C + c] = silu(acc);
      }
    /* Per-slot snapshots: after token t, its last W-1 inputs H[t+1 .. t+W-1] go to
     * spec_state_indices[n, t] (slots <= 0 skipped). */
    if (per_slot) {
      for (int32_t t = 0; t < len; ++t) {
        const int32_t ss = rows->spec_state_indices[(int64_t)n * rows->spec_cols + t];
        if (ss <= 0) continue;
        for (int32_t j = 0; j < W - 1; ++j)
          for (int64_t c = 0; c < C; ++c)
            act_copy(conv_pool, ((int64_t)ss * SL + j) * C + c, Hraw, (int64_t)(t + 1 + j) * C + c, bf);
      }
    } else if (slot > 0) {
      /* Rolled history back into the slot, after every read of it. */
      int32_t off = rows->is_spec ? 1 : len;
      int32_t ncols = rows->is_spec ? W - 2 + len : W - 1;
      for (int32_t j = 0; j < ncols; ++j)
        for (int64_t c = 0; c < C; ++c)
          act_copy(conv_pool, ((int64_t)slot * SL + j) * C + c, Hraw, (int64_t)(off + j) * C + c, bf);
    }
    free(H);
    free(Hraw);
  }
  return 0;
}

/* -------------------------------------------------------------- gated delta rule */

typedef struct {
  const ref_layer* L;
  const float* A_log;
  const float* dt_bias;
  float* ssm_pool;
  const real* qkv;
  const void* a;
  const void* b;
  const ref_rows* rows;
  void* out;
  real* out_f64;
} rec_job;

/* One (row, v-head) of one subset: load, token loop, stores. */
static void recurrent_row_head(const rec_job* J, int32_t n, int32_t h) {
  const ref_layer* L = J->L;
  const ref_rows* r = J->rows;
  const int bf = L->act_is_bf16;
  const int32_t Hk = L->num_k_heads, Hv = L->num_v_heads, dk = L->head_k_dim, dv = L->head_v_dim;
  const int64_t C = 2LL * Hk * dk + (int64_t)Hv * dv;
  const int32_t kh = h / (Hv / Hk);
  const int32_t bos = r->query_start_loc[n], len = r->query_start_loc[n + 1] - bos;
  if (len == 0) return;

  int32_t load_slot;
  int read_prior;
  if (r->is_spec) {
    load_slot = r->spec_state_indices[(int64_t)n * r->spec_cols + r->num_accepted_tokens[n] - 1];
    read_prior = load_slot > 0;
  } else {
    load_slot = acceptance_aware(r)
                    ? r->spec_state_indices[(int64_t)n * r->spec_cols + r->num_accepted_tokens[n] - 1]
                    : r->state_indices[n];
    read_prior = load_slot > 0 && (r->has_initial_state ? r->has_initial_state[n] != 0 : 1);
  }
  const int64_t head_elems = (int64_t)dv * dk;
  real* S = (real*)calloc((size_t)head_elems, sizeof(real));
  real* qn = (real*)malloc(sizeof(real) * (size_t)dk);
  real* kn = (real*)malloc(sizeof(real) * (size_t)dk);
  if (!S || !qn || !kn) { free(S); free(qn); free(kn); return; }
  if (read_prior) {
    const float* src = J->ssm_pool + ((int64_t)load_slot * Hv + h) * head_elems;
    for (int64_t e = 0; e < head_elems; ++e) S[e] = (real)src[e];
  }

  for (int32_t t = 0; t < len; ++t) {
    const int64_t i = bos + t;
    const int64_t gt = global_token(r, (int32_t)i);
    const real* q = J->qkv + i * C + (int64_t)kh * dk;
    const real* k = J->qkv + i * C + (int64_t)Hk * dk + (int64_t)kh * dk;
    const real* v = J->qkv + i * C + 2LL * Hk * dk + (int64_t)h * dv;
    real sq = (real)0, sk = (real)0;
    for (int32_t c = 0; c < dk; ++c) { sq += q[c] * q[c]; sk += k[c] * k[c]; }
    const real rq = (real)1 / R_SQRT(sq + (real)L->norm_eps), rk = (real)1 / R_SQRT(sk + (real)L->norm_eps);
    for (int32_t c = 0; c < dk; ++c) { qn[c] = q[c] * rq * (real)L->scale; kn[c] = k[c] * rk; }

    const real av = (real)act_get(J->a, gt * Hv + h, bf), bv = (real)act_get(J->b, gt * Hv + h, bf);
    const real g = -R_EXP((real)J->A_log[h]) * softplus(av + (real)J->dt_bias[h]);
    const real beta = sigmoid(bv);
    const real decay = R_EXP(g);

    /* S <- e^g S ;  u = S k^ ;  S <- S + beta (v - u) k^T ;  o = S q^ */
    for (int64_t e = 0; e < head_elems; ++e) S[e] *= decay;
    for (int32_t row = 0; row < dv; ++row) {
      real* s = S + (int64_t)row * dk;
      real u = (real)0;
      for (int32_t c = 0; c < dk; ++c) u += s[c] * kn[c];
      const real delta = beta * (v[row] - u);
      for (int32_t c = 0; c < dk; ++c) s[c] += delta * kn[c];
      real o = (real)0;
      for (int32_t c = 0; c < dk; ++c) o += s[c] * qn[c];
      act_put(J->out, (gt * Hv + h) * dv + row, bf, (double)o);
      if (J->out_f64) J->out_f64[(gt * Hv + h) * dv + row] = o;
    }
    if (r->is_spec) {
      const int32_t store_slot = r->spec_state_indices[(int64_t)n * r->spec_cols + t];
      if (store_slot > 0) {
        float* dst = J->ssm_pool + ((int64_t)store_slot * Hv + h) * head_elems;
        for (int64_t e = 0; e < head_elems; ++e) dst[e] = (float)S[e];
      }
    }
  }
  if (!r->is_spec && r->state_indices[n] > 0) {
    float* dst = J->ssm_pool + ((int64_t)r->state_indices[n] * Hv + h) * head_elems;
    for (int64_t e = 0; e < head_elems; ++e) dst[e] = (float)S[e];
  }
  free(S);
  free(qn);
  free(kn);
}

typedef struct {
  const rec_job* job;
  int32_t h0, h1;
  int32_t* next; /* shared work counter over (row, head) items */
} rec_worker;

static void* rec_worker_main(void* arg) {
  rec_worker* w = (rec_worker*)arg;
  const int32_t nh = w->h1 - w->h0;
  const int32_t total = w->job->rows->num_seqs * nh;
  for (;;) {
    int32_t item = __atomic_fetch_add(w->next, 1, __ATOMIC_RELAXED);
    if (item >= total) break;
    recurrent_row_head(w->job, item / nh, w->h0 + item % nh);
  }
  return NULL;
}

/*
 * Gated delta rule over one subset, for v-heads [h0, h1) (h1 <= 0 means all heads).
 * qkv [num_tokens, C] is the post-conv activation in local token order (real); a, b
 * [num_global, Hv] and out [num_global, Hv, dv] are in global token order (act type);
 * out_f64 (optional) receives the unrounded outputs.  Work is split over (row, head)
 * across nthreads POSIX threads; rows must use distinct slots.
 */
int gdn_ref_recurrent(const ref_layer* L, const float* A_log, const float* dt_bias, float* ssm_pool,
                      int64_t num_slots, const real* qkv, const void* a, const void* b, int32_t num_global,
                      const ref_rows* rows, void* out, real* out_f64, int32_t h0, int32_t h1,
                      int32_t nthreads) {
  if (L->num_v_heads % L->num_k_heads) return -1;
  for (int32_t n = 0; n < rows->num_seqs; ++n)
    if (check_row(rows, n, num_slots, num_global)) return -1;
  if (h1 <= 0) { h0 = 0; h1 = L->num_v_heads; }
  rec_job job = {L, A_log, dt_bias, ssm_pool, qkv, a, b, rows, out, out_f64};
  int32_t next = 0;
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  rec_worker* wk = (rec_worker*)malloc(sizeof(rec_worker) * (size_t)nthreads);
  char* live = (char*)calloc((size_t)nthreads, 1);
  if (!th || !wk || !live) { free(th); free(wk); free(live); return -2; }
  for (int32_t i = 0; i < nthreads; ++i) {
    wk[i].job = &job; wk[i].h0 = h0; wk[i].h1 = h1; wk[i].next = &next;
    /* the calling thread is worker 0; a thread that fails to start leaves its share to the others */
    if (i > 0) live[i] = pthread_create(&th[i], NULL, rec_worker_main, &wk[i]) == 0;
  }
  rec_worker_main(&wk[0]);
  for (int32_t i = 1; i < nthreads; ++i)
    if (live[i]) pthread_join(th[i], NULL);
  free(th);
  free(wk);
  free(live);
  return 0;
}
