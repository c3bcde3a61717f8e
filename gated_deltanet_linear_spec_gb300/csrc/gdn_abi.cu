// gdn_abi.cu -- the C entry points: host-side validation, workspace layout and launches.
//
// Validation follows the pages' interface rules: every optional tensor is checked before use
// ("[XE2] Support MTP of QWEN model", the review notes on unchecked optionals), the spec pair
// spec_state_indices / num_accepted_tokens comes together ("[GDN] Spec-decoding-aware attention
// kernel", Changes, gdn_attn_interface.cpp bullet), and a mixed batch only has to conserve
// tokens, not be rectangular ("[XE2] Support MTP of QWEN model", commit message).  Nothing here
// reads device memory, so every call is stream-ordered and can be captured in a CUDA graph.
#include <nvtx3/nvToolsExt.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "gdn_internal.cuh"

using namespace gdn;

namespace {

constexpr int kMaxSpecCols = 64;  // a spec row is one conv work unit of kConvSeg tokens

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

int64_t channels(const gdn_layer_desc* d) {
  return 2LL * d->num_k_heads * d->head_k_dim + (int64_t)d->num_v_heads * d->head_v_dim;
}

int check_layer(const gdn_layer_desc* d) {
  if (!d) return GDN_ERR_NULL_ARG;
  if (d->act_dtype != GDN_F32 && d->act_dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (d->num_k_heads <= 0 || d->num_v_heads <= 0 || d->num_v_heads % d->num_k_heads) return GDN_ERR_SHAPE;
  if (d->num_v_heads > 65535) return GDN_ERR_SHAPE;
  const int dk = d->head_k_dim;
  if (dk != 16 && dk != 32 && dk != 64 && dk != 128) return GDN_ERR_SHAPE;
  if (d->head_v_dim <= 0 || d->head_v_dim % 16 || d->head_v_dim > 256) return GDN_ERR_SHAPE;
  if (d->conv_width < 2 || d->conv_width > 4) return GDN_ERR_SHAPE;
  if (d->conv_state_len < d->conv_width - 1) return GDN_ERR_SHAPE;
  if (d->qkv_layout != GDN_QKV_PACKED && d->qkv_layout != GDN_QKV_PER_KHEAD) return GDN_ERR_SHAPE;
  if (d->conv_layout != GDN_CONV_ROLLED && d->conv_layout != GDN_CONV_PER_SLOT) return GDN_ERR_SHAPE;
  return GDN_OK;
}

int check_params(const gdn_layer_params* p, bool need_conv) {
  if (!p || !p->A_log || !p->dt_bias) return GDN_ERR_NULL_ARG;
  if (need_conv && !p->conv_weight) return GDN_ERR_NULL_ARG;
  if (need_conv && (!aligned16(p->conv_weight) || !aligned16(p->conv_bias))) return GDN_ERR_ALIGN;
  return GDN_OK;
}

int check_pools(const gdn_pools* p, bool need_conv) {
  if (!p || !p->ssm_pool || (need_conv && !p->conv_pool)) return GDN_ERR_NULL_ARG;
  if (p->num_slots <= 0) return GDN_ERR_SHAPE;
  if (!aligned16(p->ssm_pool) || (need_conv && !aligned16(p->conv_pool))) return GDN_ERR_ALIGN;
  return GDN_OK;
}

// A subset: shapes, pointer presence, the spec pair.  `rows` may be NULL (empty subset).
int check_rows(const gdn_layer_desc* d, const gdn_rows* r) {
  if (!r) return GDN_OK;
  if (r->num_seqs < 0 || r->num_tokens < 0 || r->num_seqs > 65535) return GDN_ERR_SHAPE;
  if (r->num_seqs == 0) return r->num_tokens == 0 ? GDN_OK : GDN_ERR_SHAPE;
  if (!r->query_start_loc) return GDN_ERR_NULL_ARG;
  const bool has_ssi = r->spec_state_indices != nullptr, has_na = r->num_accepted_tokens != nullptr;
  if (has_ssi != has_na) return GDN_ERR_SPEC_PAIR;
  if (has_ssi) {
    if (r->spec_cols < 1 || r->spec_cols > kMaxSpecCols) return GDN_ERR_SHAPE;
    if (d->conv_layout == GDN_CONV_ROLLED && r->spec_cols > d->conv_state_len - d->conv_width + 2)
      return GDN_ERR_SHAPE;
  } else if (!r->state_indices) {
    return GDN_ERR_NULL_ARG;
  }
  return GDN_OK;
}

// Spec rows have spec slots and no state_indices; a non-spec subset may carry the spec pair
// as the acceptance of its rows' previous verify step.
bool is_spec(const gdn_rows* r) { return r && r->spec_state_indices != nullptr && r->state_indices == nullptr; }
int nseq(const gdn_rows* r) { return r ? r->num_seqs : 0; }
int ntok(const gdn_rows* r) { return r ? r->num_tokens : 0; }

// Conv work units of one subset: one per spec row; an upper bound for non-spec rows.
int conv_units(const gdn_rows* r) {
  if (!r || r->num_seqs == 0) return 0;
  if (is_spec(r)) return r->num_seqs;
  return (r->num_tokens + kConvSegNS - 1) / kConvSegNS + r->num_seqs;
}

// Chunk units of the prefill rows: an upper bound from the subset's token count.
int prefill_units(const gdn_rows* r, int32_t num_prefills) {
  return (r->num_tokens + kPrefillChunk - 1) / kPrefillChunk + num_prefills;
}

PrefillLaunch prefill_args(const gdn_layer_desc* d, const gdn_layer_params* prm, const gdn_pools* pools,
                           const void* qkv, const void* a, const void* b, void* out, int32_t num_global,
                           const gdn_rows* rows, int32_t first_row, int32_t num_rows, void* ws, uint32_t* status) {
  PrefillLaunch p{};
  p.qkv = qkv;
  p.a = a;
  p.b = b;
  p.out = out;
  p.num_global = num_global;
  p.A_log = prm->A_log;
  p.dt_bias = prm->dt_bias;
  p.ssm_pool = pools->ssm_pool;
  p.num_slots = pools->num_slots;
  p.Hk = d->num_k_heads;
  p.Hv = d->num_v_heads;
  p.C = (int32_t)channels(d);
  p.scale = d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)d->head_k_dim);
  p.rows = rows_dev(rows);
  p.first_row = first_row;
  p.num_rows = num_rows;
  p.ws = static_cast<uint8_t*>(ws);
  p.status = status;
  return p;
}

float resolve_scale(const gdn_layer_desc* d) {
  return d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)d->head_k_dim);
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

ConvLaunch conv_args(const gdn_layer_desc* d, const gdn_layer_params* prm, const gdn_pools* pools,
                     const void* x, int32_t num_global, uint32_t* status) {
  ConvLaunch c{};
  c.x = x;
  c.num_global = num_global;
  c.w = prm->conv_weight;
  c.bias = prm->conv_bias;
  c.conv_pool = pools->conv_pool;
  c.num_slots = pools->num_slots;
  c.state_len = d->conv_state_len;
  c.C = (int32_t)channels(d);
  c.Hk = d->num_k_heads;
  c.dk = d->head_k_dim;
  c.Hv = d->num_v_heads;
  c.dv = d->head_v_dim;
  c.qkv_layout = d->qkv_layout;
  c.conv_layout = d->conv_layout;
  c.status = status;
  return c;
}

RecLaunch rec_args(const gdn_layer_desc* d, const gdn_layer_params* prm, const gdn_pools* pools, const void* a,
                   const void* b, void* out, int32_t num_global, uint32_t* status) {
  RecLaunch r{};
  r.a = a;
  r.b = b;
  r.out = out;
  r.num_global = num_global;
  r.A_log = prm->A_log;
  r.dt_bias = prm->dt_bias;
  r.ssm_pool = pools->ssm_pool;
  r.num_slots = pools->num_slots;
  r.Hk = d->num_k_heads;
  r.Hv = d->num_v_heads;
  r.dk = d->head_k_dim;
  r.dv = d->head_v_dim;
  r.C = (int32_t)channels(d);
  r.scale = resolve_scale(d);
  r.status = status;
  return r;
}

}  // namespace

// A named NVTX range around each compute entry point (shows in Nsight timelines; without a tool
// attached the push and pop are no-ops).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

extern "C" {

const char* gdn_status_string(int code) {
  switch (code) {
    case GDN_OK: return "ok";
    case GDN_ERR_NULL_ARG: return "a required pointer is NULL";
    case GDN_ERR_SPEC_PAIR: return "spec_state_indices and num_accepted_tokens must be given together";
    case GDN_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case GDN_ERR_CONSERVATION: return "non-spec tokens + spec tokens != num_actual_tokens";
    case GDN_ERR_WORKSPACE: return "workspace missing or too small";
    case GDN_ERR_DTYPE: return "unknown dtype";
    case GDN_ERR_CUDA: return "kernel launch failed";
    case GDN_ERR_ALIGN: return "pointer not 16-byte aligned";
    default: return "unknown gdn status";
  }
}

size_t gdn_prefill_workspace_bytes(const gdn_layer_desc* layer, const gdn_rows* rows, int32_t num_prefills) {
  if (check_layer(layer) || check_rows(layer, rows) || !rows || num_prefills <= 0) return 0;
  if (!prefill_tc_supported(layer)) return 0;
  return (size_t)prefill_units(rows, num_prefills) * (size_t)layer->num_v_heads * kRecBytes;
}

size_t gdn_workspace_bytes(const gdn_layer_desc* layer, const gdn_rows* non_spec, const gdn_rows* spec) {
  if (check_layer(layer) || check_rows(layer, non_spec) || check_rows(layer, spec)) return 0;
  const size_t C = (size_t)channels(layer);
  // fp32 post-conv q|k|v of every local token, spec subset first.
  return round256((size_t)ntok(spec) * C * 4) + round256((size_t)ntok(non_spec) * C * 4);
}

int gdn_conv_update(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                    const void* x, int32_t num_global_tokens, const gdn_rows* rows, void* y, gdn_dtype y_dtype,
                    uint32_t* d_status, void* stream) {
  NvtxRange nvtx_range("gdn_conv_update");
  int rc;
  if ((rc = check_layer(layer)) || (rc = check_params(params, true)) || (rc = check_pools(pools, true)) ||
      (rc = check_rows(layer, rows)))
    return rc;
  if (!rows) return GDN_ERR_NULL_ARG;
  if (y_dtype != GDN_F32 && y_dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (rows->num_seqs == 0) return GDN_OK;
  if (!x || !y) return GDN_ERR_NULL_ARG;
  if (!aligned16(x) || !aligned16(y)) return GDN_ERR_ALIGN;
  if (num_global_tokens < 0) return GDN_ERR_SHAPE;
  if (!rows->token_indx && rows->num_tokens > num_global_tokens) return GDN_ERR_SHAPE;
  ConvLaunch c = conv_args(layer, params, pools, x, num_global_tokens, d_status);
  c.sub[0] = rows_dev(rows);
  c.y[0] = y;
  c.units0 = conv_units(rows);
  if (c.units0 > 65535) return GDN_ERR_SHAPE;
  return cuda_rc(launch_conv(c, layer->conv_width, layer->act_dtype, y_dtype, c.units0, (cudaStream_t)stream));
}

int gdn_recurrent_step(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                       const void* qkv, gdn_dtype qkv_dtype, const void* a, const void* b, int32_t num_global_tokens,
                       const gdn_rows* rows, void* out, uint32_t* d_status, void* stream) {
  NvtxRange nvtx_range("gdn_recurrent_step");
  int rc;
  if ((rc = check_layer(layer)) || (rc = check_params(params, false)) || (rc = check_pools(pools, false)) ||
      (rc = check_rows(layer, rows)))
    return rc;
  if (!rows) return GDN_ERR_NULL_ARG;
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (rows->num_seqs == 0) return GDN_OK;
  if (!qkv || !a || !b || !out) return GDN_ERR_NULL_ARG;
  if (!aligned16(qkv)) return GDN_ERR_ALIGN;
  if (num_global_tokens < 0) return GDN_ERR_SHAPE;
  if (!rows->token_indx && rows->num_tokens > num_global_tokens) return GDN_ERR_SHAPE;
  RecLaunch r = rec_args(layer, params, pools, a, b, out, num_global_tokens, d_status);
  r.sub[0] = rows_dev(rows);
  r.qkv[0] = qkv;
  r.rows0 = rows->num_seqs;
  return cuda_rc(launch_recurrent(r, layer->act_dtype, qkv_dtype, rows->num_seqs, false, (cudaStream_t)stream));
}

int gdn_chunk_prefill(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                      const void* qkv, gdn_dtype qkv_dtype, const void* a, const void* b, int32_t num_global_tokens,
                      const gdn_rows* rows, int32_t chunk_size, void* out, void* workspace, size_t workspace_bytes,
                      uint32_t* d_status, void* stream) {
  NvtxRange nvtx_range("gdn_chunk_prefill");
  int rc;
  if ((rc = check_layer(layer)) || (rc = check_params(params, false)) || (rc = check_pools(pools, false)) ||
      (rc = check_rows(layer, rows)))
    return rc;
  if (!rows) return GDN_ERR_NULL_ARG;
  if (is_spec(rows)) return GDN_ERR_SPEC_PAIR;
  if (chunk_size != kPrefillChunk) return GDN_ERR_SHAPE;
  if (!prefill_tc_supported(layer))
    return gdn_recurrent_step(layer, params, pools, qkv, qkv_dtype, a, b, num_global_tokens, rows, out, d_status,
                              stream);
  if (qkv_dtype != GDN_F32 && qkv_dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (rows->num_seqs == 0) return GDN_OK;
  if (!qkv || !a || !b || !out) return GDN_ERR_NULL_ARG;
  if (!aligned16(qkv) || !aligned16(out)) return GDN_ERR_ALIGN;  // the scan writes 16-byte output vectors
  if (num_global_tokens < 0) return GDN_ERR_SHAPE;
  if (!rows->token_indx && rows->num_tokens > num_global_tokens) return GDN_ERR_SHAPE;
  const size_t need = gdn_prefill_workspace_bytes(layer, rows, rows->num_seqs);
  if (!workspace || workspace_bytes < need) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGN;
  const int units = prefill_units(rows, rows->num_seqs);
  if ((int64_t)units * layer->num_v_heads > (int64_t)INT32_MAX) return GDN_ERR_SHAPE;
  PrefillLaunch p = prefill_args(layer, params, pools, qkv, a, b, out, num_global_tokens, rows, 0, rows->num_seqs,
                                 workspace, d_status);
  return cuda_rc(launch_prefill(p, qkv_dtype, units, (cudaStream_t)stream));
}

int gdn_mixed_batch(const gdn_layer_desc* layer, const gdn_layer_params* params, const gdn_pools* pools,
                    const void* x, const void* a, const void* b, int32_t num_actual_tokens, const gdn_rows* non_spec,
                    int32_t num_decodes, int32_t num_prefills, const gdn_rows* spec, void* out, void* workspace,
                    size_t workspace_bytes, uint32_t* d_status, void* stream) {
  NvtxRange nvtx_range("gdn_mixed_batch");
  int rc;
  if ((rc = check_layer(layer)) || (rc = check_params(params, true)) || (rc = check_pools(pools, true)) ||
      (rc = check_rows(layer, non_spec)) || (rc = check_rows(layer, spec)))
    return rc;
  if (non_spec && is_spec(non_spec)) return GDN_ERR_SPEC_PAIR;
  if (spec && spec->num_seqs > 0 && !is_spec(spec)) return GDN_ERR_SPEC_PAIR;
  if (num_decodes < 0 || num_prefills < 0 || num_decodes + num_prefills != nseq(non_spec)) return GDN_ERR_SHAPE;
  if (ntok(non_spec) + ntok(spec) != num_actual_tokens) return GDN_ERR_CONSERVATION;
  const bool both = nseq(non_spec) > 0 && nseq(spec) > 0;
  if (both && (!non_spec->token_indx || !spec->token_indx)) return GDN_ERR_NULL_ARG;
  if (num_actual_tokens == 0) return GDN_OK;
  if (!x || !a || !b || !out) return GDN_ERR_NULL_ARG;
  if (!aligned16(x)) return GDN_ERR_ALIGN;
  // prefill rows take the tensor-core chunked path when the layer allows it
  const bool chunked = num_prefills > 0 && prefill_tc_supported(layer);
  if (chunked && !aligned16(out)) return GDN_ERR_ALIGN;  // the scan writes 16-byte output vectors
  const size_t base = gdn_workspace_bytes(layer, non_spec, spec);
  const size_t need = base + (chunked ? gdn_prefill_workspace_bytes(layer, non_spec, num_prefills) : 0);
  if (need && (!workspace || workspace_bytes < need)) return GDN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGN;

  const size_t C = (size_t)channels(layer);
  float* y_spec = static_cast<float*>(workspace);
  float* y_ns = reinterpret_cast<float*>(static_cast<char*>(workspace) + round256((size_t)ntok(spec) * C * 4));
  void* ws_prefill = static_cast<char*>(workspace) + base;
  cudaStream_t s = (cudaStream_t)stream;
  // rows of the token recurrence: the spec rows, then the decode rows (every non-spec row when
  // the prefill rows do not take the chunked path)
  const int rec_rows = nseq(spec) + (chunked ? num_decodes : nseq(non_spec));
  if (rec_rows > 65535) return GDN_ERR_SHAPE;

  // (1) conv over both subsets in one launch: spec rows first, then the non-spec units.
  ConvLaunch c = conv_args(layer, params, pools, x, num_actual_tokens, d_status);
  c.sub[0] = rows_dev(spec);
  c.y[0] = y_spec;
  c.units0 = conv_units(spec);
  c.sub[1] = rows_dev(non_spec);
  c.y[1] = y_ns;
  const int units = c.units0 + conv_units(non_spec);
  if (units > 65535) return GDN_ERR_SHAPE;
  if ((rc = cuda_rc(launch_conv(c, layer->conv_width, layer->act_dtype, GDN_F32, units, s)))) return rc;

  // (2) token recurrence over the recurrence rows, as a programmatic dependent of the conv.
  RecLaunch r = rec_args(layer, params, pools, a, b, out, num_actual_tokens, d_status);
  r.sub[0] = rows_dev(spec);
  r.qkv[0] = y_spec;
  r.rows0 = nseq(spec);
  r.sub[1] = rows_dev(non_spec);
  r.qkv[1] = y_ns;
  r.row_off1 = 0;
  if ((rc = cuda_rc(launch_recurrent(r, layer->act_dtype, GDN_F32, rec_rows, true, s)))) return rc;
  if (!chunked) return GDN_OK;

  // (3) chunked prefill of the prefill rows [num_decodes, num_decodes + num_prefills).
  const int chunk_units = prefill_units(non_spec, num_prefills);
  PrefillLaunch p = prefill_args(layer, params, pools, y_ns, a, b, out, num_actual_tokens, non_spec, num_decodes,
                                 num_prefills, ws_prefill, d_status);
  return cuda_rc(launch_prefill(p, GDN_F32, chunk_units, s));
}

}  // extern "C"
