// gdn_internal.cuh -- device-side types and helpers shared by the GDN kernels (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// One subset of rows as the kernels see it (plain values copied from gdn_rows).
struct RowsDev {
  const int32_t* qsl;
  const int32_t* tok;        // NULL = identity
  const int32_t* state_idx;  // non-spec
  const int32_t* has_init;   // non-spec, NULL = all 1
  const int32_t* spec_idx;   // spec [num_seqs, spec_cols]
  const int32_t* num_acc;    // spec
  int32_t spec_cols;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t is_spec;
};

__device__ __forceinline__ void set_status(uint32_t* st, uint32_t bit) {
  if (st) atomicOr(st, bit);
}

// Global token of local token i (identity when no token_indx), or -1 if out of range.
__device__ __forceinline__ int32_t global_token(const RowsDev& r, int32_t i, int32_t num_global, uint32_t* st) {
  int32_t g = r.tok ? __ldg(r.tok + i) : i;
  if (g < 0 || g >= num_global) {
    set_status(st, GDN_STATUS_TOKEN_RANGE);
    return -1;
  }
  return g;
}

// ---- element conversion --------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 8 consecutive elements as raw 16-byte vectors (1 for bf16, 2 for fp32): bit-exact copies.
template <typename T>
struct Raw8 {
  static constexpr int N = (int)sizeof(T) / 2;  // uint4 per 8 elements
  uint4 v[N];
};

template <typename T>
__device__ __forceinline__ Raw8<T> load_raw8(const T* p) {
  Raw8<T> r;
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < Raw8<T>::N; ++i) r.v[i] = __ldg(q + i);
  return r;
}

template <typename T>
__device__ __forceinline__ Raw8<T> zero_raw8() {
  Raw8<T> r;
#pragma unroll
  for (int i = 0; i < Raw8<T>::N; ++i) r.v[i] = make_uint4(0u, 0u, 0u, 0u);
  return r;
}

template <typename T>
__device__ __forceinline__ void store_raw8(T* p, const Raw8<T>& r) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < Raw8<T>::N; ++i) q[i] = r.v[i];
}

template <typename T>
__device__ __forceinline__ void raw8_to_f32(const Raw8<T>& r, float (&f)[8]) {
  const T* e = reinterpret_cast<const T*>(&r.v[0]);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = to_f32(e[i]);
}

template <typename T>
__device__ __forceinline__ void store_f32x8(T* p, const float (&f)[8]) {
  Raw8<T> r;
  T* e = reinterpret_cast<T*>(&r.v[0]);
#pragma unroll
  for (int i = 0; i < 8; ++i) e[i] = from_f32<T>(f[i]);
  store_raw8(p, r);
}

// ---- launch plumbing (host) ----------------------------------------------------------------

inline RowsDev rows_dev(const gdn_rows* r) {
  RowsDev d{};
  if (!r) return d;
  d.qsl = r->query_start_loc;
  d.tok = r->token_indx;
  d.state_idx = r->state_indices;
  d.has_init = r->has_initial_state;
  d.spec_idx = r->spec_state_indices;
  d.num_acc = r->num_accepted_tokens;
  d.spec_cols = r->spec_cols;
  d.num_seqs = r->num_seqs;
  d.num_tokens = r->num_tokens;
  d.is_spec = (r->spec_state_indices != nullptr) ? 1 : 0;
  return d;
}

// Conv: tokens per work unit of a long (non-spec) row.  Spec rows are one unit each.
constexpr int kConvSeg = 64;
constexpr int kConvThreads = 128;  // each thread owns 8 channels

struct ConvLaunch {
  const void* x;
  int32_t num_global;
  const void* w;
  const void* bias;
  void* conv_pool;
  int64_t num_slots;
  int32_t state_len;
  int32_t C;
  RowsDev sub[2];
  void* y[2];
  int32_t units0;  // grid.y units that belong to subset 0
  uint32_t* status;
};

struct RecLaunch {
  const void* qkv[2];
  const void* a;
  const void* b;
  void* out;
  int32_t num_global;
  const float* A_log;
  const float* dt_bias;
  float* ssm_pool;
  int64_t num_slots;
  int32_t Hk, Hv, dk, dv, C;
  float scale;
  RowsDev sub[2];
  int32_t rows0;     // grid.z rows of subset 0
  int32_t row_off1;  // first row of subset 1 handled by this launch
  uint32_t* status;
};

// Host launchers (one per kernel family); return cudaGetLastError() after the launch.
cudaError_t launch_conv(const ConvLaunch& p, int width, gdn_dtype act, gdn_dtype y_dtype, int units_total,
                        cudaStream_t s);
// pdl: launch as a programmatic dependent of the kernel just before it on the stream.
cudaError_t launch_recurrent(const RecLaunch& p, gdn_dtype act, gdn_dtype qkv_dtype, int rows_total, bool pdl,
                             cudaStream_t s);

}  // namespace gdn
