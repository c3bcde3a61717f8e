// gdn_internal.cuh -- device-side types and helpers shared by the GDN kernels (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gdn.h"

namespace gdn {

// One subset of rows as the kernels see it (plain values copied from gdn_rows).
struct RowsDev {
  const int32_t* qsl;
  const int32_t* tok;        // NULL = identity
  const int32_t* state_idx;  // non-spec
  const int32_t* has_init;   // non-spec, NULL = all 1
  const int32_t* spec_idx;   // spec [num_seqs, spec_cols]; acceptance-aware non-spec rows too
  const int32_t* num_acc;    // spec; acceptance-aware non-spec rows too (else NULL)
  int32_t spec_cols;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t is_spec;
};

// Slot of a non-spec row's prior SSM state: state_indices[n], or for acceptance-aware rows
// the previous verify step's slot of its last accepted token.  -1: num_accepted out of range.
__device__ __forceinline__ int32_t non_spec_load_slot(const RowsDev& R, int n) {
  if (R.num_acc == nullptr) return __ldg(R.state_idx + n);
  const int na = __ldg(R.num_acc + n);
  if (na < 1 || na > R.spec_cols) return -1;
  return __ldg(R.spec_idx + (int64_t)n * R.spec_cols + na - 1);
}

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

// ---- work units over variable-length rows ---------------------------------------------------

// Units of one row: ceil(L / seg_len), 0 for empty or malformed rows.
__device__ __forceinline__ int row_units(const RowsDev& r, int n, int seg_len, bool& bad) {
  const int bos = __ldg(r.qsl + n), eos = __ldg(r.qsl + n + 1);
  bad = (bos < 0 || eos < bos || eos > r.num_tokens);
  return bad ? 0 : (eos - bos + seg_len - 1) / seg_len;
}

// Maps work unit `unit` to (row, segment) over rows [first, first + count) of r, where row n
// owns ceil(L_n / seg_len) consecutive units in row order.  Warp 0 scans 32 rows at a time and
// broadcasts the answer through shared memory; every thread of the block must call it.
__device__ __forceinline__ bool locate_unit(const RowsDev& r, int first, int count, int seg_len, int unit, int& row,
                                            int& seg, uint32_t* st) {
  __shared__ int s_row, s_seg;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0, found_row = -1, found_seg = 0;
    for (int r0 = 0; r0 < count; r0 += 32) {
      int cnt = 0;
      if (r0 + lane < count) {
        bool bad;
        cnt = row_units(r, first + r0 + lane, seg_len, bad);
        if (bad && unit == 0) set_status(st, GDN_STATUS_ROW_RANGE);
      }
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int excl = inc - cnt;
      const unsigned m = __ballot_sync(0xffffffffu, unit >= base + excl && unit < base + inc);
      if (m) {
        const int src = __ffs(m) - 1;
        found_row = first + r0 + src;
        found_seg = unit - base - __shfl_sync(0xffffffffu, excl, src);
        break;
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      s_row = found_row;
      s_seg = found_seg;
    }
  }
  __syncthreads();
  row = s_row;
  seg = s_seg;
  return row >= 0;
}

// Units owned by rows [first, n): the index of row n's first unit.  Every thread must call it.
__device__ __forceinline__ int units_before(const RowsDev& r, int first, int n, int seg_len) {
  __shared__ int s_sum;
  if (threadIdx.x < 32) {
    int acc = 0;
    for (int m = first + (int)threadIdx.x; m < n; m += 32) {
      bool bad;
      acc += row_units(r, m, seg_len, bad);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (threadIdx.x == 0) s_sum = acc;
  }
  __syncthreads();
  return s_sum;
}

// ---- launch plumbing (host) ----------------------------------------------------------------

// Runs `set` (a kernel attribute call, which applies to the current device's context) once per
// device; safe to call from several host threads (a racing first call just repeats `set`).
template <typename F>
inline cudaError_t once_per_device(std::atomic<uint64_t>& done, F set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64) return set();
  const uint64_t bit = uint64_t(1) << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

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
  d.is_spec = (r->spec_state_indices != nullptr && r->state_indices == nullptr) ? 1 : 0;
  return d;
}

// Conv work units: a spec row is one unit of at most kConvSeg tokens; a non-spec row is cut into
// units of kConvSegNS tokens (short units keep each thread's chain of dependent token loads short).
constexpr int kConvSeg = 64;
constexpr int kConvSegNS = 16;
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
  int32_t Hk, dk, Hv, dv;
  int32_t qkv_layout;   // gdn_qkv_layout of x
  int32_t conv_layout;  // gdn_conv_layout of spec rows
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

// Chunked prefill (tensor-core path): chunk length and the per (chunk, v-head) record size.
constexpr int kPrefillChunk = 64;
constexpr uint32_t kRecBytes = 123904;

struct PrefillLaunch {
  const void* qkv;  // post-conv q|k|v [T_sub, C] (fp32 or bf16), local order
  const void* a;
  const void* b;
  void* out;
  int32_t num_global;
  const float* A_log;
  const float* dt_bias;
  float* ssm_pool;
  int64_t num_slots;
  int32_t Hk, Hv, C;
  float scale;
  RowsDev rows;       // a non-spec subset
  int32_t first_row;  // the prefill rows are [first_row, first_row + num_rows)
  int32_t num_rows;
  uint8_t* ws;        // units x Hv records of kRecBytes
  uint32_t* status;
  uint64_t wait_ns;         // wall-clock limit of each bounded mbarrier wait
  int32_t drop_copy_chunk;  // test hook: the scan issues no record copy for this chunk (< 0: none)
};

// Default limit of a bounded wait in the tensor-core kernels: far beyond any legitimate wait
// (a few microseconds), short enough that a lost arrival ends the launch promptly.
constexpr uint64_t kDefaultWaitNs = 1000000000ull;

// Host launchers (one per kernel family); return cudaGetLastError() after the launch.
cudaError_t launch_conv(const ConvLaunch& p, int width, gdn_dtype act, gdn_dtype y_dtype, int units_total,
                        cudaStream_t s);
// pdl: launch as a programmatic dependent of the kernel just before it on the stream.
cudaError_t launch_recurrent(const RecLaunch& p, gdn_dtype act, gdn_dtype qkv_dtype, int rows_total, bool pdl,
                             cudaStream_t s);
// The tensor-core chunked prefill handles dk = dv = 128 with bf16 activations.
bool prefill_tc_supported(const gdn_layer_desc* d);
cudaError_t launch_prefill(const PrefillLaunch& p, gdn_dtype qkv_dtype, int units_upper, cudaStream_t s);

}  // namespace gdn
