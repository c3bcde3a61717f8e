// gdn_conv.cu -- causal conv1d update with the speculative column-0 ring contract.
//
// Semantics ("[GDN] Spec-decoding-aware attention kernel", Problem and Changes: the conv ring
// is a rolled history in column 0 of the row's slots, read at offset num_accepted-1; token t of
// a K_call-token row lands at column state_len-K_call+t; the earlier columns are a shift copy
// of the pre-state; the roll into the slot must come after every read of it):
//   history h = pool[slot][a .. a+W-2] (zeros for a NULL slot or has_initial_state = 0),
//   H = h ++ x_row,  y_t = SiLU(bias + sum_i w[i] H[t+i]),
//   spec:     pool[slot][0 .. W-3+L] <- H[1 .. W-2+L]
//   non-spec: pool[slot][0 .. W-2]   <- H[L .. L+W-2]
//
// GB300 design.  The pages split the update into a staging pass and a separate roll pass
// because their work-items cover single tokens, so a row's reads and writes of its slot are
// spread over many items.  Here one thread owns 8 channels of a row for every token it touches:
// it loads the history into registers, runs the FMA chain over its tokens, and only then writes
// the new columns -- the thread that reads a slot element is the only one that writes it, after
// its read, so the roll needs no tmp buffer and no second launch.  Long non-spec rows are cut
// into 64-token segments for parallelism; segment 0 alone touches the slot (it also fetches the
// row's last W-1 inputs for the write-back), later segments rebuild their window from x.
// All accesses are 16-byte vectors along the channel axis (8 bf16 or 2x4 fp32 per thread).
#include "gdn_internal.cuh"

namespace gdn {

// Maps work unit `unit` of a non-spec subset to (row, segment); row n owns ceil(L_n / kConvSeg)
// units.  Warp 0 scans the rows 32 at a time; the answer is broadcast through shared memory.
// Every thread of the block must call it.
__device__ bool locate_unit(const RowsDev& r, int unit, int& row, int& seg, uint32_t* st) {
  __shared__ int s_row, s_seg;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0, found_row = -1, found_seg = 0;
    for (int r0 = 0; r0 < r.num_seqs; r0 += 32) {
      const int n = r0 + lane;
      int cnt = 0;
      if (n < r.num_seqs) {
        const int bos = __ldg(r.qsl + n), eos = __ldg(r.qsl + n + 1);
        if (bos < 0 || eos < bos || eos > r.num_tokens) {
          if (unit == 0) set_status(st, GDN_STATUS_ROW_RANGE);
        } else {
          cnt = (eos - bos + kConvSeg - 1) / kConvSeg;
        }
      }
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const int excl = inc - cnt;
      const bool hit = unit >= base + excl && unit < base + inc;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int src = __ffs(m) - 1;
        found_row = r0 + src;
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

template <int W, typename T>
__device__ __forceinline__ Raw8<T> pick(const Raw8<T> (&h)[W - 1], int m) {
  Raw8<T> v = h[0];
#pragma unroll
  for (int i = 1; i < W - 1; ++i)
    if (i == m) v = h[i];
  return v;
}

template <typename T, typename YT, int W>
__global__ void __launch_bounds__(kConvThreads) conv_update_kernel(const ConvLaunch p) {
  const int uy = blockIdx.y;
  const int s = uy < p.units0 ? 0 : 1;
  const RowsDev R = p.sub[s];
  const int unit = s == 0 ? uy : uy - p.units0;
  int n, seg;
  if (R.is_spec) {
    n = unit;
    seg = 0;
    if (n >= R.num_seqs) return;
  } else if (!locate_unit(R, unit, n, seg, p.status)) {
    return;
  }
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
  if (c0 >= p.C) return;
  const bool reporter = (c0 == 0);

  const int32_t bos = __ldg(R.qsl + n), eos = __ldg(R.qsl + n + 1);
  if (bos < 0 || eos < bos || eos > R.num_tokens) {
    if (reporter) set_status(p.status, GDN_STATUS_ROW_RANGE);
    return;
  }
  const int L = eos - bos;
  if (L == 0) return;
  if (R.is_spec && L > R.spec_cols) {
    if (reporter) set_status(p.status, GDN_STATUS_ROW_RANGE);
    return;
  }
  const int t0 = seg * kConvSeg;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + kConvSeg);

  int slot, anchor;
  bool read_prior;
  if (R.is_spec) {
    const int na = __ldg(R.num_acc + n);
    if (na < 1 || na > R.spec_cols) {
      if (reporter) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
      return;
    }
    slot = __ldg(R.spec_idx + (int64_t)n * R.spec_cols);
    anchor = na - 1;
    read_prior = slot > 0;
  } else {
    slot = __ldg(R.state_idx + n);
    anchor = 0;
    read_prior = slot > 0 && (R.has_init == nullptr || __ldg(R.has_init + n) != 0);
  }
  if (slot >= p.num_slots) {
    if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
    slot = 0;
    read_prior = false;
  }

  const T* __restrict__ x = static_cast<const T*>(p.x);
  T* __restrict__ pool = static_cast<T*>(p.conv_pool);
  const T* __restrict__ wp = static_cast<const T*>(p.w);
  const int64_t C = p.C;

  float w[W][8], bias[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
#pragma unroll
    for (int i = 0; i < W; ++i) w[i][e] = to_f32(wp[(c0 + e) * W + i]);
    bias[e] = p.bias ? to_f32(static_cast<const T*>(p.bias)[c0 + e]) : 0.f;
  }

  // Window of the W-1 inputs before the current token, and (segment 0) the raw history.
  Raw8<T> hraw[W - 1];
  float win[W - 1][8];
#pragma unroll
  for (int i = 0; i < W - 1; ++i) {
    if (seg == 0) {
      hraw[i] = read_prior ? load_raw8(pool + ((int64_t)slot * p.state_len + anchor + i) * C + c0) : zero_raw8<T>();
      raw8_to_f32(hraw[i], win[i]);
    } else {
      const int g = global_token(R, bos + t0 - (W - 1) + i, p.num_global, p.status);
      const Raw8<T> v = g >= 0 ? load_raw8(x + (int64_t)g * C + c0) : zero_raw8<T>();
      raw8_to_f32(v, win[i]);
      hraw[i] = v;
    }
  }

  YT* __restrict__ y = static_cast<YT*>(p.y[s]);
  for (int t = t0; t < t1; ++t) {
    const int g = global_token(R, bos + t, p.num_global, p.status);
    float xf[8];
    raw8_to_f32(g >= 0 ? load_raw8(x + (int64_t)g * C + c0) : zero_raw8<T>(), xf);
    float out[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float acc = bias[e];
#pragma unroll
      for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][e], win[i][e], acc);
      acc = fmaf(w[W - 1][e], xf[e], acc);
      out[e] = acc / (1.0f + expf(-acc));
    }
    store_f32x8(y + (int64_t)(bos + t) * C + c0, out);
#pragma unroll
    for (int i = 0; i < W - 2; ++i)
#pragma unroll
      for (int e = 0; e < 8; ++e) win[i][e] = win[i + 1][e];
#pragma unroll
    for (int e = 0; e < 8; ++e) win[W - 2][e] = xf[e];
  }

  // Roll: this thread read its slot elements above and is their only writer.
  if (seg == 0 && slot > 0) {
    const int off = R.is_spec ? 1 : L;
    const int ncols = R.is_spec ? W - 2 + L : W - 1;
    for (int j = 0; j < ncols; ++j) {
      const int m = off + j;
      Raw8<T> v;
      if (m < W - 1) {
        v = pick<W>(hraw, m);
      } else {
        const int g = global_token(R, bos + m - (W - 1), p.num_global, p.status);
        v = g >= 0 ? load_raw8(x + (int64_t)g * C + c0) : zero_raw8<T>();
      }
      store_raw8(pool + ((int64_t)slot * p.state_len + j) * C + c0, v);
    }
  }
}

template <typename T, typename YT>
static cudaError_t launch_w(const ConvLaunch& p, int width, int units, cudaStream_t s) {
  const dim3 grid((p.C / 8 + kConvThreads - 1) / kConvThreads, units);
  switch (width) {
    case 2: conv_update_kernel<T, YT, 2><<<grid, kConvThreads, 0, s>>>(p); break;
    case 3: conv_update_kernel<T, YT, 3><<<grid, kConvThreads, 0, s>>>(p); break;
    case 4: conv_update_kernel<T, YT, 4><<<grid, kConvThreads, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_conv(const ConvLaunch& p, int width, gdn_dtype act, gdn_dtype y_dtype, int units_total,
                        cudaStream_t s) {
  if (units_total <= 0) return cudaSuccess;
  if (act == GDN_BF16)
    return y_dtype == GDN_F32 ? launch_w<__nv_bfloat16, float>(p, width, units_total, s)
                              : launch_w<__nv_bfloat16, __nv_bfloat16>(p, width, units_total, s);
  return y_dtype == GDN_F32 ? launch_w<float, float>(p, width, units_total, s)
                            : launch_w<float, __nv_bfloat16>(p, width, units_total, s);
}

}  // namespace gdn
