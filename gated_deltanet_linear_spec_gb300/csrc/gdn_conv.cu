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
// it loads the slot's history into registers before anything else, and from then on it is the
// only reader and writer of those slot elements, so it writes the rolled columns as the tokens
// stream through -- no tmp buffer, no second launch, no race.  Long non-spec rows are cut into
// 16-token segments for parallelism; segment 0 alone touches the slot (it fetches the row's last
// W-1 inputs for the write-back when the row is longer than one segment), later segments rebuild
// their window from x.  All accesses are 16-byte vectors along the channel axis (8 bf16 or
// 2x4 fp32 per thread); the token index and x loads of 4 tokens are issued together.
// The kernel lets the dependent recurrence grid launch early (programmatic dependent launch):
// that grid only reads this kernel's output after griddepcontrol.wait.
#include "gdn_internal.cuh"

namespace gdn {

// SiLU(x) = x / (1 + e^-x) with the hardware exponential and fast division: a few ulp of
// fp32, far inside what the path's tolerances allow, at a fraction of the IEEE cost.  For
// x < -88 the exponential overflows and the quotient is -0.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Position in x of packed channel c: the identity for the packed layout; for the per-k-head
// layout, k-head g's group holds q_g, k_g and the v of its Hv/Hk v-heads.  A thread's 8 channels
// never straddle a head, so they stay contiguous in x.
__device__ __forceinline__ int64_t x_channel(const ConvLaunch& p, int c) {
  if (p.qkv_layout == GDN_QKV_PACKED) return c;
  const int G = p.Hv / p.Hk, group = 2 * p.dk + G * p.dv;
  const int qk = p.Hk * p.dk;
  if (c < qk) return (int64_t)(c / p.dk) * group + c % p.dk;
  if (c < 2 * qk) return (int64_t)((c - qk) / p.dk) * group + p.dk + (c - qk) % p.dk;
  const int vc = c - 2 * qk, hv = vc / p.dv;
  return (int64_t)(hv / G) * group + 2 * p.dk + (hv % G) * p.dv + vc % p.dv;
}

template <typename T, typename YT, int W>
__global__ void __launch_bounds__(kConvThreads, 4) conv_update_kernel(const ConvLaunch p) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int uy = blockIdx.y;
  const int s = uy < p.units0 ? 0 : 1;
  const RowsDev R = p.sub[s];
  const int unit = s == 0 ? uy : uy - p.units0;
  int n, seg;
  if (R.is_spec) {
    n = unit;
    seg = 0;
    if (n >= R.num_seqs) return;
  } else if (!locate_unit(R, 0, R.num_seqs, kConvSegNS, unit, n, seg, p.status)) {
    return;
  }
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * 8;
  if (c0 >= p.C) return;
  const bool reporter = (c0 == 0);

  // Loads that do not depend on one another go out together: the row's token range, its
  // acceptance, its own (or column-0) slot, and the thread's weights.
  const int32_t bos = __ldg(R.qsl + n), eos = __ldg(R.qsl + n + 1);
  const int na = R.num_acc ? __ldg(R.num_acc + n) : 1;
  const int own = R.is_spec ? __ldg(R.spec_idx + (int64_t)n * R.spec_cols) : __ldg(R.state_idx + n);
  const bool has_init = R.is_spec || R.has_init == nullptr || __ldg(R.has_init + n) != 0;
  // Weights and bias of the thread's 8 channels: 8*W contiguous elements, 16-byte vectors.
  float w[W][8], bias[8];
  {
    constexpr int NW = 8 * W * (int)sizeof(T) / 16;
    uint4 wv[NW];
    const uint4* wsrc = reinterpret_cast<const uint4*>(static_cast<const T*>(p.w) + (int64_t)c0 * W);
#pragma unroll
    for (int i = 0; i < NW; ++i) wv[i] = __ldg(wsrc + i);
    const T* we = reinterpret_cast<const T*>(wv);
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int i = 0; i < W; ++i) w[i][e] = to_f32(we[e * W + i]);
  }
  if (p.bias) {
    float bb[8];
    raw8_to_f32(load_raw8(static_cast<const T*>(p.bias) + c0), bb);
#pragma unroll
    for (int e = 0; e < 8; ++e) bias[e] = bb[e];
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) bias[e] = 0.f;
  }

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
  const int seg_len = R.is_spec ? kConvSeg : kConvSegNS;
  const int t0 = seg * seg_len;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + seg_len);

  int slot, anchor;  // the row's conv slot; the history's column offset
  int rd;            // the slot the history is read from
  bool read_prior;
  const bool per_slot = R.is_spec && p.conv_layout == GDN_CONV_PER_SLOT;
  if (R.num_acc && (na < 1 || na > R.spec_cols)) {
    if (reporter) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
    return;
  }
  if (R.is_spec) {
    // rolled: the history sits in column 0's slot at offset na-1; per slot: it is the snapshot
    // taken after the last accepted token
    slot = rd = per_slot ? __ldg(R.spec_idx + (int64_t)n * R.spec_cols + na - 1) : own;
    anchor = per_slot ? 0 : na - 1;
    read_prior = rd > 0;
  } else {
    slot = rd = own;
    anchor = 0;
    if (R.num_acc) {  // acceptance-aware row: the history its previous verify step accepted
      if (p.conv_layout == GDN_CONV_PER_SLOT) rd = __ldg(R.spec_idx + (int64_t)n * R.spec_cols + na - 1);
      else anchor = na - 1;
    }
    read_prior = rd > 0 && has_init;
  }
  if (slot >= p.num_slots || rd >= p.num_slots) {
    if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
    if (slot >= p.num_slots) slot = 0;
    read_prior = false;
  }

  const T* __restrict__ x = static_cast<const T*>(p.x);
  const int64_t xc = x_channel(p, c0);  // where this thread's 8 channels sit in a row of x
  T* __restrict__ pool = static_cast<T*>(p.conv_pool);
  const int64_t C = p.C;
  const int64_t slot_base = (int64_t)slot * p.state_len * C + c0;
  const int64_t hist_base = (int64_t)(read_prior ? rd : 0) * p.state_len * C + c0;

  // Raw window of the W-1 inputs before the current token: the slot's history (segment 0)
  // or the row's previous inputs (later segments).
  Raw8<T> win[W - 1];
#pragma unroll
  for (int i = 0; i < W - 1; ++i) {
    if (seg == 0) {
      win[i] = read_prior ? load_raw8(pool + hist_base + (int64_t)(anchor + i) * C) : zero_raw8<T>();
    } else {
      const int g = global_token(R, bos + t0 - (W - 1) + i, p.num_global, p.status);
      win[i] = g >= 0 ? load_raw8(x + (int64_t)g * C + xc) : zero_raw8<T>();
    }
  }
  // From here on this thread owns its slot elements: every read of them is done.
  const bool writer = (seg == 0 && slot > 0);
  const bool spec_ring = writer && R.is_spec && !per_slot;
  if (spec_ring) {
    // spec: columns 0..W-3 <- H[1..W-2] (the shifted history); token t goes to column W-2+t below.
#pragma unroll
    for (int j = 0; j < W - 2; ++j) store_raw8(pool + slot_base + (int64_t)j * C, win[j + 1]);
  }

  YT* __restrict__ y = static_cast<YT*>(p.y[s]);
  constexpr int G = 4;  // tokens whose loads are issued together
  for (int tg = t0; tg < t1; tg += G) {
    int gt[G];
#pragma unroll
    for (int k = 0; k < G; ++k) gt[k] = (tg + k < t1) ? global_token(R, bos + tg + k, p.num_global, p.status) : -1;
    Raw8<T> xr[G];
#pragma unroll
    for (int k = 0; k < G; ++k) xr[k] = gt[k] >= 0 ? load_raw8(x + (int64_t)gt[k] * C + xc) : zero_raw8<T>();
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const int t = tg + k;
      if (t >= t1) break;
      float hf[W - 1][8], xf[8], out[8];
#pragma unroll
      for (int i = 0; i < W - 1; ++i) raw8_to_f32(win[i], hf[i]);
      raw8_to_f32(xr[k], xf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float acc = bias[e];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][e], hf[i][e], acc);
        acc = fmaf(w[W - 1][e], xf[e], acc);
        out[e] = silu(acc);
      }
      store_f32x8(y + (int64_t)(bos + t) * C + c0, out);
      if (spec_ring) store_raw8(pool + slot_base + (int64_t)(W - 2 + t) * C, xr[k]);
#pragma unroll
      for (int i = 0; i < W - 2; ++i) win[i] = win[i + 1];
      win[W - 2] = xr[k];
      if (per_slot) {  // the snapshot after token t goes to spec_state_indices[n, t]
        const int ss = __ldg(R.spec_idx + (int64_t)n * R.spec_cols + t);
        if (ss >= p.num_slots) {
          if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
        } else if (ss > 0) {
          T* dst = pool + (int64_t)ss * p.state_len * C + c0;
#pragma unroll
          for (int j = 0; j < W - 1; ++j) store_raw8(dst + (int64_t)j * C, win[j]);
        }
      }
    }
  }

  // non-spec: columns 0..W-2 <- the row's last W-1 inputs H[L..L+W-2].
  if (writer && !R.is_spec) {
    if (t1 == L) {
      // this unit saw the row's end: the window holds exactly H[L..L+W-2]
#pragma unroll
      for (int j = 0; j < W - 1; ++j) store_raw8(pool + slot_base + (int64_t)j * C, win[j]);
    } else {
#pragma unroll
      for (int j = 0; j < W - 1; ++j) {
        const int g = global_token(R, bos + L - (W - 1) + j, p.num_global, p.status);
        store_raw8(pool + slot_base + (int64_t)j * C, g >= 0 ? load_raw8(x + (int64_t)g * C + xc) : zero_raw8<T>());
      }
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
