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
// 2x4 fp32 per thread).  A spec unit issues the token index and x loads of 4 tokens together;
// a non-spec unit of bf16 activations issues every window and token row of the thread's column
// at once as cp.async copies into shared memory (no register held while they are in flight).
// The kernel lets the dependent recurrence grid launch early (programmatic dependent launch):
// that grid only reads this kernel's output after griddepcontrol.wait.
#include "gdn_conv_core.cuh"

namespace gdn {

#ifndef GDN_CONV_VE
#define GDN_CONV_VE 8  // channels per thread
#endif
#ifndef GDN_CONV_MINB
#define GDN_CONV_MINB 4  // resident CTAs per SM the register allocation must allow
#endif
constexpr int kConvVE = GDN_CONV_VE;

template <typename T, typename YT, int W>
__global__ void __launch_bounds__(kConvThreads, GDN_CONV_MINB) conv_update_kernel(const ConvLaunch p) {
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
  const int c0 = (blockIdx.x * kConvThreads + threadIdx.x) * kConvVE;
  if (c0 >= p.C) return;
  const bool reporter = (c0 == 0);

  // Loads that do not depend on one another go out together: the row's token range, its
  // acceptance, its own (or column-0) slot, and the thread's weights.
  const ConvRow row = conv_row(R, n);
  ConvThread<T, W, kConvVE> ct;
  ct.load_params(p, c0);

  if (row.bos < 0 || row.eos < row.bos || row.eos > R.num_tokens) {
    if (reporter) set_status(p.status, GDN_STATUS_ROW_RANGE);
    return;
  }
  const int L = row.eos - row.bos;
  if (L == 0) return;
  if (R.is_spec && L > R.spec_cols) {
    if (reporter) set_status(p.status, GDN_STATUS_ROW_RANGE);
    return;
  }
  const int seg_len = R.is_spec ? kConvSeg : kConvSegNS;
  const int t0 = seg * seg_len;
  if (t0 >= L) return;
  const int t1 = min(L, t0 + seg_len);

  YT* __restrict__ y = static_cast<YT*>(p.y[s]);
  auto sink = [&](int t, const float(&out)[kConvVE]) {
    store_f32v<YT, kConvVE>(y + (int64_t)(row.bos + t) * p.C + c0, out);
  };
  if constexpr (sizeof(RawV<T, kConvVE>) == 16) {
    if (!R.is_spec) {  // non-spec units: every input row in flight at once through shared memory
      __shared__ RawV<T, kConvVE> stage[(kConvSegNS + W - 1) * kConvThreads];
      if (!ct.begin_staged(p, R, n, row, seg, t0, t1, reporter, stage + threadIdx.x)) return;
      ct.tokens_staged(t0, t1, stage + threadIdx.x, sink);
      ct.finish(p, R, row, t1 == L);
      return;
    }
  }
  if (!ct.begin(p, R, n, row, seg, t0, reporter)) return;
  ct.tokens(p, R, n, row, t0, t1, reporter, sink);
  ct.finish(p, R, row, t1 == L);
}

template <typename T, typename YT>
static cudaError_t launch_w(const ConvLaunch& p, int width, int units, cudaStream_t s) {
  const dim3 grid((p.C / kConvVE + kConvThreads - 1) / kConvThreads, units);
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
