// gdn_conv_core.cuh -- one thread's share of the causal conv1d update: VE channels of one row.
//
// Semantics ("[GDN] Spec-decoding-aware attention kernel", Problem and Changes: the conv ring is
// a rolled history in column 0 of the row's slots, read at offset num_accepted-1; token t of a
// K_call-token row lands at column state_len-K_call+t; the earlier columns are a shift copy of
// the pre-state; the roll into the slot must come after every read of it):
//   history h = pool[slot][a .. a+W-2] (zeros for a NULL slot or has_initial_state = 0),
//   H = h ++ x_row,  y_t = SiLU(bias + sum_i w[i] H[t+i]),
//   spec:     pool[slot][0 .. W-3+L] <- H[1 .. W-2+L]
//   non-spec: pool[slot][0 .. W-2]   <- H[L .. L+W-2]
//   per-slot spec layout ("[XE2] Support MTP of QWEN model", review thread): the history is read
//   from spec_state_indices[n, num_accepted-1] at offset 0, and after token t the last W-1
//   inputs go to columns 0..W-2 of spec_state_indices[n, t].
//
// The thread that reads a slot's history for its VE channels is the only one that ever writes
// those slot elements, and it writes them only after its reads, so the roll needs no staging
// buffer and no second pass.  The conv kernel runs it with 8 channels per thread (16-byte
// accesses for bf16); the channel count is a parameter so that a kernel short of registers can
// take fewer.
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

// VE consecutive elements of type T as raw 32-bit words (bit-exact copies), moved with the
// widest vector access their size allows: 16-byte accesses when the size is a multiple of 16
// bytes, else 8-byte, else 4-byte ones (the callers' offsets are aligned to the access size).
template <typename T, int VE>
struct RawV {
  static constexpr int NW = VE * (int)sizeof(T) / 4;
  static_assert(NW >= 1 && VE * (int)sizeof(T) % 4 == 0, "whole 32-bit words");
  uint32_t w[NW];
};

template <typename T, int VE>
__device__ __forceinline__ RawV<T, VE> load_rawv(const T* p) {
  RawV<T, VE> r;
  constexpr int NW = RawV<T, VE>::NW;
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + i);
      r.w[4 * i] = v.x; r.w[4 * i + 1] = v.y; r.w[4 * i + 2] = v.z; r.w[4 * i + 3] = v.w;
    }
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p) + i);
      r.w[2 * i] = v.x; r.w[2 * i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) r.w[i] = __ldg(reinterpret_cast<const unsigned int*>(p) + i);
  }
  return r;
}

template <typename T, int VE>
__device__ __forceinline__ RawV<T, VE> zero_rawv() {
  RawV<T, VE> r;
#pragma unroll
  for (int i = 0; i < RawV<T, VE>::NW; ++i) r.w[i] = 0u;
  return r;
}

template <typename T, int VE>
__device__ __forceinline__ void store_rawv(T* p, const RawV<T, VE>& r) {
  constexpr int NW = RawV<T, VE>::NW;
  if constexpr (NW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i)
      reinterpret_cast<uint4*>(p)[i] = make_uint4(r.w[4 * i], r.w[4 * i + 1], r.w[4 * i + 2], r.w[4 * i + 3]);
  } else if constexpr (NW % 2 == 0) {
#pragma unroll
    for (int i = 0; i < NW / 2; ++i) reinterpret_cast<uint2*>(p)[i] = make_uint2(r.w[2 * i], r.w[2 * i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) reinterpret_cast<unsigned int*>(p)[i] = r.w[i];
  }
}

template <typename T, int VE>
__device__ __forceinline__ void rawv_to_f32(const RawV<T, VE>& r, float (&f)[VE]) {
  const T* e = reinterpret_cast<const T*>(&r.w[0]);
#pragma unroll
  for (int i = 0; i < VE; ++i) f[i] = to_f32(e[i]);
}

template <typename T, int VE>
__device__ __forceinline__ void store_f32v(T* p, const float (&f)[VE]) {
  RawV<T, VE> r;
  T* e = reinterpret_cast<T*>(&r.w[0]);
#pragma unroll
  for (int i = 0; i < VE; ++i) e[i] = from_f32<T>(f[i]);
  store_rawv<T, VE>(p, r);
}

// SiLU(x) = x / (1 + e^-x) with the hardware exponential and fast division: a few ulp of fp32,
// far inside what the path's tolerances allow, at a fraction of the IEEE cost.  For x < -88 the
// exponential overflows and the quotient is -0.
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// Position in x of packed channel c: the identity for the packed layout; for the per-k-head
// layout, k-head g's group holds q_g, k_g and the v of its Hv/Hk v-heads.  A thread's channels
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

// The row-level facts the conv needs, read once (the loads go out together).
struct ConvRow {
  int32_t bos, eos;
  int na;        // num_accepted (1 when the subset carries none)
  int own;       // the row's conv slot: spec_state_indices[n, 0] or state_indices[n]
  bool has_init;
};

__device__ __forceinline__ ConvRow conv_row(const RowsDev& R, int n) {
  ConvRow r;
  r.bos = __ldg(R.qsl + n);
  r.eos = __ldg(R.qsl + n + 1);
  r.na = R.num_acc ? __ldg(R.num_acc + n) : 1;
  r.own = R.is_spec ? __ldg(R.spec_idx + (int64_t)n * R.spec_cols) : __ldg(R.state_idx + n);
  r.has_init = R.is_spec || R.has_init == nullptr || __ldg(R.has_init + n) != 0;
  return r;
}

template <typename T, int W, int VE>
struct ConvThread {
  float w[W][VE], bias[VE];
  RawV<T, VE> win[W - 1];  // raw inputs of the W-1 tokens before the next one
  int64_t xc;              // where the thread's VE channels sit in a row of x
  int64_t slot_base;   // pool offset of the row's slot, at the thread's channels
  int c0;
  int slot;            // the row's conv slot (0 when it must not be written)
  bool per_slot, spec_ring, writer;

  // Weights and bias of channels c0 .. c0+VE-1: VE*W contiguous elements.
  __device__ __forceinline__ void load_params(const ConvLaunch& p, int c) {
    c0 = c;
    const RawV<T, VE * W> wv = load_rawv<T, VE * W>(static_cast<const T*>(p.w) + (int64_t)c0 * W);
    const T* we = reinterpret_cast<const T*>(&wv.w[0]);
#pragma unroll
    for (int e = 0; e < VE; ++e)
#pragma unroll
      for (int i = 0; i < W; ++i) w[i][e] = to_f32(we[e * W + i]);
    if (p.bias) {
      float bb[VE];
      rawv_to_f32(load_rawv<T, VE>(static_cast<const T*>(p.bias) + c0), bb);
#pragma unroll
      for (int e = 0; e < VE; ++e) bias[e] = bb[e];
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) bias[e] = 0.f;
    }
  }

  // Resolves the slots and loads the window for a unit that starts at token t0 (segment seg of
  // the row).  Segment 0 reads the slot's history and, for rolled spec rows, writes the shifted
  // history (columns 0..W-3) at once; later segments rebuild their window from x.  Returns false
  // when the row must be skipped (num_accepted out of range).
  __device__ __forceinline__ bool begin(const ConvLaunch& p, const RowsDev& R, int n, const ConvRow& row, int seg,
                                        int t0, bool reporter) {
    int anchor, rd;
    bool read_prior;
    per_slot = R.is_spec && p.conv_layout == GDN_CONV_PER_SLOT;
    if (R.num_acc && (row.na < 1 || row.na > R.spec_cols)) {
      if (reporter) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
      return false;
    }
    if (R.is_spec) {
      // rolled: the history sits in column 0's slot at offset na-1; per slot: it is the
      // snapshot taken after the last accepted token
      slot = rd = per_slot ? __ldg(R.spec_idx + (int64_t)n * R.spec_cols + row.na - 1) : row.own;
      anchor = per_slot ? 0 : row.na - 1;
      read_prior = rd > 0;
    } else {
      slot = rd = row.own;
      anchor = 0;
      if (R.num_acc) {  // acceptance-aware row: the history its previous verify step accepted
        if (p.conv_layout == GDN_CONV_PER_SLOT) rd = __ldg(R.spec_idx + (int64_t)n * R.spec_cols + row.na - 1);
        else anchor = row.na - 1;
      }
      read_prior = rd > 0 && row.has_init;
    }
    if (slot >= p.num_slots || rd >= p.num_slots) {
      if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
      if (slot >= p.num_slots) slot = 0;
      read_prior = false;
    }
    const T* __restrict__ x = static_cast<const T*>(p.x);
    xc = x_channel(p, c0);
    T* __restrict__ pool = static_cast<T*>(p.conv_pool);
    const int64_t C = p.C;
    slot_base = (int64_t)slot * p.state_len * C + c0;
    const int64_t hist_base = (int64_t)(read_prior ? rd : 0) * p.state_len * C + c0;
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
      if (seg == 0) {
        win[i] = read_prior ? load_rawv<T, VE>(pool + hist_base + (int64_t)(anchor + i) * C) : zero_rawv<T, VE>();
      } else {
        const int g = global_token(R, row.bos + t0 - (W - 1) + i, p.num_global, p.status);
        win[i] = g >= 0 ? load_rawv<T, VE>(x + (int64_t)g * C + xc) : zero_rawv<T, VE>();
      }
    }
    // From here on this thread owns its slot elements: every read of them is done.
    writer = (seg == 0 && slot > 0);
    spec_ring = writer && R.is_spec && !per_slot;
    if (spec_ring) {
      // spec: columns 0..W-3 <- H[1..W-2] (the shifted history); token t goes to column W-2+t.
#pragma unroll
      for (int j = 0; j < W - 2; ++j) store_rawv<T, VE>(pool + slot_base + (int64_t)j * C, win[j + 1]);
    }
    return true;
  }

  // Tokens [ta, tb) of the row: y_t (fp32) handed to sink(t, y[VE]); the ring columns or per-slot
  // snapshots of those tokens written as they pass.  The x loads of 4 tokens go out together.
  template <typename Sink>
  __device__ __forceinline__ void tokens(const ConvLaunch& p, const RowsDev& R, int n, const ConvRow& row, int ta,
                                         int tb, bool reporter, Sink&& sink) {
    const T* __restrict__ x = static_cast<const T*>(p.x);
    T* __restrict__ pool = static_cast<T*>(p.conv_pool);
    const int64_t C = p.C;
    constexpr int G = 4;  // tokens whose loads are issued together
    for (int tg = ta; tg < tb; tg += G) {
      int gt[G];
#pragma unroll
      for (int k = 0; k < G; ++k) gt[k] = (tg + k < tb) ? global_token(R, row.bos + tg + k, p.num_global, p.status) : -1;
      RawV<T, VE> xr[G];
#pragma unroll
      for (int k = 0; k < G; ++k) xr[k] = gt[k] >= 0 ? load_rawv<T, VE>(x + (int64_t)gt[k] * C + xc) : zero_rawv<T, VE>();
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int t = tg + k;
        if (t >= tb) break;
        float hf[W - 1][VE], xf[VE], out[VE];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) rawv_to_f32(win[i], hf[i]);
        rawv_to_f32(xr[k], xf);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          float acc = bias[e];
#pragma unroll
          for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][e], hf[i][e], acc);
          acc = fmaf(w[W - 1][e], xf[e], acc);
          out[e] = silu(acc);
        }
        sink(t, out);
        if (spec_ring) store_rawv<T, VE>(pool + slot_base + (int64_t)(W - 2 + t) * C, xr[k]);
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
            for (int j = 0; j < W - 1; ++j) store_rawv<T, VE>(dst + (int64_t)j * C, win[j]);
          }
        }
      }
    }
  }

  // A non-spec unit's inputs through shared memory: the W-1 window rows (the slot's history for
  // segment 0, the previous x rows otherwise) and the unit's token rows [t0, t1) go out at once as
  // 16-byte cp.async copies into this thread's own column of `stage` (row r at stage[r * kConvThreads]),
  // so that no register is held while they are in flight; the window is then taken into
  // registers.  The same slot resolution as begin() for a non-spec row.  Returns false when the
  // row must be skipped (num_accepted out of range).
  __device__ __forceinline__ bool begin_staged(const ConvLaunch& p, const RowsDev& R, int n, const ConvRow& row,
                                               int seg, int t0, int t1, bool reporter, RawV<T, VE>* stage) {
    static_assert(sizeof(RawV<T, VE>) == 16, "one 16-byte copy per row");
    if (R.num_acc && (row.na < 1 || row.na > R.spec_cols)) {
      if (reporter) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
      return false;
    }
    per_slot = false;
    slot = row.own;
    int rd = row.own, anchor = 0;
    if (R.num_acc) {  // acceptance-aware row: the history its previous verify step accepted
      if (p.conv_layout == GDN_CONV_PER_SLOT) rd = __ldg(R.spec_idx + (int64_t)n * R.spec_cols + row.na - 1);
      else anchor = row.na - 1;
    }
    bool read_prior = rd > 0 && row.has_init;
    if (slot >= p.num_slots || rd >= p.num_slots) {
      if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
      if (slot >= p.num_slots) slot = 0;
      read_prior = false;
    }
    const T* __restrict__ x = static_cast<const T*>(p.x);
    const T* __restrict__ pool = static_cast<const T*>(p.conv_pool);
    xc = x_channel(p, c0);
    const int64_t C = p.C;
    slot_base = (int64_t)slot * p.state_len * C + c0;
    const int64_t hist_base = (int64_t)(read_prior ? rd : 0) * p.state_len * C + c0;
    // every token index first (no copy is issued between them), then every copy
    constexpr int kRows = kConvSegNS + W - 1;
    int g[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int t = t0 - (W - 1) + r;  // token of staged row r
      g[r] = -1;
      if (t >= t0 ? t < t1 : seg > 0) g[r] = global_token(R, row.bos + t, p.num_global, p.status);
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int t = t0 - (W - 1) + r;
      const T* src = nullptr;
      if (t < t0 && seg == 0) {
        if (read_prior) src = pool + hist_base + (int64_t)(anchor + r) * C;
      } else if (g[r] >= 0) {
        src = x + (int64_t)g[r] * C + xc;
      }
      RawV<T, VE>* dst = stage + r * kConvThreads;
      if (src) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                     "l"(src)
                     : "memory");
      } else if (t < t1) {
        *dst = zero_rawv<T, VE>();
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
    for (int i = 0; i < W - 1; ++i) win[i] = stage[i * kConvThreads];
    // From here on this thread owns its slot elements: every read of them is done.
    writer = (seg == 0 && slot > 0);
    spec_ring = false;
    return true;
  }

  // Tokens [ta, tb) of a unit staged by begin_staged: y_t handed to sink(t, y[VE]).
  template <typename Sink>
  __device__ __forceinline__ void tokens_staged(int ta, int tb, const RawV<T, VE>* stage, Sink&& sink) {
    for (int t = ta; t < tb; ++t) {
      const RawV<T, VE> xr = stage[(W - 1 + t - ta) * kConvThreads];
      float hf[W - 1][VE], xf[VE], out[VE];
#pragma unroll
      for (int i = 0; i < W - 1; ++i) rawv_to_f32(win[i], hf[i]);
      rawv_to_f32(xr, xf);
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        float acc = bias[e];
#pragma unroll
        for (int i = 0; i < W - 1; ++i) acc = fmaf(w[i][e], hf[i][e], acc);
        acc = fmaf(w[W - 1][e], xf[e], acc);
        out[e] = silu(acc);
      }
      sink(t, out);
#pragma unroll
      for (int i = 0; i < W - 2; ++i) win[i] = win[i + 1];
      win[W - 2] = xr;
    }
  }

  // Non-spec rows: columns 0..W-2 <- the row's last W-1 inputs H[L..L+W-2].  `saw_end`: this
  // thread's tokens reached the row's end, so the window holds exactly those inputs.
  __device__ __forceinline__ void finish(const ConvLaunch& p, const RowsDev& R, const ConvRow& row, bool saw_end) {
    if (!writer || R.is_spec) return;
    T* __restrict__ pool = static_cast<T*>(p.conv_pool);
    const int64_t C = p.C;
    const int L = row.eos - row.bos;
    if (saw_end) {
#pragma unroll
      for (int j = 0; j < W - 1; ++j) store_rawv<T, VE>(pool + slot_base + (int64_t)j * C, win[j]);
    } else {
      const T* __restrict__ x = static_cast<const T*>(p.x);
#pragma unroll
      for (int j = 0; j < W - 1; ++j) {
        const int g = global_token(R, row.bos + L - (W - 1) + j, p.num_global, p.status);
        store_rawv<T, VE>(pool + slot_base + (int64_t)j * C, g >= 0 ? load_rawv<T, VE>(x + (int64_t)g * C + xc) : zero_rawv<T, VE>());
      }
    }
  }
};

}  // namespace gdn
