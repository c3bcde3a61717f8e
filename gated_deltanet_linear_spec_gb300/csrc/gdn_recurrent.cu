// gdn_recurrent.cu -- token-by-token gated delta rule for decode and speculative-verify rows.
//
// Semantics ("[GDN] Spec-decoding-aware attention kernel", Changes, gated_delta_rule.hpp:
// load slot spec_state_indices[n, num_accepted[n]-1], per-token store slot
// spec_state_indices[n, t], slot <= 0 = no prior state / no store; the non-spec rows load and
// store state_indices[n], except that rows carrying their previous verify step's acceptance load
// spec_state_indices[n, num_accepted-1]).  Per (token, v-head h):
//   g = -exp(A_log[h]) softplus(a + dt_bias[h]),  beta = sigmoid(b),
//   q^ = q / sqrt(|q|^2 + 1e-6) * scale,  k^ = k / sqrt(|k|^2 + 1e-6),
//   S <- e^g S (I - beta k^ k^T) + beta v k^T,   o = S q^.
// The a/b gates are read at token_indx, the same index as the q|k|v row ("[Bugfix] Align Qwen
// GDN gates with speculative tokens", Purpose).
//
// GB300 design.  Decode/verify is fp32-state streaming: each (row, head) reads one 64 KiB state
// and writes one per verify token, ~4 flops per byte, so the kernel is built for HBM, not the
// tensor pipe.  Rows of S are independent (row i only needs s_i.k^, s_i.q^ and v_i), so one CTA
// owns a (sequence, v-head, TPC dv-tiles of DVT rows) block and needs no cross-CTA exchange.
// Most of a CTA's life is the latency of its dependent token-preparation loads (row metadata,
// then q|k|v and the gates), so a CTA carries TPC tiles (two by default) through one
// preparation: the other tiles' states arrive in shared memory by cp.async meanwhile and are
// swapped into registers in turn once the previous tile's tokens are done.  LPR lanes share a
// state row, each holding DK/LPR fp32 in registers; lane l of a row takes the 16-byte words
// l, l+LPR, l+2*LPR, ... so every warp-wide 128-bit load/store covers 32*16 bytes in LPR-word
// runs per row.  The two dot products per token are reduced with
// xor-shuffles inside the row's lanes, using
//   S_t q^ = e^g (S_{t-1} q^) + delta (k^.q^),  delta = beta (v - e^g S_{t-1} k^),
// so both reductions run on the loaded state in one pass.  The prior state is issued as
// streaming 128-bit loads before the token data is staged, so the state fetch overlaps the
// norm/gate prologue -- and, in the mixed-batch path, the tail of the conv grid, which this
// kernel follows as a programmatic dependent launch.  Each thread stores exactly the elements
// it loaded, after loading them, so the load slot may also be a store slot (t = num_accepted-1)
// without a hazard.
#include "gdn_internal.cuh"

namespace gdn {

#ifndef GDN_REC_LD_HINT
#define GDN_REC_LD_HINT 0  // 0: L1 no-allocate; 1: also ask L2 for 256-byte prefetch
#endif
#ifndef GDN_REC_ST_HINT
#define GDN_REC_ST_HINT 1  // 0: default store; 1: streaming (.cs) store, evict-first in L2
#endif

// Streaming 128-bit load of the prior state.  Not the non-coherent (.nc) path: the launch may
// store to the slot it loads from (spec rows store token num_accepted-1's state there), and .nc
// is only defined for data that stays unwritten for the kernel's lifetime.
__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
  float4 v;
#if GDN_REC_LD_HINT == 1
  asm volatile("ld.global.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
#else
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
#endif
  return v;
}

__device__ __forceinline__ void st_f4(float4* p, const float4& v) {
#if GDN_REC_ST_HINT == 1
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
#else
  asm volatile("st.global.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
#endif
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

#ifndef GDN_REC_MINB
#define GDN_REC_MINB 8  // resident CTAs per SM the register allocation must allow
#endif

template <typename ACT, typename QT, int DK, int DVT, int LPR, int TB, int TPC>
__global__ void __launch_bounds__(DVT* LPR, GDN_REC_MINB) recurrent_kernel(const RecLaunch p) {
  static_assert(TPC == 1 || TPC == 2 || TPC == 4, "1, 2 or 4 tiles per CTA");
  constexpr int NT = DVT * LPR;
  constexpr int EPT = DK / LPR;  // fp32 state elements per thread
  constexpr int NV = EPT / 4;    // float4 words per thread
  constexpr int NWARP = NT / 32;
  constexpr int KPL = (DK + 31) / 32;  // q/k elements per lane in the norm prologue
  constexpr int TPW = (TB + NWARP - 1) / NWARP;  // tokens each warp prepares
  static_assert(EPT % 4 == 0 && NT % 32 == 0 && (LPR & (LPR - 1)) == 0, "bad tile");

  __shared__ __align__(16) float sQ[TB][DK];
  __shared__ __align__(16) float sK[TB][DK];
  __shared__ __align__(16) float sV[TB][DVT * TPC];
  __shared__ float sO[TB][DVT * TPC];
  // the states of the tiles not in registers, one slot each (each thread only touches the
  // elements it owns, so no barrier guards them)
  __shared__ __align__(16) float4 sSt[TPC > 1 ? (TPC - 1) * NV * NT : 1];
  __shared__ float sEg[TB], sBeta[TB], sKQ[TB];
  __shared__ int32_t sStore[TB], sGt[TB];

  const int tid = threadIdx.x;
  const int rr = tid / LPR;  // state row within the tile
  const int ln = tid % LPR;  // lane within the row
  const int h = blockIdx.y;
  const int kh = h / (p.Hv / p.Hk);
  const int dv0 = blockIdx.x * DVT * TPC;
  const int z = blockIdx.z;
  const int s = z < p.rows0 ? 0 : 1;
  const RowsDev R = p.sub[s];
  const int n = s == 0 ? z : z - p.rows0 + p.row_off1;
  const bool reporter = (tid == 0 && blockIdx.x == 0 && h == 0);

  // The prior state is the long pole: resolve its slot with as few dependent loads as possible
  // (num_accepted -> spec_state_indices) and issue it before the row's token range is checked.
  // Reading a valid slot is harmless even when the row turns out to be skipped.
  const int32_t bos = __ldg(R.qsl + n), eos = __ldg(R.qsl + n + 1);
  int load_slot = 0, na = 1;
  bool read_prior, bad_accept = false;
  if (R.is_spec) {
    na = __ldg(R.num_acc + n);
    const bool na_ok = na >= 1 && na <= R.spec_cols;
    load_slot = na_ok ? __ldg(R.spec_idx + (int64_t)n * R.spec_cols + na - 1) : 0;
    read_prior = load_slot > 0;
  } else {
    load_slot = __ldg(R.state_idx + n);
    if (R.num_acc) {  // acceptance-aware row: the slot of its last accepted token
      const int a = __ldg(R.num_acc + n);
      bad_accept = a < 1 || a > R.spec_cols;
      load_slot = bad_accept ? 0 : __ldg(R.spec_idx + (int64_t)n * R.spec_cols + a - 1);
    }
    read_prior = load_slot > 0 && (R.has_init == nullptr || __ldg(R.has_init + n) != 0);
  }
  const bool slot_ok = load_slot < p.num_slots;
  read_prior = read_prior && slot_ok;

  const int64_t head_elems = (int64_t)p.dv * DK;
  const int64_t row_off = ((int64_t)h * p.dv + dv0 + rr) * DK;  // within one slot
  const int64_t slot_elems = (int64_t)p.Hv * head_elems;

  // 1. prior state -> registers (streaming loads, issued first); a second tile's state goes to
  //    shared memory through cp.async, in flight during the token preparation
  float4 S[NV];
  if (read_prior) {
    const float4* src = reinterpret_cast<const float4*>(p.ssm_pool + load_slot * slot_elems + row_off) + ln;
#pragma unroll
    for (int i = 0; i < NV; ++i) S[i] = ld_stream_f4(src + i * LPR);
    if constexpr (TPC > 1) {
#pragma unroll
      for (int k = 0; k < TPC - 1; ++k)
#pragma unroll
        for (int i = 0; i < NV; ++i)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(
                           &sSt[(k * NV + i) * NT + tid])),
                       "l"(src + (int64_t)(k + 1) * DVT * DK / 4 + i * LPR)
                       : "memory");
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  } else {
#pragma unroll
    for (int i = 0; i < NV; ++i) S[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (TPC > 1) {
#pragma unroll
      for (int i = 0; i < (TPC - 1) * NV; ++i) sSt[i * NT + tid] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // tile_at[0]: the tile whose state is in registers; tile_at[k]: the tile in slot k - 1
  int tile_at[TPC];
#pragma unroll
  for (int k = 0; k < TPC; ++k) tile_at[k] = k;

  // row checks (the loads above stay in flight)
  int L = eos - bos;
  uint32_t skip = 0;
  if (bos < 0 || eos < bos || eos > R.num_tokens) skip = GDN_STATUS_ROW_RANGE;
  else if (L == 0) skip = 0x80000000u;
  else if (R.is_spec && L > R.spec_cols) skip = GDN_STATUS_ROW_RANGE;
  else if (R.is_spec && (na < 1 || na > R.spec_cols)) skip = GDN_STATUS_NUM_ACCEPTED;
  else if (bad_accept) skip = GDN_STATUS_NUM_ACCEPTED;
  if (skip) {
    if (reporter && skip != 0x80000000u) set_status(p.status, skip);
    if constexpr (TPC > 1) asm volatile("cp.async.wait_all;" ::: "memory");  // no copy outlives the CTA
    return;
  }
  if (!slot_ok && reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);

  const QT* __restrict__ qkv = static_cast<const QT*>(p.qkv[s]);
  const ACT* __restrict__ ga = static_cast<const ACT*>(p.a);
  const ACT* __restrict__ gb = static_cast<const ACT*>(p.b);
  ACT* __restrict__ out = static_cast<ACT*>(p.out);
  const int warp = tid / 32, lane = tid % 32;
  const float neg_A = -expf(__ldg(p.A_log + h));
  const float dtb = __ldg(p.dt_bias + h);

  // Gate inputs, global tokens and store slots of a token batch, through lane 0 of each token's
  // warp (warp w takes tokens w, w+NWARP, ...).  None of them comes from the conv grid: the
  // first batch's token indices and store slots are loaded before the wait for that grid (not
  // used until after it, so nothing stalls on them there), the gate inputs they address right
  // after the q|k|v copies are issued.
  float av[TPW], bv[TPW];
  int gt_[TPW], ss_[TPW];
  auto load_tokens = [&](int tb0, int nt) {
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int t = warp + u * NWARP;
      gt_[u] = -1;
      ss_[u] = -1;
      if (t < nt && lane == 0) {
        const int32_t i = bos + tb0 + t;
        gt_[u] = R.tok ? __ldg(R.tok + i) : i;
        if (R.is_spec) ss_[u] = __ldg(R.spec_idx + (int64_t)n * R.spec_cols + tb0 + t);
      }
    }
  };
  auto load_gates = [&](int nt) {
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int t = warp + u * NWARP;
      av[u] = bv[u] = 0.f;
      if (t < nt && lane == 0) {
        int gt = gt_[u];
        if (gt < 0 || gt >= p.num_global) {
          set_status(p.status, GDN_STATUS_TOKEN_RANGE);
          gt = -1;
        }
        gt_[u] = gt;
        if (gt >= 0) {
          av[u] = to_f32(ga[(int64_t)gt * p.Hv + h]);
          bv[u] = to_f32(gb[(int64_t)gt * p.Hv + h]);
        }
      }
    }
  };
  load_tokens(0, min(TB, L));

  // q|k|v may come from the conv grid launched just before (programmatic dependent launch):
  // everything above touched only the state pool, the gates and metadata; wait for that grid.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int tb0 = 0; tb0 < L; tb0 += TB) {
    const int nt = min(TB, L - tb0);
    if (tb0) __syncthreads();  // previous batch's shared data fully consumed

    // 2a. every load of the token preparation is issued at once, so the preparation costs one
    //     round trip: raw q and k rows and this tile's v slice land in shared memory through
    //     cp.async (no registers held), the gate inputs and store slots through lane 0 of each
    //     token's warp.  Warp w prepares tokens w, w+NWARP, ...
    if constexpr (sizeof(QT) == 4 && DK % 4 == 0 && (DVT * TPC) % 4 == 0) {
      constexpr int QC = DK / 4, VC = DVT * TPC / 4;  // 16-byte chunks per q/k row and per v slice
      for (int idx = tid; idx < nt * (2 * QC + VC); idx += NT) {
        const int t = idx / (2 * QC + VC), c = idx % (2 * QC + VC);
        const int64_t i = bos + tb0 + t;
        const QT* src;
        float* dst;
        if (c < QC) {
          src = qkv + i * p.C + (int64_t)kh * DK + 4 * c;
          dst = &sQ[t][4 * c];
        } else if (c < 2 * QC) {
          src = qkv + i * p.C + (int64_t)p.Hk * DK + (int64_t)kh * DK + 4 * (c - QC);
          dst = &sK[t][4 * (c - QC)];
        } else {
          src = qkv + i * p.C + 2LL * p.Hk * DK + (int64_t)h * p.dv + dv0 + 4 * (c - 2 * QC);
          dst = &sV[t][4 * (c - 2 * QC)];
        }
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                     "l"(src)
                     : "memory");
      }
    } else {
      for (int idx = tid; idx < nt * (2 * DK + DVT * TPC); idx += NT) {
        const int t = idx / (2 * DK + DVT * TPC), c = idx % (2 * DK + DVT * TPC);
        const int64_t i = bos + tb0 + t;
        if (c < DK) sQ[t][c] = to_f32(qkv[i * p.C + (int64_t)kh * DK + c]);
        else if (c < 2 * DK) sK[t][c - DK] = to_f32(qkv[i * p.C + (int64_t)p.Hk * DK + (int64_t)kh * DK + c - DK]);
        else sV[t][c - 2 * DK] = to_f32(qkv[i * p.C + 2LL * p.Hk * DK + (int64_t)h * p.dv + dv0 + c - 2 * DK]);
      }
    }
    if (tb0) load_tokens(tb0, nt);
    load_gates(nt);
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // 2b. the arithmetic, in place: L2-normalised q^ (scaled), k^, k^.q^, gates, slots
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int t = warp + u * NWARP;
      if (t >= nt) continue;
      float qv[KPL], kv[KPL], sq = 0.f, sk = 0.f;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const int c = lane + 32 * j;
        qv[j] = c < DK ? sQ[t][c] : 0.f;
        kv[j] = c < DK ? sK[t][c] : 0.f;
        sq = fmaf(qv[j], qv[j], sq);
        sk = fmaf(kv[j], kv[j], sk);
      }
      sq = warp_sum(sq);
      sk = warp_sum(sk);
      const float rq = 1.0f / sqrtf(sq + 1e-6f), rk = 1.0f / sqrtf(sk + 1e-6f);
      float kq = 0.f;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        const int c = lane + 32 * j;
        if (c < DK) {
          const float qn = qv[j] * rq * p.scale, kn = kv[j] * rk;
          sQ[t][c] = qn;
          sK[t][c] = kn;
          kq = fmaf(qn, kn, kq);
        }
      }
      kq = warp_sum(kq);
      if (lane == 0) {
        sKQ[t] = kq;
        sGt[t] = gt_[u];
        const float xs = av[u] + dtb;
        const float sp = xs > 20.f ? xs : log1pf(expf(xs));
        sEg[t] = expf(neg_A * sp);
        sBeta[t] = 1.0f / (1.0f + expf(-bv[u]));
        int ss = ss_[u];
        if (ss >= p.num_slots) {
          set_status(p.status, GDN_STATUS_SLOT_RANGE);
          ss = 0;
        }
        sStore[t] = ss;
      }
    }
    __syncthreads();

    // 3. the recurrence, token by token, for the tile in registers and then for each other
    //    tile, swapped in from its shared-memory slot
#pragma unroll
    for (int pass = 0; pass < TPC; ++pass) {
      if (pass > 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const float4 o = sSt[((pass - 1) * NV + i) * NT + tid];
          sSt[((pass - 1) * NV + i) * NT + tid] = S[i];
          S[i] = o;
        }
        const int t_ = tile_at[0];
        tile_at[0] = tile_at[pass];
        tile_at[pass] = t_;
      }
      const int col = tile_at[0] * DVT + rr;  // this thread's state row among the CTA's rows
      const int64_t tile_off = row_off + (int64_t)tile_at[0] * DVT * DK;
      for (int t = 0; t < nt; ++t) {
        const float4* k4 = reinterpret_cast<const float4*>(sK[t]) + ln;
        const float4* q4 = reinterpret_cast<const float4*>(sQ[t]) + ln;
        float dk_ = 0.f, dq_ = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const float4 kf = k4[i * LPR], qf = q4[i * LPR];
          dk_ = fmaf(S[i].x, kf.x, fmaf(S[i].y, kf.y, fmaf(S[i].z, kf.z, fmaf(S[i].w, kf.w, dk_))));
          dq_ = fmaf(S[i].x, qf.x, fmaf(S[i].y, qf.y, fmaf(S[i].z, qf.z, fmaf(S[i].w, qf.w, dq_))));
        }
#pragma unroll
        for (int o = LPR / 2; o >= 1; o >>= 1) {
          dk_ += __shfl_xor_sync(0xffffffffu, dk_, o);
          dq_ += __shfl_xor_sync(0xffffffffu, dq_, o);
        }
        const float eg = sEg[t], beta = sBeta[t];
        const float delta = beta * (sV[t][col] - eg * dk_);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const float4 kf = k4[i * LPR];
          S[i].x = fmaf(delta, kf.x, eg * S[i].x);
          S[i].y = fmaf(delta, kf.y, eg * S[i].y);
          S[i].z = fmaf(delta, kf.z, eg * S[i].z);
          S[i].w = fmaf(delta, kf.w, eg * S[i].w);
        }
        if (ln == 0) sO[t][col] = fmaf(delta, sKQ[t], eg * dq_);
        const int ss = sStore[t];
        if (ss > 0) {
          float4* dst = reinterpret_cast<float4*>(p.ssm_pool + ss * slot_elems + tile_off) + ln;
#pragma unroll
          for (int i = 0; i < NV; ++i) st_f4(dst + i * LPR, S[i]);
        }
      }
    }
    __syncthreads();

    // 4. outputs, scattered to the tokens' global positions
    for (int idx = tid; idx < nt * DVT * TPC; idx += NT) {
      const int t = idx / (DVT * TPC), r = idx % (DVT * TPC);
      const int gt = sGt[t];
      if (gt >= 0) out[((int64_t)gt * p.Hv + h) * p.dv + dv0 + r] = from_f32<ACT>(sO[t][r]);
    }
  }

  if (!R.is_spec) {
    const int ss = __ldg(R.state_idx + n);
    if (ss >= p.num_slots) {
      if (reporter) set_status(p.status, GDN_STATUS_SLOT_RANGE);
    } else if (ss > 0) {
      float4* dst = reinterpret_cast<float4*>(p.ssm_pool + ss * slot_elems + row_off + (int64_t)tile_at[0] * DVT * DK) + ln;
#pragma unroll
      for (int i = 0; i < NV; ++i) st_f4(dst + i * LPR, S[i]);
#pragma unroll
      for (int k = 1; k < TPC; ++k) {  // the other tiles, from their slots
        dst = reinterpret_cast<float4*>(p.ssm_pool + ss * slot_elems + row_off + (int64_t)tile_at[k] * DVT * DK) + ln;
#pragma unroll
        for (int i = 0; i < NV; ++i) st_f4(dst + i * LPR, sSt[((k - 1) * NV + i) * NT + tid]);
      }
    }
  }
}

#ifndef GDN_REC_TPC
#define GDN_REC_TPC 2  // most tiles of state rows per CTA (they share one token preparation)
#endif
#ifndef GDN_REC_DVT
#define GDN_REC_DVT 16  // state rows per CTA
#endif
#ifndef GDN_REC_LPR
#define GDN_REC_LPR 8  // lanes per state row (16 fp32 each at dk = 128)
#endif

template <typename ACT, typename QT, int DK, int DVT, int TPC>
static cudaError_t launch_tile(const RecLaunch& p, int rows, bool pdl, cudaStream_t s) {
  constexpr int LPR = (DK / GDN_REC_LPR >= 4) ? GDN_REC_LPR : DK / 4;
  constexpr int TB = 8;
  const int tiles = p.dv / (DVT * TPC);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, p.Hv, rows);
  cfg.blockDim = dim3(DVT * LPR);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  int na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, recurrent_kernel<ACT, QT, DK, DVT, LPR, TB, TPC>, p);
}

// As many tiles per CTA (up to GDN_REC_TPC) as dv holds evenly: one token preparation serves
// them all.
template <typename ACT, typename QT, int DK>
static cudaError_t launch_dv(const RecLaunch& p, int rows, bool pdl, cudaStream_t s) {
  if (GDN_REC_TPC >= 4 && p.dv % (4 * GDN_REC_DVT) == 0) return launch_tile<ACT, QT, DK, GDN_REC_DVT, 4>(p, rows, pdl, s);
  if (GDN_REC_TPC >= 2 && p.dv % (2 * GDN_REC_DVT) == 0) return launch_tile<ACT, QT, DK, GDN_REC_DVT, 2>(p, rows, pdl, s);
  if (p.dv % GDN_REC_DVT == 0) return launch_tile<ACT, QT, DK, GDN_REC_DVT, 1>(p, rows, pdl, s);
  return launch_tile<ACT, QT, DK, 16, 1>(p, rows, pdl, s);
}

template <typename ACT, typename QT>
static cudaError_t launch_dk(const RecLaunch& p, int rows, bool pdl, cudaStream_t s) {
  switch (p.dk) {
    case 16: return launch_dv<ACT, QT, 16>(p, rows, pdl, s);
    case 32: return launch_dv<ACT, QT, 32>(p, rows, pdl, s);
    case 64: return launch_dv<ACT, QT, 64>(p, rows, pdl, s);
    case 128: return launch_dv<ACT, QT, 128>(p, rows, pdl, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_recurrent(const RecLaunch& p, gdn_dtype act, gdn_dtype qkv_dtype, int rows_total, bool pdl,
                             cudaStream_t s) {
  if (rows_total <= 0) return cudaSuccess;
  cudaError_t e;
  if (act == GDN_BF16)
    e = qkv_dtype == GDN_F32 ? launch_dk<__nv_bfloat16, float>(p, rows_total, pdl, s)
                             : launch_dk<__nv_bfloat16, __nv_bfloat16>(p, rows_total, pdl, s);
  else
    e = qkv_dtype == GDN_F32 ? launch_dk<float, float>(p, rows_total, pdl, s)
                             : launch_dk<float, __nv_bfloat16>(p, rows_total, pdl, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gdn
