// gdn_prefill.cu -- chunked prefill of the gated delta rule on tcgen05 tensor cores.
//
// The pages run prefill rows through a chunked gated-delta-rule kernel ("[XE2] Support MTP of
// QWEN model", Copilot overview: XE2 chunk gated delta rule with token-remapped output writes).
// The chunk form used here is the WY / UT-transform form of the same recurrence (Yang et al.,
// "Parallelizing Linear Transformers with the Delta Rule over Sequence Length", 2024; Yang, Kautz
// and Hatamizadeh, "Gated Delta Networks", 2025).  For a chunk of c tokens with state S_0
// (dv x dk), cumulative log-decay G_t = g_1 + .. + g_t, gamma_t = e^{G_t}:
//   A[t,s] = beta_t e^{G_t - G_s} (k_t . k_s) for s < t,   T = (I + A)^-1      (unit lower)
//   W = T diag(beta gamma) K,   U~ = T diag(beta) V                           (S-independent)
//   U = U~ - W S_0^T,   O = diag(gamma) Q S_0^T + P U,  P[t,s] = e^{G_t - G_s} (q_t . k_s), s <= t
//   S_c = gamma_c S_0 + U^T K',   K'_s = e^{G_c - G_s} k_s
// Everything that does not depend on S_0 is computed for all chunks at once by the prep kernel
// (one CTA per (row, chunk, v-head)); the scan kernel (one CTA per (row, v-head)) walks the
// chunks in order, keeping the fp32 state in tensor memory.
//
// Tensor cores.  Every product is a tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulation)
// issued by one thread, with operands in 128B-swizzled shared memory and accumulators in TMEM.
// Products that reach the state use a bf16 hi/lo split of both operands and three MMAs (about
// 1e-5 relative error); the output-only products (S q and U P) use one.  All MMAs have M = 128:
// they are arranged so the 128 rows are the head dimension or [q; k] stacked, e.g. W^T =
// (beta gamma K)^T T^T.  The scan kernel's chunk inputs are written by the prep kernel as exact
// shared-memory images and arrive with one bulk copy, prefetched while the previous chunk's
// outputs are drained; its MMAs are committed in the order the state needs them (U, then the
// state update, then the output), so the state readback never waits on output work.  T is
// solved column by column on the CUDA cores.
//
// Path limits: dk = dv = 128 and bf16 activations; other shapes use the token recurrence.
// Every wait on an mbarrier is bounded; a timeout sets GDN_STATUS_WAIT_TIMEOUT, drains, frees
// TMEM and returns.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"

namespace gdn {

namespace {

constexpr int kCh = kPrefillChunk;  // tokens per chunk
constexpr int kD = 128;             // dk = dv on this path

// Per (chunk, v-head) record written by the prep kernel, read by the scan kernel.
constexpr uint32_t kWnHi = 0;       // -W   [t][dk]  bf16 hi image (K-major, 2 atoms)   16 KiB
constexpr uint32_t kWnLo = 16384;   //               bf16 lo image                       16 KiB
constexpr uint32_t kKpHi = 32768;   // K'^T [dk][s]  bf16 hi image (1 atom)               16 KiB
constexpr uint32_t kKpLo = 49152;   //               bf16 lo image                       16 KiB
constexpr uint32_t kQp = 65536;     // gamma q^ [t][dk] bf16 image                       16 KiB
constexpr uint32_t kP = 81920;      // P    [t][s]   bf16 image                           8 KiB
constexpr uint32_t kImgBytes = 90112;  // the images above: one bulk copy
constexpr uint32_t kUt = 90112;     // U~   [t][dv]  fp32                                32 KiB
constexpr uint32_t kMeta = 122880;  // gamma_c (fp32)
constexpr uint32_t kScanCopy = kMeta + 16;  // what the scan kernel copies per chunk
static_assert(kRecBytes >= kScanCopy && kUt == kImgBytes, "record layout");

constexpr int kPrepSmem = 81920 + 1024;
constexpr int kScanSmem = 98304 + (int)kScanCopy + 1024;

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float warp_sum32(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 4 consecutive values of row r starting at column k (k % 4 == 0) as bf16 hi/lo into two images.
__device__ __forceinline__ void put4_pair(uint8_t* hi_img, uint8_t* lo_img, int r, int k, int kb, const float* x) {
  __nv_bfloat16 h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[i] = __float2bfloat16_rn(x[i]);
    l[i] = __float2bfloat16_rn(x[i] - __bfloat162float(h[i]));
  }
  const uint32_t off = tc::img_off(r, k, kb);
  *reinterpret_cast<uint2*>(hi_img + off) = *reinterpret_cast<const uint2*>(h);
  *reinterpret_cast<uint2*>(lo_img + off) = *reinterpret_cast<const uint2*>(l);
}

__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
  const float x = a + dt_bias;
  return -expf(A_log) * (x > 20.f ? x : log1pf(expf(x)));
}

// ------------------------------------------------------------------------------------------
// Prep: one CTA per (row, chunk, v-head); 128 threads.
template <typename QT>
__global__ void __launch_bounds__(128) chunk_prep_kernel(const PrefillLaunch p) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = align1k(dyn_smem);
  uint8_t* qk_hi = sm;  // [q^; k^] [128][128] images (MMA 1)
  uint8_t* qk_lo = sm + 32768;
  float* sA = reinterpret_cast<float*>(sm);           // A [64][65]      (after MMA 1)
  float* sT = reinterpret_cast<float*>(sm + 16640);   // T [64][65]
  uint8_t* kb_hi = sm;  // (beta gamma k^)^T [128][64]  (after T is imaged)
  uint8_t* kb_lo = sm + 16384;
  uint8_t* vb_hi = sm + 32768;  // (beta v)^T [128][64]
  uint8_t* vb_lo = sm + 49152;
  uint8_t* t_hi = sm + 65536;  // T [64][64]
  uint8_t* t_lo = sm + 73728;
  __shared__ float sG[kCh], sBeta[kCh], sRk[kCh];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y;
  const int kh = h / (p.Hv / p.Hk);
  int n, c;
  if (!locate_unit(p.rows, p.first_row, p.num_rows, kCh, blockIdx.x, n, c, p.status)) return;
  const int bos = __ldg(p.rows.qsl + n);
  const int L = __ldg(p.rows.qsl + n + 1) - bos;
  const int t0 = c * kCh, nc = min(kCh, L - t0);
  uint8_t* rec = p.ws + ((size_t)blockIdx.x * p.Hv + h) * kRecBytes;
  const QT* qkv = static_cast<const QT*>(p.qkv);
  const int64_t C = p.C;
  const int qoff = kh * kD, koff = p.Hk * kD + kh * kD, voff = 2 * p.Hk * kD + h * kD;

  // 1. gates (padded tokens: g = 0, beta = 0), TMEM and barrier
  if (tid < kCh) {
    float g = 0.f, beta = 0.f;
    if (tid < nc) {
      const int gt = global_token(p.rows, bos + t0 + tid, p.num_global, p.status);
      if (gt >= 0) {
        const __nv_bfloat16* ga = static_cast<const __nv_bfloat16*>(p.a);
        const __nv_bfloat16* gb = static_cast<const __nv_bfloat16*>(p.b);
        g = gate_g(__bfloat162float(ga[(int64_t)gt * p.Hv + h]), __ldg(p.A_log + h), __ldg(p.dt_bias + h));
        beta = 1.f / (1.f + expf(-__bfloat162float(gb[(int64_t)gt * p.Hv + h])));
      }
    }
    sG[tid] = g;
    sBeta[tid] = beta;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
  if (tid == 32) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    float acc = 0.f;
    for (int t = 0; t < kCh; ++t) {
      acc += sG[t];
      sG[t] = acc;  // G_t, inclusive
    }
  }
  __syncthreads();

  // 2. q^ (scaled) and k^ rows of the [q^; k^] images, and the gamma q^ record rows; warp w
  //    takes tokens 16w .. 16w+15, four at a time so their loads are in flight together
  for (int i0 = 0; i0 < 16; i0 += 4) {
    float q[4][4], k[4][4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int t = warp * 16 + i0 + b;
#pragma unroll
      for (int e = 0; e < 4; ++e) q[b][e] = k[b][e] = 0.f;
      if (t < nc) {
        const QT* row = qkv + (int64_t)(bos + t0 + t) * C;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          q[b][e] = to_f32(row[qoff + 4 * lane + e]);
          k[b][e] = to_f32(row[koff + 4 * lane + e]);
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int t = warp * 16 + i0 + b;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sq = fmaf(q[b][e], q[b][e], sq);
        sk = fmaf(k[b][e], k[b][e], sk);
      }
      sq = warp_sum32(sq);
      sk = warp_sum32(sk);
      const float rq = 1.0f / sqrtf(sq + 1e-6f), rk = 1.0f / sqrtf(sk + 1e-6f);
      if (lane == 0) sRk[t] = rk;
      const float gam = expf(sG[t]);
      float qn[4], kn[4], qg[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qn[e] = q[b][e] * rq * p.scale;
        kn[e] = k[b][e] * rk;
        qg[e] = gam * qn[e];
      }
      put4_pair(qk_hi, qk_lo, t, 4 * lane, 2, qn);
      put4_pair(qk_hi, qk_lo, kCh + t, 4 * lane, 2, kn);
      __nv_bfloat16 hq[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) hq[e] = __float2bfloat16_rn(qg[e]);
      *reinterpret_cast<uint2*>(rec + kQp + tc::img_off(t, 4 * lane, 2)) = *reinterpret_cast<const uint2*>(hq);
    }
  }
  tc::fence_async_smem();
  tc::fence_before();
  __syncthreads();

  // 3. MMA 1: D1 (columns 0..63) = [q^; k^] k^T, three passes
  if (tid == 0) {
    tc::fence_after();
    const uint32_t id = tc::idesc_bf16(128, 64);
    const uint32_t ah = tc::smem_addr(qk_hi), al = tc::smem_addr(qk_lo);
    for (int s = 0; s < 8; ++s) {
      const uint32_t off = (s >> 2) * 1024 + (s & 3) * 32;
      tc::mma3(tmem, tc::sdesc(ah + off, 2048), tc::sdesc(al + off, 2048), tc::sdesc(ah + 16384 + off, 2048),
               tc::sdesc(al + 16384 + off, 2048), id, s == 0);
    }
    tc::commit(&bar);
  }
  bool ok = __syncthreads_and(tc::mbar_wait(&bar, 0));
  if (ok) {
    tc::fence_after();
    // 4. P rows to the record (warps 0, 1: q rows); A rows to shared memory (warps 2, 3: k rows)
    float v0[32], v1[32];
    tc::tmem_ld32(tc::tmem_lane_col(tmem, warp, 0), v0);
    tc::tmem_ld32(tc::tmem_lane_col(tmem, warp, 32), v1);
    const int t = (warp & 1) * 32 + lane;
    const float Gt = sG[t];
    if (warp < 2) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = 8 * j + e;
          const float qk = s < 32 ? v0[s & 31] : v1[s & 31];
          x[e] = s <= t ? expf(Gt - sG[s]) * qk : 0.f;
        }
        *reinterpret_cast<uint4*>(rec + kP + tc::img_off(t, 8 * j, 1)) = tc::pack8(x);
      }
    } else {
      const float bt = sBeta[t];
#pragma unroll
      for (int s = 0; s < kCh; ++s) {
        const float kk = s < 32 ? v0[s & 31] : v1[s & 31];
        sA[t * 65 + s] = s < t ? bt * expf(Gt - sG[s]) * kk : 0.f;
      }
    }
    __syncthreads();

    // 5. T = (I + A)^-1, column s by thread s: T[t][s] = -sum_{s<=j<t} A[t][j] T[j][s]
    if (tid < kCh) {
      const int s = tid;
      for (int t2 = 0; t2 < s; ++t2) sT[t2 * 65 + s] = 0.f;
      sT[s * 65 + s] = 1.f;
      for (int t2 = s + 1; t2 < kCh; ++t2) {
        float acc0 = 0.f, acc1 = 0.f;
        int j = s;
        for (; j + 1 < t2; j += 2) {
          acc0 = fmaf(sA[t2 * 65 + j], sT[j * 65 + s], acc0);
          acc1 = fmaf(sA[t2 * 65 + j + 1], sT[(j + 1) * 65 + s], acc1);
        }
        if (j < t2) acc0 = fmaf(sA[t2 * 65 + j], sT[j * 65 + s], acc0);
        sT[t2 * 65 + s] = -(acc0 + acc1);
      }
    }
    __syncthreads();
    // 6a. T image (rows t, K = s): thread -> row tid/2, 32 columns
    {
      const int tt = tid >> 1, s0 = (tid & 1) * 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = sT[tt * 65 + s0 + 8 * j + e];
        uint4 hi, lo;
        tc::split8(x, hi, lo);
        const uint32_t off = tc::img_off(tt, s0 + 8 * j, 1);
        *reinterpret_cast<uint4*>(t_hi + off) = hi;
        *reinterpret_cast<uint4*>(t_lo + off) = lo;
      }
    }
    __syncthreads();  // T consumed; the region is reused below
    // 6b. (beta gamma k^)^T and (beta v)^T images (shared memory) and the K'^T record images,
    //     row d = tid; the column loads of 16 tokens are issued together
    {
      const int d = tid;
      const float Gc = sG[kCh - 1];
#pragma unroll 1
      for (int s0 = 0; s0 < kCh; s0 += 16) {
        float kr[16], vr[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int s = s0 + e;
          kr[e] = vr[e] = 0.f;
          if (s < nc) {
            const QT* row = qkv + (int64_t)(bos + t0 + s) * C;
            kr[e] = to_f32(row[koff + d]);
            vr[e] = to_f32(row[voff + d]);
          }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float xk[8], xv[8], xp[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int s = s0 + 8 * half + e;
            const float kn = kr[8 * half + e] * sRk[s], bs = sBeta[s];
            xk[e] = bs * expf(sG[s]) * kn;
            xv[e] = bs * vr[8 * half + e];
            xp[e] = s < nc ? expf(Gc - sG[s]) * kn : 0.f;
          }
          uint4 hi, lo;
          const uint32_t off = tc::img_off(d, s0 + 8 * half, 1);
          tc::split8(xk, hi, lo);
          *reinterpret_cast<uint4*>(kb_hi + off) = hi;
          *reinterpret_cast<uint4*>(kb_lo + off) = lo;
          tc::split8(xv, hi, lo);
          *reinterpret_cast<uint4*>(vb_hi + off) = hi;
          *reinterpret_cast<uint4*>(vb_lo + off) = lo;
          tc::split8(xp, hi, lo);
          *reinterpret_cast<uint4*>(rec + kKpHi + off) = hi;
          *reinterpret_cast<uint4*>(rec + kKpLo + off) = lo;
        }
      }
      if (tid == 0) *reinterpret_cast<float*>(rec + kMeta) = expf(Gc);
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();

    // 7. MMA 2, 3: W^T (cols 64..127) = (beta gamma k^)^T T^T;  U~^T (cols 128..191) = (beta v)^T T^T
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id = tc::idesc_bf16(128, 64);
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = s * 32;
        const uint64_t th = tc::sdesc(tc::smem_addr(t_hi) + off, 1024), tl = tc::sdesc(tc::smem_addr(t_lo) + off, 1024);
        tc::mma3(tmem + 64, tc::sdesc(tc::smem_addr(kb_hi) + off, 1024), tc::sdesc(tc::smem_addr(kb_lo) + off, 1024),
                 th, tl, id, s == 0);
        tc::mma3(tmem + 128, tc::sdesc(tc::smem_addr(vb_hi) + off, 1024), tc::sdesc(tc::smem_addr(vb_lo) + off, 1024),
                 th, tl, id, s == 0);
      }
      tc::commit(&bar);
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar, 1));
    if (ok) {
      tc::fence_after();
      // 8. -W (hi/lo images, staged in shared memory) and U~ (fp32) from TMEM, lane = row d
      const int d = 32 * warp + lane;
      uint8_t* wn_hi = sm;  // the MMA 2/3 operands are consumed: reuse their space
      uint8_t* wn_lo = sm + 16384;
      float* ut = reinterpret_cast<float*>(rec + kUt);
      for (int half = 0; half < 2; ++half) {
        float w[32];
        tc::tmem_ld32(tc::tmem_lane_col(tmem, warp, 64 + 32 * half), w);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = -w[i];
          const __nv_bfloat16 hi = __float2bfloat16_rn(x);
          const __nv_bfloat16 lo = __float2bfloat16_rn(x - __bfloat162float(hi));
          const uint32_t off = tc::img_off(32 * half + i, d, 2);
          *reinterpret_cast<__nv_bfloat16*>(wn_hi + off) = hi;
          *reinterpret_cast<__nv_bfloat16*>(wn_lo + off) = lo;
        }
        tc::tmem_ld32(tc::tmem_lane_col(tmem, warp, 128 + 32 * half), w);
#pragma unroll
        for (int i = 0; i < 32; ++i) ut[(32 * half + i) * kD + d] = w[i];
      }
      __syncthreads();
      const uint4* src = reinterpret_cast<const uint4*>(sm);
      uint4* dst = reinterpret_cast<uint4*>(rec + kWnHi);
#pragma unroll 4
      for (int i = tid; i < 32768 / 16; i += 128) dst[i] = src[i];
    }
  }
  if (!ok) {
    if (tid == 0) set_status(p.status, GDN_STATUS_WAIT_TIMEOUT);
    tc::mbar_wait(&bar, 0);  // bounded: let any issued MMA drain before TMEM is released
    tc::mbar_wait(&bar, 1);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------------------------------
// Scan: one CTA per (row, v-head); 128 threads, thread d owns row d of the state.
__global__ void __launch_bounds__(128, 1) chunk_scan_kernel(const PrefillLaunch p) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = align1k(dyn_smem);
  uint8_t* s_hi = sm;  // S [dv][dk] images (A operand), 32 KiB each
  uint8_t* s_lo = sm + 32768;
  uint8_t* u_hi = sm + 65536;  // U^T [dv][s] images, 16 KiB each; then the output staging
  uint8_t* u_lo = sm + 81920;
  uint8_t* ops = sm + 98304;  // the chunk record: images, U~, gamma_c (kScanCopy bytes)
  __nv_bfloat16* o_stage = reinterpret_cast<__nv_bfloat16*>(u_hi);  // [t][dv]
  __shared__ __align__(8) uint64_t bar_mma, bar_tma;
  __shared__ uint32_t tmem_base;
  __shared__ int sGt[kCh];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x;
  const int n = p.first_row + blockIdx.y;
  const int base_unit = units_before(p.rows, p.first_row, n, kCh);
  const int bos = __ldg(p.rows.qsl + n), eos = __ldg(p.rows.qsl + n + 1);
  if (bos < 0 || eos < bos || eos > p.rows.num_tokens || eos == bos) return;  // malformed rows flagged by prep
  const int L = eos - bos;
  const int nch = (L + kCh - 1) / kCh;
  int slot = __ldg(p.rows.state_idx + n);
  const int load_slot = non_spec_load_slot(p.rows, n);
  if (load_slot < 0) {  // acceptance-aware row with num_accepted out of range
    if (tid == 0 && h == 0) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
    return;
  }
  bool read_prior = load_slot > 0 && (p.rows.has_init == nullptr || __ldg(p.rows.has_init + n) != 0);
  if (slot >= p.num_slots || load_slot >= p.num_slots) {
    if (tid == 0 && h == 0) set_status(p.status, GDN_STATUS_SLOT_RANGE);
    if (slot >= p.num_slots) slot = 0;
    read_prior = false;
  }
  const int d = 32 * warp + lane;
  float* gS = p.ssm_pool + ((int64_t)slot * p.Hv + h) * kD * kD + (int64_t)d * kD;
  const float* gS0 = p.ssm_pool + ((int64_t)(read_prior ? load_slot : 0) * p.Hv + h) * kD * kD + (int64_t)d * kD;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);

  if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
  if (tid == 32) {
    tc::mbar_init(&bar_mma, 1);
    tc::mbar_init(&bar_tma, 1);
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tS = tmem_base, tU = tmem_base + 128, tO = tmem_base + 192;
  auto record = [&](int c) { return p.ws + ((size_t)(base_unit + c) * p.Hv + h) * kRecBytes; };

  // initial state: fp32 master in TMEM (lane d) and its hi/lo images (row d)
  for (int c0 = 0; c0 < kD; c0 += 32) {
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      float4 f = read_prior ? *reinterpret_cast<const float4*>(gS0 + c0 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j] = f.x; v[j + 1] = f.y; v[j + 2] = f.z; v[j + 3] = f.w;
    }
    tc::tmem_st32(tc::tmem_lane_col(tS, warp, c0), v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 hi, lo;
      tc::split8(v + 8 * j, hi, lo);
      const uint32_t off = tc::img_off(d, c0 + 8 * j, 2);
      *reinterpret_cast<uint4*>(s_hi + off) = hi;
      *reinterpret_cast<uint4*>(s_lo + off) = lo;
    }
  }
  tc::tmem_st_wait();
  tc::fence_async_smem();
  if (tid == 0) {
    tc::expect_tx(&bar_tma, kScanCopy);
    tc::bulk_g2s(ops, record(0), kScanCopy, &bar_tma);
  }

  bool ok = true;
  uint32_t tma_phase = 0, mma_phase = 0;
  for (int c = 0; c < nch && ok; ++c) {
    if (tid < kCh) {
      const int t = c * kCh + tid;
      sGt[tid] = t < L ? global_token(p.rows, bos + t, p.num_global, p.status) : -1;
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar_tma, tma_phase));
    tma_phase ^= 1;
    if (!ok) break;
    // U accumulator <- U~^T (row d), and S <- gamma_c S (this chunk's MMAs read the old S images)
    {
      const float gamma_c = *reinterpret_cast<const float*>(ops + kMeta);
      const float* ut = reinterpret_cast<const float*>(ops + kUt);
      for (int half = 0; half < 2; ++half) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = ut[(32 * half + i) * kD + d];
        tc::tmem_st32(tc::tmem_lane_col(tU, warp, 32 * half), v);
      }
      for (int c0 = 0; c0 < kD; c0 += 32) {
        float v[32];
        tc::tmem_ld32(tc::tmem_lane_col(tS, warp, c0), v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= gamma_c;
        tc::tmem_st32(tc::tmem_lane_col(tS, warp, c0), v);
      }
      tc::tmem_st_wait();
    }
    tc::fence_before();
    __syncthreads();
    // U^T += S (-W)^T (three passes) -> commit;  O^T = S q'^T
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id64 = tc::idesc_bf16(128, 64);
      const uint32_t sh = tc::smem_addr(s_hi), sl = tc::smem_addr(s_lo), ob = tc::smem_addr(ops);
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = (s >> 2) * 1024 + (s & 3) * 32;
        tc::mma3(tU, tc::sdesc(sh + off, 2048), tc::sdesc(sl + off, 2048), tc::sdesc(ob + kWnHi + off, 2048),
                 tc::sdesc(ob + kWnLo + off, 2048), id64, false);
      }
      tc::commit(&bar_mma);
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = (s >> 2) * 1024 + (s & 3) * 32;
        tc::mma(tO, tc::sdesc(sh + off, 2048), tc::sdesc(ob + kQp + off, 2048), id64, s > 0 ? 1u : 0u);
      }
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar_mma, mma_phase));
    mma_phase ^= 1;
    if (!ok) break;
    tc::fence_after();
    // U^T images (row d)
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_col(tU, warp, 32 * half), v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 hi, lo;
        tc::split8(v + 8 * j, hi, lo);
        const uint32_t off = tc::img_off(d, 32 * half + 8 * j, 1);
        *reinterpret_cast<uint4*>(u_hi + off) = hi;
        *reinterpret_cast<uint4*>(u_lo + off) = lo;
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
    // S += U^T K' (three passes, N = 128) -> commit;  O^T += U^T P^T -> commit
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id64 = tc::idesc_bf16(128, 64), id128 = tc::idesc_bf16(128, 128);
      const uint32_t uh = tc::smem_addr(u_hi), ul = tc::smem_addr(u_lo), ob = tc::smem_addr(ops);
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = s * 32;
        tc::mma3(tS, tc::sdesc(uh + off, 1024), tc::sdesc(ul + off, 1024), tc::sdesc(ob + kKpHi + off, 1024),
                 tc::sdesc(ob + kKpLo + off, 1024), id128, false);
      }
      tc::commit(&bar_mma);
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = s * 32;
        tc::mma(tO, tc::sdesc(uh + off, 1024), tc::sdesc(ob + kP + off, 1024), id64, 1u);
      }
      tc::commit(&bar_mma);
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar_mma, mma_phase));
    mma_phase ^= 1;
    if (!ok) break;
    tc::fence_after();
    // images of the new state for the next chunk (every MMA that read the old ones is done)
    for (int c0 = 0; c0 < kD; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_col(tS, warp, c0), v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 hi, lo;
        tc::split8(v + 8 * j, hi, lo);
        const uint32_t off = tc::img_off(d, c0 + 8 * j, 2);
        *reinterpret_cast<uint4*>(s_hi + off) = hi;
        *reinterpret_cast<uint4*>(s_lo + off) = lo;
      }
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar_mma, mma_phase));
    mma_phase ^= 1;
    if (!ok) break;
    tc::fence_after();
    if (tid == 0 && c + 1 < nch) {  // the record is consumed: prefetch the next chunk's
      tc::expect_tx(&bar_tma, kScanCopy);
      tc::bulk_g2s(ops, record(c + 1), kScanCopy, &bar_tma);
    }
    // outputs: O^T row d, column t -> staged [t][d] -> 16-byte stores to out[token][h][:]
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_col(tO, warp, 32 * half), v);
#pragma unroll
      for (int i = 0; i < 32; ++i) o_stage[(32 * half + i) * kD + d] = __float2bfloat16_rn(v[i]);
    }
    tc::fence_async_smem();
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int idx = tid + 128 * k;  // 64 tokens x 16 words
      const int t = idx >> 4, w = idx & 15;
      const int gt = sGt[t];
      if (gt >= 0)
        *reinterpret_cast<uint4*>(out + ((int64_t)gt * p.Hv + h) * kD + 8 * w) =
            *reinterpret_cast<const uint4*>(o_stage + t * kD + 8 * w);
    }
    __syncthreads();
  }

  if (!ok) {
    if (tid == 0) set_status(p.status, GDN_STATUS_WAIT_TIMEOUT);
    tc::mbar_wait(&bar_mma, mma_phase);  // bounded drains of anything still in flight
    tc::mbar_wait(&bar_tma, tma_phase);
  } else if (slot > 0) {
    for (int c0 = 0; c0 < kD; c0 += 32) {
      float v[32];
      tc::tmem_ld32(tc::tmem_lane_col(tS, warp, c0), v);
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        *reinterpret_cast<float4*>(gS + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

template <typename QT>
cudaError_t launch_prep(const PrefillLaunch& p, int units, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel<QT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  chunk_prep_kernel<QT><<<dim3(units, p.Hv), 128, kPrepSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const gdn_layer_desc* d) {
  return d->head_k_dim == kD && d->head_v_dim == kD && d->act_dtype == GDN_BF16;
}

cudaError_t launch_prefill(const PrefillLaunch& p, gdn_dtype qkv_dtype, int units_upper, cudaStream_t s) {
  if (p.num_rows <= 0 || units_upper <= 0) return cudaSuccess;
  cudaError_t e = qkv_dtype == GDN_F32 ? launch_prep<float>(p, units_upper, s) : launch_prep<__nv_bfloat16>(p, units_upper, s);
  if (e != cudaSuccess) return e;
  static bool configured = false;
  if (!configured) {
    e = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  chunk_scan_kernel<<<dim3(p.Hv, p.num_rows), 128, kScanSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn
