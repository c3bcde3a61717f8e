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
// (one CTA per (row, chunk, v-head)); the scan kernel (one CTA per (row, v-head, quarter of dv))
// walks the chunks in order, keeping its 32 rows of the fp32 state in tensor memory.
//
// Tensor cores.  Every product is a tcgen05.mma (kind::f16, bf16 inputs, fp32 accumulation)
// with operands in swizzled shared memory and accumulators in TMEM.  Products that reach the
// state use a bf16 hi/lo split of both operands and three MMAs (about 1e-5 relative error); the
// output-only products use one.  Operands are K-major, or MN-major where that lets a thread
// write its row of values as 16-byte chunks (a K-major [k][m] tile with the 128-byte swizzle is
// read as the MN-major [m][k] operand; the scan's N = 32 operands use the 64-byte swizzle).
// The prep kernel solves T = (I + A)^-1 on the CUDA cores in 16 x 16 blocks and writes every
// chunk input of the scan as an exact shared-memory image; the scan copies a chunk's record in
// with bulk copies two chunks ahead and spreads its MMA issue over three threads.
//
// Path limits: dk = dv = 128 and bf16 activations; other shapes use the token recurrence.
// Every wait on an mbarrier is bounded; a timeout sets GDN_STATUS_WAIT_TIMEOUT, drains, frees
// TMEM and returns.
#include "gdn_internal.cuh"
#include "gdn_tc.cuh"
#include "gdn_testing.h"

namespace gdn {

namespace {

constexpr int kCh = kPrefillChunk;  // tokens per chunk
constexpr int kD = 128;             // dk = dv on this path

// Per (chunk, v-head) record written by the prep kernel, read by the scan kernel.
constexpr uint32_t kWnHi = 0;       // -W   [dk][t]  bf16 hi image (read MN-major)       16 KiB
constexpr uint32_t kWnLo = 16384;   //               bf16 lo image                       16 KiB
constexpr uint32_t kKpHi = 32768;   // K'   [s][dk]  bf16 hi image (2 atoms; read MN-major) 16 KiB
constexpr uint32_t kKpLo = 49152;   //               bf16 lo image                       16 KiB
constexpr uint32_t kQp = 65536;     // gamma q^ [t][dk] bf16 image                       16 KiB
constexpr uint32_t kP = 81920;      // P    [t][s]   bf16 image                           8 KiB
constexpr uint32_t kImgBytes = 90112;  // the images above: one bulk copy
constexpr uint32_t kUt = 90112;     // U~   [dv/32][t][32] fp32 (a quarter of dv each)  32 KiB
constexpr uint32_t kMeta = 122880;  // gamma_c (fp32)
static_assert(kRecBytes >= kMeta + 16 && kUt == kImgBytes, "record layout");

constexpr int kAStride = 68;  // floats per row of A in shared memory (16-byte aligned rows)
constexpr int kPrepThreads = 256;  // 8 warps: warps w and w + 4 share TMEM lane quarter w
constexpr int kPrepSmem = 81920 + kCh * kAStride * 4 + 1024;

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

// Four consecutive activations (16-byte aligned fp32 or 8-byte aligned bf16) as fp32.
__device__ __forceinline__ void load4(const float* p, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4*>(p);
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float (&x)[4]) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}

// g = -exp(A_log) softplus(a + dt_bias), held at -256 or above: e^g is 0 in fp32 from about
// -104 on either way, and the floor keeps a chunk's cumulative sum finite (an infinite or NaN g
// would turn every difference G_t - G_s of the chunk into NaN).
__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
  const float x = a + dt_bias;
  return fmaxf(-expf(A_log) * (x > 20.f ? x : log1pf(expf(x))), -256.f);
}

// Error-free sum: s + e == a + b exactly (Knuth's TwoSum; no operation here may be contracted or
// reassociated, and nvcc does neither for additions).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// (ah + al) + (bh + bl) as a normalised pair (hi carries the fp32 rounding of the sum).
__device__ __forceinline__ void add_pair(float ah, float al, float bh, float bl, float& h, float& l) {
  float s, e;
  two_sum(ah, bh, s, e);
  e += al + bl;
  h = s + e;
  l = e - (h - s);
}

// One 16 x 16 block T_ij of T = (I + A)^-1 (i > j), for the NR rows r0 .. r0+NR-1 of column c:
// M = sum_{k=j}^{i-1} A_ik T_kj into sM (solve_m), then T_ij = -T_ii M (solve_t).  T is stored
// transposed in the upper half of the A array (T[t][s] at sA[s][t]); in a diagonal block only
// the entries on or above the diagonal of that storage are T.
template <int NR>
__device__ __forceinline__ void solve_m(const float* sA, float* sM, int i, int j, int c, int r0) {
  float m[NR];
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) m[rr] = 0.f;
#pragma unroll 1
  for (int k = j; k < i; ++k) {
#pragma unroll
    for (int mm = 0; mm < 16; mm += 4) {
      float4 tv = *reinterpret_cast<const float4*>(sA + (16 * j + c) * kAStride + 16 * k + mm);
      if (k == j) {
        tv.x = mm >= c ? tv.x : 0.f;
        tv.y = mm + 1 >= c ? tv.y : 0.f;
        tv.z = mm + 2 >= c ? tv.z : 0.f;
        tv.w = mm + 3 >= c ? tv.w : 0.f;
      }
#pragma unroll
      for (int rr = 0; rr < NR; ++rr) {
        const float4 a = *reinterpret_cast<const float4*>(sA + (16 * i + r0 + rr) * kAStride + 16 * k + mm);
        m[rr] = fmaf(a.x, tv.x, m[rr]);
        m[rr] = fmaf(a.y, tv.y, m[rr]);
        m[rr] = fmaf(a.z, tv.z, m[rr]);
        m[rr] = fmaf(a.w, tv.w, m[rr]);
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) sM[(r0 + rr) * 16 + c] = m[rr];
}

template <int NR>
__device__ __forceinline__ void solve_t(float* sA, const float* sM, int i, int j, int c, int r0) {
  float acc[NR];
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) acc[rr] = 0.f;
#pragma unroll
  for (int mm = 0; mm < 16; ++mm) {  // T_ii[r][mm] (mm <= r) sits at row 16i+mm, column 16i+r
    const float* trow = sA + (16 * i + mm) * kAStride + 16 * i + r0;
    const float mv = sM[mm * 16 + c];
#pragma unroll
    for (int rr = 0; rr < NR; ++rr) acc[rr] = fmaf(mm <= r0 + rr ? trow[rr] : 0.f, mv, acc[rr]);
  }
#pragma unroll
  for (int rr = 0; rr < NR; ++rr) sA[(16 * j + c) * kAStride + 16 * i + r0 + rr] = -acc[rr];
}

// ------------------------------------------------------------------------------------------
// Prep: one CTA per (row, chunk, v-head); 256 threads (8 warps).
template <typename QT>
__global__ void __launch_bounds__(kPrepThreads, 2) chunk_prep_kernel(const PrefillLaunch p) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = align1k(dyn_smem);
  uint8_t* qk_hi = sm;  // [q^; k^] [128][128] images (MMA 1); then [beta v; beta gamma k^] rows (MMA 2, 3)
  uint8_t* qk_lo = sm + 32768;
  float* sA = reinterpret_cast<float*>(sm + 81920);  // A [64][kAStride]  (after MMA 1)
  uint8_t* t_hi = sm + 65536;  // T [64][64]
  uint8_t* t_lo = sm + 73728;
  // cumulative log-decay G_t as a pair sG + sGl: after a strongly decaying token G is large
  // while the later differences G_t - G_s that weight the chunk products stay small, and a single
  // fp32 sum would lose them to cancellation
  __shared__ float sG[kCh], sGl[kCh], sBeta[kCh], sRk[kCh], sBG[kCh];
  __shared__ float sMs[3][256];  // per-block 16 x 16 scratch of the blocked solve
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

  // the gate inputs of the chunk's tokens (threads 0 .. nc-1) go out before the row copies, so
  // that their latency runs under the copy issue
  float a_in = 0.f, b_in = 0.f;
  bool has_gate = false;
  if (tid < nc) {
    const int gt = global_token(p.rows, bos + t0 + tid, p.num_global, p.status);
    if (gt >= 0) {
      a_in = __bfloat162float(static_cast<const __nv_bfloat16*>(p.a)[(int64_t)gt * p.Hv + h]);
      b_in = __bfloat162float(static_cast<const __nv_bfloat16*>(p.b)[(int64_t)gt * p.Hv + h]);
      has_gate = true;
    }
  }
  const float a_log = __ldg(p.A_log + h), dt_b = __ldg(p.dt_bias + h);

  // 0. every row the chunk reads starts its trip to shared memory at once (cp.async, no
  //    registers held): the q and k rows into the image region they are turned into (one
  //    commit group), the v rows into the T / A region, which nothing uses before the first
  //    product completes; right after it they become the beta v operand rows (a second group)
  constexpr uint32_t kQStage = 0, kKStage = 32768;  // [kCh][kD] QT each, up to 32 KiB
  constexpr uint32_t kVStage = 65536;               // [kCh][kD] QT at sm + kVStage, up to 32 KiB
  {
    constexpr int RCH = kD * (int)sizeof(QT) / 16;  // 16-byte chunks per row
    const uint32_t dq = tc::smem_addr(sm + kQStage), dkk = tc::smem_addr(sm + kKStage);
    const uint8_t* srcq = reinterpret_cast<const uint8_t*>(qkv + (int64_t)(bos + t0) * C + qoff);
    const uint8_t* srck = reinterpret_cast<const uint8_t*>(qkv + (int64_t)(bos + t0) * C + koff);
    for (int i = tid; i < nc * RCH; i += kPrepThreads) {
      const int64_t go = (int64_t)(i / RCH) * C * (int64_t)sizeof(QT) + 16 * (i % RCH);
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dq + 16 * i), "l"(srcq + go) : "memory");
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dkk + 16 * i), "l"(srck + go) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  {
    constexpr int VCH = kD * (int)sizeof(QT) / 16;  // 16-byte chunks per v row
    const uint32_t dst0 = tc::smem_addr(sm + kVStage);
    const uint8_t* src0 = reinterpret_cast<const uint8_t*>(qkv + (int64_t)(bos + t0) * C + voff);
    for (int i = tid; i < nc * VCH; i += kPrepThreads)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst0 + 16 * i),
                   "l"(src0 + (int64_t)(i / VCH) * C * (int64_t)sizeof(QT) + 16 * (i % VCH))
                   : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  // 1. gates (padded tokens: g = 0, beta = 0), TMEM and barrier
  if (tid < kCh) {
    float g = 0.f, beta = 0.f;
    if (has_gate) {
      g = gate_g(a_in, a_log, dt_b);
      beta = 1.f / (1.f + expf(-b_in));
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
  if (warp == 0) {  // G_t = g_1 + .. + g_t (inclusive): lane l sums tokens 2l, 2l+1, then a warp scan
    const float g0 = sG[2 * lane], g1 = sG[2 * lane + 1];
    float xh, xl;
    two_sum(g0, g1, xh, xl);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float yh = __shfl_up_sync(0xffffffffu, xh, o), yl = __shfl_up_sync(0xffffffffu, xl, o);
      if (lane >= o) add_pair(yh, yl, xh, xl, xh, xl);
    }
    float eh = __shfl_up_sync(0xffffffffu, xh, 1), el = __shfl_up_sync(0xffffffffu, xl, 1);
    if (lane == 0) eh = el = 0.f;
    float h0, l0, h1, l1;
    add_pair(eh, el, g0, 0.f, h0, l0);
    add_pair(h0, l0, g1, 0.f, h1, l1);
    sG[2 * lane] = h0;
    sGl[2 * lane] = l0;
    sG[2 * lane + 1] = h1;
    sGl[2 * lane + 1] = l1;
  }
  __syncthreads();

  // 2. q^ (scaled) and k^ rows of the [q^; k^] images, and the gamma q^ record rows; warp w
  //    takes tokens 8w .. 8w+7: their raw rows from shared memory into registers, then (once
  //    every warp holds its rows) the images over the raw rows
  {
    asm volatile("cp.async.wait_group 1;" ::: "memory");  // the q and k rows (v may still be in flight)
    __syncthreads();
    float q[8][4], k[8][4];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int t = warp * 8 + b;
      if (t < nc) {
        load4(reinterpret_cast<const QT*>(sm + kQStage) + t * kD + 4 * lane, q[b]);
        load4(reinterpret_cast<const QT*>(sm + kKStage) + t * kD + 4 * lane, k[b]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) q[b][e] = k[b][e] = 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int t = warp * 8 + b;
      float sq = 0.f, sk = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sq = fmaf(q[b][e], q[b][e], sq);
        sk = fmaf(k[b][e], k[b][e], sk);
      }
      sq = warp_sum32(sq);
      sk = warp_sum32(sk);
      // hardware reciprocal square root (2 ulp): well inside what the chunk products carry
      const float rq = rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
      if (lane == 0) sRk[t] = rk;
      const float gam = __expf(sG[t]);  // gamma_t for the bf16 gamma q^ rows (output products only)
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
  if (tid < kCh) sBG[tid] = sBeta[tid] * expf(sG[tid]);  // beta_t gamma_t, the row scale of k^ in W
  bool ok = __syncthreads_and(tc::mbar_wait(&bar, 0, p.wait_ns));
  if (ok) {
    tc::fence_after();
    // 3b. the rows beta_s v_s into the q^ half of the images, which MMA 1 no longer needs (the
    //     A operand of MMA 3, read MN-major like MMA 2's); the staged v rows are consumed here,
    //     before the A rows below overwrite their shared memory
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    for (int i = tid; i < kCh * (kD / 4); i += kPrepThreads) {
      const int t = i / (kD / 4), d0 = 4 * (i % (kD / 4));
      float x[4] = {0.f, 0.f, 0.f, 0.f};
      if (t < nc) {
        load4(reinterpret_cast<const QT*>(sm + kVStage) + t * kD + d0, x);
        const float bs = sBeta[t];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= bs;
      }
      put4_pair(qk_hi, qk_lo, t, d0, 2, x);
    }
    __syncthreads();
    // 4. P rows to the record (lane quarters 0, 1: q rows); A rows to shared memory (quarters
    //    2, 3: k rows); warp w reads columns 32 (w / 4) .. +31 of its quarter's rows
    const int quarter = warp & 3, chalf = warp >> 2;
    float v0[32];
    tc::tmem_ld32(tc::tmem_lane_col(tmem, quarter, 32 * chalf), v0);
    const int t = (quarter & 1) * 32 + lane;
    const float Gt = sG[t], Gtl = sGl[t];
    if (quarter < 2) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = 32 * chalf + 8 * j + e;
          x[e] = s <= t ? __expf((Gt - sG[s]) + (Gtl - sGl[s])) * v0[8 * j + e] : 0.f;
        }
        *reinterpret_cast<uint4*>(rec + kP + tc::img_off(t, 32 * chalf + 8 * j, 1)) = tc::pack8(x);
      }
    } else {
      const float bt = sBeta[t];
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = 32 * chalf + j + e;
          x[e] = s < t ? bt * __expf((Gt - sG[s]) + (Gtl - sGl[s])) * v0[j + e] : 0.f;
        }
        *reinterpret_cast<float4*>(sA + t * kAStride + 32 * chalf + j) = make_float4(x[0], x[1], x[2], x[3]);
      }
    }
    __syncthreads();

    if (warp < 4) {
      // 5. T = (I + A)^-1 on warps 0-3 in 16 x 16 blocks: the diagonal blocks (I + A_bb)^-1 by
      //    forward substitution (warps 0-1), then T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj in order
      //    of i - j, the blocks of a distance spread over the four warps.  T is kept transposed
      //    in the upper half of the A array: T[t][s] (t >= s) at sA[s][t] (A is strictly lower,
      //    and A_ii is not read again once T_ii exists).
      if (warp < 2) {
        const int o = 16 * (2 * warp + (lane >> 4)), c = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r) {  // entries at and above the diagonal of A are zero
          float acc = r == c ? 1.f : 0.f;
#pragma unroll
          for (int m = 0; m < ((r + 3) & ~3); m += 4) {
            const float4 a = *reinterpret_cast<const float4*>(sA + (o + r) * kAStride + o + m);
            acc = fmaf(-a.x, x[m], acc);
            acc = fmaf(-a.y, x[m + 1], acc);
            acc = fmaf(-a.z, x[m + 2], acc);
            acc = fmaf(-a.w, x[m + 3], acc);
          }
          x[r] = acc;
        }
        __syncwarp();
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r >= c) sA[(o + c) * kAStride + o + r] = x[r];
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const int c = lane & 15;
#pragma unroll 1
      for (int dist = 1; dist < 4; ++dist) {
        // distance 1: three blocks, one warp each; 2: two blocks, two warps each; 3: one block
        const int wpb = dist == 1 ? 1 : (dist == 2 ? 2 : 4);
        const int bi = warp / wpb, part = warp % wpb;
        const bool active = dist + bi < 4;
        const int i = dist + bi, j = i - dist;
        float* sM = sMs[bi < 3 ? bi : 0];
        if (active) {
          if (dist == 1) solve_m<8>(sA, sM, i, j, c, (lane >> 4) * 8);
          else if (dist == 2) solve_m<4>(sA, sM, i, j, c, part * 8 + (lane >> 4) * 4);
          else solve_m<2>(sA, sM, i, j, c, part * 4 + (lane >> 4) * 2);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (active) {
          if (dist == 1) solve_t<8>(sA, sM, i, j, c, (lane >> 4) * 8);
          else if (dist == 2) solve_t<4>(sA, sM, i, j, c, part * 8 + (lane >> 4) * 4);
          else solve_t<2>(sA, sM, i, j, c, part * 4 + (lane >> 4) * 2);
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
    } else {
      // 6b. meanwhile, on warps 4-7: the A operand of MMA 2, read MN-major (a [s][d] tile laid
      //     out like a K-major one): the k^ rows of the [q^; k^] images scaled in place by
      //     beta_s gamma_s; on the way, the record's K' rows e^{G_c - G_s} k^_s (the same layout).
      const float Gc = sG[kCh - 1], Gcl = sGl[kCh - 1];
      for (int i = tid - 128; i < kCh * (kD / 8); i += 128) {
        const int t = i / (kD / 8), d0 = 8 * (i % (kD / 8));
        const uint32_t off = tc::img_off(kCh + t, d0, 2);
        const uint4 h = *reinterpret_cast<const uint4*>(qk_hi + off), l = *reinterpret_cast<const uint4*>(qk_lo + off);
        const __nv_bfloat16* hb = reinterpret_cast<const __nv_bfloat16*>(&h);
        const __nv_bfloat16* lb = reinterpret_cast<const __nv_bfloat16*>(&l);
        float kn[8], x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) kn[e] = __bfloat162float(hb[e]) + __bfloat162float(lb[e]);
        const float f = sBG[t], fp = expf((Gc - sG[t]) + (Gcl - sGl[t]));  // padded tokens: k^ = 0
        uint4 nh, nl;
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = fp * kn[e];
        tc::split8(x, nh, nl);
        const uint32_t roff = tc::img_off(t, d0, 2);
        *reinterpret_cast<uint4*>(rec + kKpHi + roff) = nh;
        *reinterpret_cast<uint4*>(rec + kKpLo + roff) = nl;
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = f * kn[e];
        tc::split8(x, nh, nl);
        *reinterpret_cast<uint4*>(qk_hi + off) = nh;
        *reinterpret_cast<uint4*>(qk_lo + off) = nl;
      }
      if (tid == 128) *reinterpret_cast<float*>(rec + kMeta) = expf(Gc);
    }
    __syncthreads();
    // 6a. T image (rows t, K = s) once the solve is done, on all eight warps: row tid % 64,
    //     columns 16 (tid / 64) .. +15
    {
      const int t2 = tid & 63, g0 = 16 * (tid >> 6);
#pragma unroll
      for (int g8 = g0; g8 < g0 + 16; g8 += 8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s2 = g8 + e;
          x[e] = s2 <= t2 ? sA[s2 * kAStride + t2] : 0.f;
        }
        uint4 hi, lo;
        tc::split8(x, hi, lo);
        const uint32_t off = tc::img_off(t2, g8, 1);
        *reinterpret_cast<uint4*>(t_hi + off) = hi;
        *reinterpret_cast<uint4*>(t_lo + off) = lo;
      }
    }
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();

    // 7. MMA 2, 3: W^T (cols 64..127) = (beta gamma K^)^T T^T;  U~^T (cols 128..191) = (beta V)^T T^T,
    //    A operands MN-major from the [s][d] rows (two 64-wide d atoms 1 KiB apart, 8-row s groups
    //    2 KiB apart), B = T, K-major
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id = tc::idesc_bf16_amn(128, 64);
      const uint32_t kh = tc::smem_addr(qk_hi) + 16384, kl = tc::smem_addr(qk_lo) + 16384;
      const uint32_t vh = tc::smem_addr(qk_hi), vl = tc::smem_addr(qk_lo);
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = s * 32, aoff = s * 4096;
        const uint64_t th = tc::sdesc(tc::smem_addr(t_hi) + off, 1024), tl = tc::sdesc(tc::smem_addr(t_lo) + off, 1024);
        tc::mma3(tmem + 64, tc::sdesc_lbo(kh + aoff, 1024, 2048), tc::sdesc_lbo(kl + aoff, 1024, 2048), th, tl, id,
                 s == 0);
        tc::mma3(tmem + 128, tc::sdesc_lbo(vh + aoff, 1024, 2048), tc::sdesc_lbo(vl + aoff, 1024, 2048), th, tl, id,
                 s == 0);
      }
      tc::commit(&bar);
    }
    ok = __syncthreads_and(tc::mbar_wait(&bar, 1, p.wait_ns));
    if (ok) {
      tc::fence_after();
      // 8. -W and U~ (fp32) from TMEM, lane = row d, warp w taking columns 32 (w / 4) .. +31,
      //    staged in shared memory exactly as the record holds them (the MMA operands there are
      //    consumed) and stored by two bulk copies: -W^T row d as row d of a [dk][t] image (read
      //    MN-major by the scan), U~ as [dv/32][t][32]
      const int quarter = warp & 3, half = warp >> 2;
      const int d = 32 * quarter + lane;
      float* ut = reinterpret_cast<float*>(sm + 32768);
      float w[32];
      tc::tmem_ld32(tc::tmem_lane_col(tmem, quarter, 64 + 32 * half), w);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = -w[8 * c + e];
        uint4 hi, lo;
        tc::split8(x, hi, lo);
        const uint32_t off = tc::img_off(d, 32 * half + 8 * c, 1);
        *reinterpret_cast<uint4*>(sm + kWnHi + off) = hi;
        *reinterpret_cast<uint4*>(sm + kWnLo + off) = lo;
      }
      tc::tmem_ld32(tc::tmem_lane_col(tmem, quarter, 128 + 32 * half), w);
#pragma unroll
      for (int i = 0; i < 32; ++i) ut[((d >> 5) * kCh + 32 * half + i) * 32 + (d & 31)] = w[i];
      tc::fence_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc::bulk_s2g(rec + kWnHi, sm + kWnHi, 32768);
        tc::bulk_s2g(rec + kUt, sm + 32768, 32768);
        tc::bulk_store_commit();
        tc::bulk_store_wait();
      }
    }
  }
  if (!ok) {
    if (tid == 0) set_status(p.status, GDN_STATUS_WAIT_TIMEOUT);
    tc::mbar_wait(&bar, 0, p.wait_ns);  // bounded: let any issued MMA drain before TMEM is released
    tc::mbar_wait(&bar, 1, p.wait_ns);
    asm volatile("cp.async.wait_all;" ::: "memory");  // and the staged v rows (if MMA 1 never came)
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------------------------------
// Scan: one CTA per (row, v-head, quarter of dv); 128 threads.  The state rows are independent
// given the chunk inputs (U, O and the new state of dv row j read only row j of S_0), so each
// CTA carries 32 rows of S.  It keeps S^T (lane = dk, column = its 32 dv) in TMEM so the state
// update is an M = 128 MMA:  S_c^T = gamma_c S_0^T + K'^T U.  U and O are M = 64 accumulators
// (row t of a 64-row accumulator sits in TMEM lane t % 16 + 32 (t / 16)); TMEM columns: S^T
// [0, 32), U [32, 64), O of even / odd chunks [64, 96) / [96, 128).
//   U   = U~ - W S_0^T          A = -W [t][dk],     B = S_0 [dv][dk]      (three passes)
//   O   = (gamma q^) S_0^T      A = gamma q^ [t][dk], B = S_0 [dv][dk]    (one pass)
//   S^T += K'^T U               A = K'^T [dk][s],    B = U^T [dv][s]      (three passes)
//   O  += P U                   A = P [t][s],        B = U^T [dv][s]      (one pass)
// Chunk records arrive by bulk copy into two buffers, two chunks ahead.
constexpr int kQuarters = kD / 32;
constexpr uint32_t kBufUt = kImgBytes;          // this CTA's quarter of U~, [t][32] fp32
constexpr uint32_t kBufMeta = kImgBytes + 8192;  // gamma_c
constexpr uint32_t kBufBytes = kBufMeta + 1024;  // 1 KiB-aligned buffers
constexpr uint32_t kBufCopy = kImgBytes + 8192 + 16;
constexpr uint32_t kSImg = 2 * kBufBytes;        // S_0 [32][128] hi, lo: 8 KiB each
constexpr uint32_t kUImg = kSImg + 16384;        // U^T [32][64] hi, lo: 4 KiB each
constexpr int kScanSmemNew = (int)kUImg + 8192 + 1024;
// kScanWpq warps share each TMEM lane quarter (warp w takes quarter w % 4) and split its 32
// columns, so every phase that moves the state, U or O between TMEM, registers and shared memory
// has 1 / kScanWpq of the work per warp on the chunk chain.
#ifndef GDN_SCAN_WPQ
#define GDN_SCAN_WPQ 2
#endif
constexpr int kScanWpq = GDN_SCAN_WPQ;        // 1, 2 or 4
constexpr int kScanThreads = 128 * kScanWpq;
constexpr int kScanCols = 32 / kScanWpq;      // TMEM columns per warp
constexpr int kScanHalf = kScanCols / 2;      // U columns per lane (lanes 16..31 take the upper half)
static_assert(kScanWpq == 1 || kScanWpq == 2 || kScanWpq == 4, "1, 2 or 4 warps per lane quarter");
constexpr int kTokFirst = kScanThreads >= 256 ? kScanThreads - kCh : 96;  // first token-loading thread
static_assert(kTokFirst > 64, "the product issuers (threads 0, 32, 64) load no token index");
static_assert(kScanSmemNew <= 232448, "scan shared memory");

__global__ void __launch_bounds__(kScanThreads, 1) chunk_scan_kernel(const PrefillLaunch p) {
  extern __shared__ uint8_t dyn_smem[];
  uint8_t* sm = align1k(dyn_smem);
  uint8_t* s_hi = sm + kSImg;
  uint8_t* s_lo = s_hi + 8192;
  uint8_t* u_hi = sm + kUImg;
  uint8_t* u_lo = u_hi + 4096;
  // one barrier per commit point, each committed and waited once per chunk (so a wait is never
  // more than one phase behind): U ready; state update done; O done; the first O half done.
  // Thread 0 issues the U and state products, thread 32 the output products, so neither
  // stream of MMAs waits behind the other's issue.
  __shared__ __align__(8) uint64_t bar_mma[5], bar_tma[2];
  __shared__ uint32_t tmem_base;
  __shared__ int sGt[2][kCh];  // global tokens of the chunk whose outputs are pending

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x / kQuarters, q = blockIdx.x % kQuarters;
  const int n = p.first_row + blockIdx.y;
  const int base_unit = units_before(p.rows, p.first_row, n, kCh);
  const int bos = __ldg(p.rows.qsl + n), eos = __ldg(p.rows.qsl + n + 1);
  if (bos < 0 || eos < bos || eos > p.rows.num_tokens || eos == bos) return;  // malformed rows flagged by prep
  const int L = eos - bos;
  const int nch = (L + kCh - 1) / kCh;
  int slot = __ldg(p.rows.state_idx + n);
  const int load_slot = non_spec_load_slot(p.rows, n);
  if (load_slot < 0) {  // acceptance-aware row with num_accepted out of range
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, GDN_STATUS_NUM_ACCEPTED);
    return;
  }
  bool read_prior = load_slot > 0 && (p.rows.has_init == nullptr || __ldg(p.rows.has_init + n) != 0);
  if (slot >= p.num_slots || load_slot >= p.num_slots) {
    if (tid == 0 && blockIdx.x == 0) set_status(p.status, GDN_STATUS_SLOT_RANGE);
    if (slot >= p.num_slots) slot = 0;
    read_prior = false;
  }
  const int wq = warp & 3, ch = warp >> 2;  // TMEM lane quarter; which kScanCols of its 32 columns
  const int dk = 32 * wq + lane;            // this thread's TMEM lane of S^T
  const int dv0 = 32 * q;
  // element (dv0 + j, dk) of the state is at base + j * kD
  float* gS = p.ssm_pool + ((int64_t)slot * p.Hv + h) * kD * kD + (int64_t)dv0 * kD + dk;
  const float* gS0 = p.ssm_pool + ((int64_t)(read_prior ? load_slot : 0) * p.Hv + h) * kD * kD + (int64_t)dv0 * kD + dk;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);

  if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
  if (tid == 32) {
    for (int i = 0; i < 5; ++i) tc::mbar_init(&bar_mma[i], 1);
    tc::mbar_init(&bar_tma[0], 1);
    tc::mbar_init(&bar_tma[1], 1);
    tc::mbar_init_fence();
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  // O alternates between two accumulators: chunk c's outputs are drained while chunk c + 1 runs
  const uint32_t tS = tmem_base, tU = tmem_base + 32, tO0 = tmem_base + 64, tU2 = tmem_base + 128;
  auto store_outputs = [&](int c) {  // row t of O -> kScanCols bf16 of out[token][h][dv0 + ..]
    float o[kScanCols];
    tc::tmem_ld<kScanCols>(tc::tmem_lane_col(tO0 + 32 * (c & 1), warp, kScanCols * ch), o);
    if (lane < 16) {
      const int gt = sGt[c & 1][16 * wq + lane];
      if (gt >= 0) {
        uint4* dst = reinterpret_cast<uint4*>(out + ((int64_t)gt * p.Hv + h) * kD + dv0 + kScanCols * ch);
#pragma unroll
        for (int i = 0; i < kScanCols / 8; ++i) dst[i] = tc::pack8(o + 8 * i);
      }
    }
  };
  // chunk c's record -> buffer c & 1 (thread 0).  The test hook drop_copy_chunk leaves one
  // chunk's copy out, so the wait for it runs out with nothing in flight.
  auto issued = [&](int c) { return c != p.drop_copy_chunk; };
  auto issue = [&](int c) {
    if (!issued(c)) return;
    const uint8_t* rec = p.ws + ((size_t)(base_unit + c) * p.Hv + h) * kRecBytes;
    uint8_t* buf = sm + (c & 1) * kBufBytes;
    uint64_t* bar = &bar_tma[c & 1];
    tc::expect_tx(bar, kBufCopy);
    tc::bulk_g2s(buf, rec, kImgBytes, bar);
    tc::bulk_g2s(buf + kBufUt, rec + kUt + q * 8192, 8192, bar);
    tc::bulk_g2s(buf + kBufMeta, rec + kMeta, 16, bar);
  };
  if (tid == 0) {
    issue(0);
    if (nch > 1) issue(1);
  }
  // copies issued into / waited for (successfully) in each buffer, for the drain after a timeout
  int tma_issued[2] = {issued(0) ? 1 : 0, nch > 1 && issued(1) ? 1 : 0}, tma_done[2] = {0, 0};
  int mma_commits[5] = {0, 0, 0, 0, 0}, mma_done[5] = {0, 0, 0, 0, 0};

  // initial state: images of S_0 (unscaled) and gamma_0 S_0^T in TMEM
  float v[kScanCols];
#pragma unroll
  for (int j = 0; j < kScanCols; ++j) v[j] = read_prior ? gS0[(int64_t)(kScanCols * ch + j) * kD] : 0.f;
  tc::put_mn32_row(s_hi, s_lo, dk, v, kScanCols / 8 * ch, kScanCols / 8);
  bool ok = __syncthreads_and(tc::mbar_wait(&bar_tma[0], 0, p.wait_ns));
  if (ok) tma_done[0] = 1;
  if (ok) {
    const float g0 = *reinterpret_cast<const float*>(sm + kBufMeta);
#pragma unroll
    for (int j = 0; j < kScanCols; ++j) v[j] *= g0;
    tc::tmem_st<kScanCols>(tc::tmem_lane_col(tS, warp, kScanCols * ch), v);
    tc::tmem_st_wait();
  }
  tc::fence_async_smem();
  tc::fence_before();
  __syncthreads();

  for (int c = 0; c < nch && ok; ++c) {
    const int b = c & 1;
    uint8_t* buf = sm + b * kBufBytes;
    // the chunk's global tokens, loaded by the last warps (none of which issues products, so a
    // gathered row's index loads never hold the products behind them)
    for (int i = tid - kTokFirst; i >= 0 && i < kCh; i += kScanThreads - kTokFirst) {
      const int t = c * kCh + i;
      sGt[b][i] = t < L ? global_token(p.rows, bos + t, p.num_global, p.status) : -1;
    }
    const uint32_t tO = tO0 + 32 * b;
    // U = -W S_0^T (three passes) -> commit (thread 0);  O = (gamma q^) S_0^T -> commit (thread 32)
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id = tc::idesc_bf16_abmn(64, 32);  // -W rows and S images both MN-major
      const uint32_t bb = tc::smem_addr(buf), sh = tc::smem_addr(s_hi), sl = tc::smem_addr(s_lo);
      for (int s = 0; s < 4; ++s) {  // first half of K into tU, the second half on thread 64
        tc::mma3(tU, tc::sdesc_lbo(bb + kWnHi + 2048 * s, 16, 1024), tc::sdesc_lbo(bb + kWnLo + 2048 * s, 16, 1024),
                 tc::sdesc_mn32(sh + 1024 * s), tc::sdesc_mn32(sl + 1024 * s), id, s == 0);
      }
      tc::commit(&bar_mma[0]);
    } else if (tid == 64) {
      tc::fence_after();
      const uint32_t id = tc::idesc_bf16_abmn(64, 32);
      const uint32_t bb = tc::smem_addr(buf), sh = tc::smem_addr(s_hi), sl = tc::smem_addr(s_lo);
      for (int s = 4; s < 8; ++s) {
        tc::mma3(tU2, tc::sdesc_lbo(bb + kWnHi + 2048 * s, 16, 1024), tc::sdesc_lbo(bb + kWnLo + 2048 * s, 16, 1024),
                 tc::sdesc_mn32(sh + 1024 * s), tc::sdesc_mn32(sl + 1024 * s), id, s == 4);
      }
      tc::commit(&bar_mma[4]);
    } else if (tid == 32) {
      tc::fence_after();
      const uint32_t id = tc::idesc_bf16_bmn(64, 32);
      const uint32_t bb = tc::smem_addr(buf), sh = tc::smem_addr(s_hi);
      for (int s = 0; s < 8; ++s) {
        const uint32_t off = (s >> 2) * 1024 + (s & 3) * 32;
        tc::mma(tO, tc::sdesc(bb + kQp + off, 2048), tc::sdesc_mn32(sh + 1024 * s), id, s > 0 ? 1u : 0u);
      }
      tc::commit(&bar_mma[3]);
    }
    ++mma_commits[0];
    ++mma_commits[3];
    ++mma_commits[4];
    if (c > 0) store_outputs(c - 1);  // while the U products run
    // this lane's U~ values (independent of the products): rows t of this warp's quarter sit in
    // lanes 0..15 of it; of the warp's kScanCols columns, lanes 16..31 take over the upper half
    const int sh = lane >> 4, t = 16 * wq + (lane & 15);
    const int ucol = kScanCols * ch + kScanHalf * sh;  // this lane's first U column
    float4 utv[kScanHalf / 4];
    {
      const float4* ut = reinterpret_cast<const float4*>(buf + kBufUt) + t * 8 + ucol / 4;
#pragma unroll
      for (int j4 = 0; j4 < kScanHalf / 4; ++j4) utv[j4] = ut[j4];
    }
    // Each warp goes on as soon as U is ready (the issuing thread's warp joins after issuing the
    // output products); the block-wide barrier comes only before the next products are issued.
    const bool u_ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar_mma[0], mma_done[0] & 1, p.wait_ns) &&
                                                  tc::mbar_wait(&bar_mma[4], mma_done[4] & 1, p.wait_ns));
    ++mma_done[0];
    ++mma_done[4];
    // U += U~; U^T images (row = dv, column = t)
    if (u_ok) {
      tc::fence_after();
      float u[kScanCols], u2[kScanCols];
      tc::tmem_ld2<kScanCols>(tc::tmem_lane_col(tU, warp, kScanCols * ch), u,
                              tc::tmem_lane_col(tU2, warp, kScanCols * ch), u2);
#pragma unroll
      for (int j = 0; j < kScanCols; ++j) u[j] += u2[j];
      float w[kScanHalf];
#pragma unroll
      for (int j = 0; j < kScanHalf; ++j) {
        const float upper = __shfl_sync(0xffffffffu, u[kScanHalf + j], lane & 15);
        w[j] = sh ? upper : u[j];
      }
#pragma unroll
      for (int j4 = 0; j4 < kScanHalf / 4; ++j4) {
        const float4 f = utv[j4];
        w[4 * j4] += f.x; w[4 * j4 + 1] += f.y; w[4 * j4 + 2] += f.z; w[4 * j4 + 3] += f.w;
      }
      if constexpr (kScanHalf >= 8) tc::put_mn32_row(u_hi, u_lo, t, w, ucol / 8, kScanHalf / 8);
      else tc::put_mn32_half(u_hi, u_lo, t, w, ucol / 8, (ucol / 4) & 1);
    }
    tc::fence_async_smem();
    tc::fence_before();
    ok = __syncthreads_and(u_ok);
    if (!ok) break;
    // S^T += K'^T U (three passes) -> commit (thread 0);  O += P U -> commit (thread 32)
    if (tid == 0) {
      tc::fence_after();
      const uint32_t id128 = tc::idesc_bf16_abmn(128, 32);  // K' rows read MN-major
      const uint32_t bb = tc::smem_addr(buf), uh = tc::smem_addr(u_hi), ul = tc::smem_addr(u_lo);
      for (int s = 0; s < 4; ++s) {
        tc::mma3(tS, tc::sdesc_lbo(bb + kKpHi + 4096 * s, 1024, 2048), tc::sdesc_lbo(bb + kKpLo + 4096 * s, 1024, 2048),
                 tc::sdesc_mn32(uh + 1024 * s), tc::sdesc_mn32(ul + 1024 * s), id128, false);
      }
      tc::commit(&bar_mma[1]);
    } else if (tid == 32) {  // after its own first half, in issue order on this thread
      tc::fence_after();
      const uint32_t id64 = tc::idesc_bf16_bmn(64, 32);
      const uint32_t bb = tc::smem_addr(buf), uh = tc::smem_addr(u_hi);
      for (int s = 0; s < 4; ++s) {
        const uint32_t off = s * 32;
        tc::mma(tO, tc::sdesc(bb + kP + off, 1024), tc::sdesc_mn32(uh + 1024 * s), id64, 1u);
      }
      tc::commit(&bar_mma[2]);
    }
    ++mma_commits[1];
    ++mma_commits[2];
    // the state images are rewritten below: the state products and the first output half (which
    // read them) must be done
    const bool s_ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar_mma[1], mma_done[1] & 1, p.wait_ns) &&
                                                  tc::mbar_wait(&bar_mma[3], mma_done[3] & 1, p.wait_ns));
    ++mma_done[1];
    ++mma_done[3];
    bool tma_ok = true;
    if (s_ok) {
      tc::fence_after();
      // the new state: gamma_{c+1} S^T back into TMEM (in flight while the images for the next
      // chunk are written)
      tc::tmem_ld<kScanCols>(tc::tmem_lane_col(tS, warp, kScanCols * ch), v);
      if (c + 1 < nch) {
        const int nb = (c + 1) & 1;
        tma_ok = tc::mbar_wait(&bar_tma[nb], tma_done[nb] & 1, p.wait_ns);
        if (tma_ok) ++tma_done[nb];
        const float gn = *reinterpret_cast<const float*>(sm + nb * kBufBytes + kBufMeta);
        float sv[kScanCols];
#pragma unroll
        for (int j = 0; j < kScanCols; ++j) sv[j] = v[j] * gn;
        tc::tmem_st<kScanCols>(tc::tmem_lane_col(tS, warp, kScanCols * ch), sv);
        tc::put_mn32_row(s_hi, s_lo, dk, v, kScanCols / 8 * ch, kScanCols / 8);
      } else if (slot > 0) {
#pragma unroll
        for (int j = 0; j < kScanCols; ++j) gS[(int64_t)(kScanCols * ch + j) * kD] = v[j];
      }
    }
    const bool mma_ok = s_ok && tc::mbar_wait(&bar_mma[2], mma_done[2] & 1, p.wait_ns);
    ok = __syncthreads_and(tma_ok && mma_ok);
    ++mma_done[2];
    if (!ok) break;
    tc::fence_after();
    if (tid == 0 && c + 2 < nch) {  // this buffer is consumed: fetch chunk c + 2 into it
      issue(c + 2);
    }
    if (c + 2 < nch && issued(c + 2)) ++tma_issued[b];
    if (c + 1 == nch) store_outputs(c);
    tc::tmem_st_wait();
    tc::fence_async_smem();
    tc::fence_before();
    __syncthreads();
  }

  if (!ok) {
    if (tid == 0) set_status(p.status, GDN_STATUS_WAIT_TIMEOUT);
    // bounded drains of anything still in flight (the wait that failed included) before TMEM
    // and shared memory are released
    for (int i = 0; i < 5; ++i)
      for (int k = mma_done[i] > 0 ? mma_done[i] - 1 : 0; k < mma_commits[i]; ++k)
        tc::mbar_wait(&bar_mma[i], k & 1, p.wait_ns);
    // copies: only those issued and not yet seen complete (a copy the test hook left out is
    // neither, so nothing waits for it again)
    for (int bb = 0; bb < 2; ++bb)
      for (int k = tma_done[bb]; k < tma_issued[bb]; ++k) tc::mbar_wait(&bar_tma[bb], k & 1, p.wait_ns);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

template <typename QT>
cudaError_t launch_prep(const PrefillLaunch& p, int units, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(chunk_prep_kernel<QT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmem);
  });
  if (e != cudaSuccess) return e;
  chunk_prep_kernel<QT><<<dim3(units, p.Hv), kPrepThreads, kPrepSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

namespace {
// Test hooks (gdn_testing.h): a shorter wait limit and a record copy left out on purpose.
std::atomic<uint64_t> g_test_wait_ns{0};
std::atomic<int32_t> g_test_drop_chunk{-1};
}  // namespace

bool prefill_tc_supported(const gdn_layer_desc* d) {
  return d->head_k_dim == kD && d->head_v_dim == kD && d->act_dtype == GDN_BF16;
}

cudaError_t launch_prefill(const PrefillLaunch& args, gdn_dtype qkv_dtype, int units_upper, cudaStream_t s) {
  if (args.num_rows <= 0 || units_upper <= 0) return cudaSuccess;
  PrefillLaunch p = args;
  const uint64_t wait = g_test_wait_ns.load(std::memory_order_relaxed);
  p.wait_ns = wait ? wait : kDefaultWaitNs;
  p.drop_copy_chunk = g_test_drop_chunk.load(std::memory_order_relaxed);
  cudaError_t e = qkv_dtype == GDN_F32 ? launch_prep<float>(p, units_upper, s) : launch_prep<__nv_bfloat16>(p, units_upper, s);
  if (e != cudaSuccess) return e;
  static std::atomic<uint64_t> configured{0};
  e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmemNew);
  });
  if (e != cudaSuccess) return e;
  chunk_scan_kernel<<<dim3(p.Hv * kQuarters, p.num_rows), kScanThreads, kScanSmemNew, s>>>(p);
  return cudaGetLastError();
}

}  // namespace gdn

extern "C" int gdn_testing_set_prefill_faults(uint64_t wait_ns, int32_t drop_copy_chunk) {
  gdn::g_test_wait_ns.store(wait_ns, std::memory_order_relaxed);
  gdn::g_test_drop_chunk.store(drop_copy_chunk < 0 ? -1 : drop_copy_chunk, std::memory_order_relaxed);
  return GDN_OK;
}
