// Codebook keys with the TurboQuantProd residual sketch and the outlier
// two-stream store (turboquant_cache page: the class docstring's bit-packed
// key layout -- codebook indices at b_mse bits and QJL sign bits at one bit
// each -- __init__'s sign and residual-norm arrays and outlier cache,
// append_key, _unpack_signs_block and memory_bytes).  For key t of a slot:
//   split   (n_out > 0 and t >= split_from): o = x[channels] is stored as
//           int8 codes with an fp16 scale s = max(max|o| / 127, 1e-8), and
//           those channels of x are set to 0;
//   MSE     u = R^T x / ||x||, idx_k = the nearest centroid (the lower one at
//           a midpoint), fp16 norm n16;
//   sketch  (m > 0) r = x - n16 R c[idx]; sign bit j = [(S r)_j > 0]; the
//           residual norm ||r|| in fp16.
// Fetch returns n16 R c[idx] + sqrt(pi/2)/m ||r||16 S^T (2 bits - 1) plus the
// outlier channels' int8 decode.
//
// CUDA cores, one CTA per (tile of tokens, slot).  The products run as
// register-tiled fp32 GEMMs from shared memory against the layer's tables in
// global memory (L1/L2-resident), summed 16 terms at a time, so a sum of K
// terms carries at most gamma_{16 + K/16} sum |terms| of rounding error.  The
// integer decisions (centroid indices, sign bits, outlier codes) and the fp16
// norm are made as exact arithmetic makes them: each has a fast fp32 value
// with a proven bound, and the few within their bound of a boundary are
// re-decided in float64 (indices, norms, outlier codes) or double-float
// arithmetic (sign bits, which need the residual exactly).  The residual norm
// is a stored floating-point value: its fp32 value is rounded to fp16.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "kvc_ff.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kU = 5.9604644775390625e-08f;  // 2^-24
constexpr int kPThreads = 256;
constexpr int kTT = 32;        // tokens per append tile
constexpr int kFT = 64;        // tokens per fetch tile
constexpr int kBlk = 16;       // terms per partial sum
constexpr int kW1 = 256;       // columns of W1: R in 0 .. D-1, S^T in 128 .. 128+m-1
constexpr int kY = 128;        // first column of S x in W1 and in the z | S x tile
constexpr int kW2 = 128;       // columns of (S R)^T (zero beyond m)
constexpr float kQjlCoef = 1.2533141373155003f;  // sqrt(pi / 2)

__device__ __forceinline__ float gamma_n(int n) { return (float)n * kU / (1.f - (float)n * kU); }

__device__ __forceinline__ float load_in(const void* x, int dt, int64_t off) {
  if (dt == KVC_F32) return static_cast<const float*>(x)[off];
  if (dt == KVC_F16) return __half2float(static_cast<const __half*>(x)[off]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[off]);
}

__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_sumd(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ ff2 warp_sum_ff(ff2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff2 w{__shfl_xor_sync(kFull, v.hi, o), __shfl_xor_sync(kFull, v.lo, o)};
    v = ff_add(v, w);
  }
  return v;
}

// True when every real in [lo, hi] rounds to the same fp16.
__device__ __forceinline__ bool same_half(float lo, float hi) {
  return __half_as_ushort(__float2half_rn(lo)) == __half_as_ushort(__float2half_rn(hi));
}

// acc[i][j] = sum_k A[r0 + i][k] B[k][c0 + j], i < TM, j < 8; A in shared
// memory (row stride lda), B in global memory (row stride ldb floats, rows
// 16-byte aligned), K a multiple of kBlk.
template <int TM>
__device__ __forceinline__ void gemm_rows(const float* As, int lda, const float* __restrict__ B,
                                          int ldb, int K, int r0, int c0, float (&acc)[TM][8]) {
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int k0 = 0; k0 < K; k0 += kBlk) {
    float part[TM][8];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[i][j] = 0.f;
#pragma unroll 4
    for (int k = k0; k < k0 + kBlk; ++k) {
      const float4 b0 = __ldg(reinterpret_cast<const float4*>(B + (size_t)k * ldb + c0));
      const float4 b1 = __ldg(reinterpret_cast<const float4*>(B + (size_t)k * ldb + c0 + 4));
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const float a = As[(r0 + i) * lda + k];
#pragma unroll
        for (int j = 0; j < 8; ++j) part[i][j] = fmaf(a, bv[j], part[i][j]);
      }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] += part[i][j];
  }
}

// The same product with B staged through shared memory in chunks of kBlk
// rows (Bs: kBlk x NC floats, NC the columns staged, a multiple of 8), the
// next chunk's global loads in flight while the current one is used.  The
// thread's 8 columns are c0 .. c0 + 3 and NC/2 + c0 .. NC/2 + c0 + 3 (c0 a
// multiple of 4), so a warp's 16-byte reads of a B row are contiguous.  Every
// thread of the CTA calls it (it synchronises).
template <int TM, int NC>
__device__ __forceinline__ void gemm_staged(const float* As, int lda, const float* __restrict__ B,
                                            int ldb, int K, float* Bs, int r0, int c0,
                                            float (&acc)[TM][8]) {
  constexpr int kVec = kBlk * NC / 4;                    // float4s per chunk
  constexpr int kPer = (kVec + kPThreads - 1) / kPThreads;
  const int tid = threadIdx.x;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  float4 pre[kPer];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int v = tid + q * kPThreads;
      if (v < kVec) {
        const int rr = v / (NC / 4), cc = v - rr * (NC / 4);
        pre[q] = __ldg(reinterpret_cast<const float4*>(B + (size_t)(k0 + rr) * ldb) + cc);
      }
    }
  };
  fetch(0);
  for (int k0 = 0; k0 < K; k0 += kBlk) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int v = tid + q * kPThreads;
      if (v < kVec) reinterpret_cast<float4*>(Bs)[v] = pre[q];
    }
    __syncthreads();
    if (k0 + kBlk < K) fetch(k0 + kBlk);
    float part[TM][8];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[i][j] = 0.f;
#pragma unroll 4
    for (int k = 0; k < kBlk; ++k) {
      const float4 b0 = *reinterpret_cast<const float4*>(Bs + k * NC + c0);
      const float4 b1 = *reinterpret_cast<const float4*>(Bs + k * NC + NC / 2 + c0);
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const float a = As[(r0 + i) * lda + k0 + k];
#pragma unroll
        for (int j = 0; j < 8; ++j) part[i][j] = fmaf(a, bv[j], part[i][j]);
      }
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] += part[i][j];
    __syncthreads();  // the chunk is overwritten next
  }
}

// Shared-memory layout of the append tile (floats unless noted).
struct AppSmem {
  static constexpr int xs = 0;                          // [kTT][D] x with outliers zeroed
  static constexpr int zy = xs + kTT * kProdMaxD;       // [kTT][kW1] z | S x; (S R) c over z
  static constexpr int cs = zy + kTT * kW1;             // [kTT][D + 4] c[idx] (padded rows)
  static constexpr int tok = cs + kTT * (kProdMaxD + 4);  // [kTT][8] per-token scalars
  // scratch: the staged B chunks of the products, then the residuals of the
  // exact sign decisions ([8 warps][2][D]) and the sign queue (int [kTT m + 1])
  static constexpr int scr = tok + kTT * 8;
  static constexpr int rr = scr;
  static constexpr int nscr = 8 * 2 * kProdMaxD + (kTT * kProdMaxM + 1);
  static constexpr int nfloats = scr + (nscr > kBlk * kW1 ? nscr : kBlk * kW1);
  static constexpr int idx_b = nfloats * 4;             // bytes: [kTT][D] centroid indices
  static constexpr int sgn_b = idx_b + kTT * kProdMaxD;  // [kTT][m] sign bits
  static constexpr int o8_b = sgn_b + kTT * kProdMaxM;  // [kTT][n_out] outlier codes
  static constexpr int q_b = (rr + 8 * 2 * kProdMaxD) * 4;  // the sign queue, inside scr
  static constexpr int row_b = o8_b + kTT * kProdMaxOut;  // [kTT][P] staged rows
  static constexpr int bytes(int P) { return row_b + kTT * P + 16; }
};
// per-token scalars in AppSmem::tok
enum { kN32 = 0, kN16, kNB, kCN, kZC, kG16, kOS, kValid };

template <int D>
__global__ void __launch_bounds__(kPThreads, 2) append_prod_kernel(const Params p, const AppendArgs a) {
  extern __shared__ __align__(16) unsigned char sm[];
  float* fsm = reinterpret_cast<float*>(sm);
  float* xs = fsm + AppSmem::xs;
  float* zy = fsm + AppSmem::zy;
  float* cs = fsm + AppSmem::cs;
  float* tk = fsm + AppSmem::tok;
  uint8_t* idx_s = sm + AppSmem::idx_b;
  uint8_t* sgn_s = sm + AppSmem::sgn_b;
  int8_t* o8_s = reinterpret_cast<int8_t*>(sm + AppSmem::o8_b);
  int* queue = reinterpret_cast<int*>(sm + AppSmem::q_b);
  uint8_t* row_s = sm + AppSmem::row_b;

  constexpr int CS = D + 4;  // row stride of cs: rows 2 apart fall in different banks
  const int m = p.m, nout = p.n_out, L = p.cb_levels;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slot = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kTT;
  const int nt = (int)min((int64_t)kTT, a.T - t0);
  const int b = slot / p.H, h = slot - b * p.H;
  const int64_t xbase = (int64_t)b * a.sb + (int64_t)h * a.sh;
  __shared__ float cb[256], mids[256], vn[kProdMaxD];
  for (int j = tid; j < L; j += kPThreads) {
    cb[j] = p.codebook[j];
    if (j + 1 < L) mids[j] = p.mids[j];
  }
  for (int k = tid; k < D; k += kPThreads) vn[k] = p.vnorm[k];

  // 1. rows (fp32; rows past the call's end are zero)
  for (int e = tid; e < kTT * D; e += kPThreads) {
    const int t = e / D, i = e - t * D;
    xs[t * D + i] = t < nt ? load_in(a.x, p.in_dtype, xbase + (t0 + t) * a.st + i) : 0.f;
  }
  __syncthreads();

  // 2. outlier split and 3. norms, one warp per token
  unsigned n_ref_side = 0;
  for (int t = warp; t < kTT; t += kPThreads / 32) {
    const int64_t tg = a.t_base + t0 + t;
    float* x = xs + t * D;
    if (nout) {
      const bool split = t < nt && tg >= p.split_from;
      float v = 0.f;
      int ch = 0;
      if (lane < nout) {
        ch = p.channels[(size_t)slot * nout + lane];
        v = split ? x[ch] : 0.f;
      }
      const float amax = warp_maxf(fabsf(v));
      // s = max(amax / 127, 1e-8) as float64 computes it; amax < 2e-6 (the
      // floor, subnormal scales) takes float64 throughout
      const bool tiny_o = amax < 2e-6f;
      float s16 = 0.f;
      if (split) {
        float q;
        if (tiny_o) {
          q = (float)rint((double)v / fmax((double)amax / 127.0, 1e-8));
        } else {
          const float u = v * (127.f / amax);  // within 1.5e-5 of v / s
          const float au = fabsf(u);
          q = rintf(u);
          if (fabsf(au - floorf(au) - 0.5f) < 1e-4f) q = (float)rint((double)v / ((double)amax / 127.0));
        }
        if (lane < nout) o8_s[t * kProdMaxOut + lane] = (int8_t)fminf(fmaxf(q, -127.f), 127.f);
        // fp16(s): fl32(amax / 127) and float64's value both lie within 2u of
        // amax / 127, so one fp16 for that interval decides it
        const float s32 = amax / 127.f;
        if (!tiny_o && same_half(s32 * (1.f - 2.f * kU), s32 * (1.f + 2.f * kU)))
          s16 = __half2float(__float2half_rn(s32));
        else
          s16 = __half2float(__double2half(fmax((double)amax / 127.0, 1e-8)));
      } else if (lane < nout) {
        o8_s[t * kProdMaxOut + lane] = 0;
      }
      __syncwarp();
      if (split && lane < nout) x[ch] = 0.f;
      __syncwarp();
      if (lane == 0) tk[t * 8 + kOS] = s16;
    }
    // ||x||: lane-sequential sums and a 5-level tree: |error| <= gamma_{D/32+5} ||x||^2
    float s2 = 0.f;
    for (int i = lane; i < D; i += 32) s2 = fmaf(x[i], x[i], s2);
    s2 = warp_sumf(s2);
    const float g = gamma_n(D / 32 + 5);
    const float n32 = sqrtf(s2);
    float n16;
    if (same_half(sqrtf(s2 * (1.f - g)) * (1.f - kU), sqrtf(s2 * (1.f + 2.f * g)) * (1.f + 2.f * kU))) {
      n16 = __half2float(__float2half_rn(n32));
    } else {
      double d2 = 0.0;
      for (int i = lane; i < D; i += 32) d2 = fma((double)x[i], (double)x[i], d2);
      d2 = warp_sumd(d2);
      n16 = __half2float(__double2half(sqrt(d2)));
      if (lane == 0) ++n_ref_side;
    }
    if (lane == 0) {
      tk[t * 8 + kN32] = n32;
      tk[t * 8 + kN16] = n16;
      tk[t * 8 + kNB] = n32 * (1.f + g) + 1e-30f;  // >= ||x||
      tk[t * 8 + kValid] = t < nt ? 1.f : 0.f;
    }
  }
  __syncthreads();

  // 4. z | S x = x W1: thread (ty, tx) takes tokens 4 ty .. 4 ty + 3, columns 8 tx ..
  {
    const int tx = tid & 31, ty = tid >> 5;
    float acc[4][8];
    gemm_staged<4, kW1>(xs, D, p.W1, kW1, D, fsm + AppSmem::scr, 4 * ty, 4 * tx, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float* o = zy + (4 * ty + i) * kW1 + 4 * tx;
      *reinterpret_cast<float4*>(o) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(o + kW1 / 2) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
  }
  __syncthreads();

  // 5. centroid indices: idx = #{midpoints < z / ||x||}, exact near a midpoint
  unsigned n_ref_code = 0;
  const float gz = gamma_n(kBlk + D / kBlk);
  const float gn = gamma_n(D / 32 + 5);
  for (int e = tid; e < kTT * D; e += kPThreads) {
    const int t = e / D, k = e - t * D;
    const float z = zy[t * kW1 + k];
    const float n32 = tk[t * 8 + kN32];
    const bool tiny = n32 < 1e-18f;  // ||x||^2 may have underflowed: float64 path
    const float u = tiny ? 0.f : z / n32;
    int lo = 0, hi = L - 1;  // first index j with u <= mids[j] (L - 1 if none)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (u <= mids[mid]) hi = mid; else lo = mid + 1;
    }
    int idx = lo;
    // |u32 - z / ||x|| | <= gamma_z ||R_k|| + (gamma_n / 2 + 2u) |u32|
    const float del = 1.02f * (gz * vn[k] + (0.5f * gn + 2.f * kU) * fabsf(u)) + 1e-30f;
    const bool near = (idx > 0 && u - mids[idx - 1] <= del) || (idx < L - 1 && mids[idx] - u <= del);
    if ((near || tiny) && tk[t * 8 + kValid] != 0.f) {
      // float64: z and ||x|| summed in float64, then the oracle's comparison
      // of |u - c_j| (the lower index on equal distances)
      const float* x = xs + t * D;
      double z64 = 0.0, n2 = 0.0;
      for (int i = 0; i < D; ++i) {
        z64 = fma((double)x[i], (double)p.Vt[(size_t)k * D + i], z64);
        n2 = fma((double)x[i], (double)x[i], n2);
      }
      const double u64 = n2 > 0.0 ? z64 / sqrt(n2) : 0.0;
      int best = 0;
      double bd = fabs(u64 - (double)cb[0]);
      for (int j = 1; j < L; ++j) {
        const double dj = fabs(u64 - (double)cb[j]);
        if (dj < bd) {
          bd = dj;
          best = j;
        }
      }
      idx = best;
      ++n_ref_code;
    }
    idx_s[t * kProdMaxD + k] = (uint8_t)idx;
    cs[t * CS + k] = cb[idx];
  }
  __syncthreads();

  // 6. per token: ||c[idx]||, <z, c>, and the residual norm
  //    ||r||^2 = ||x||^2 - 2 n16 <z, c> + n16^2 ||R c||^2 with ||R c|| = ||c||
  //    to fp32 precision (R orthogonal); rounded to fp16
  for (int t = warp; t < kTT; t += kPThreads / 32) {
    float c2 = 0.f, zc = 0.f, x2 = 0.f;
    for (int k = lane; k < D; k += 32) {
      const float c = cs[t * CS + k];
      c2 = fmaf(c, c, c2);
      zc = fmaf(zy[t * kW1 + k], c, zc);
      x2 = fmaf(xs[t * D + k], xs[t * D + k], x2);
    }
    c2 = warp_sumf(c2);
    zc = warp_sumf(zc);
    x2 = warp_sumf(x2);
    if (lane == 0) {
      const float n16 = tk[t * 8 + kN16];
      const float g2 = fmaxf(x2 - 2.f * n16 * zc + n16 * n16 * c2, 0.f);
      tk[t * 8 + kCN] = sqrtf(c2) * (1.f + 1e-6f) + 1e-30f;
      tk[t * 8 + kG16] = __half2float(__float2half_rn(sqrtf(g2)));
    }
  }
  __syncthreads();

  // 7. (S R) c[idx] into zy's first columns (z is no longer needed)
  if (m) {
    const int tx = tid & 15, ty = tid >> 4;  // tokens 2 ty, 2 ty + 1; columns 8 tx ..
    float acc[2][8];
    gemm_staged<2, kW2>(cs, CS, p.SRt, kW2, D, fsm + AppSmem::scr, 2 * ty, 4 * tx, acc);
    if (tid == 0) queue[kTT * kProdMaxM] = 0;  // the scratch holds the queue from here
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float* o = zy + (2 * ty + i) * kW1 + 4 * tx;
      *reinterpret_cast<float4*>(o) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      *reinterpret_cast<float4*>(o + kW2 / 2) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    __syncthreads();

    // 8. sign bits: s_j = (S x)_j - n16 ((S R) c)_j, with
    //    |s32 - s| <= gamma_z ||S_j|| ||x|| + n16 (gamma_z + 2u) ||(S R)_j|| ||c||
    //                 + u n16 |(S R c)_j| + u |s32|
    for (int e = tid; e < kTT * kProdMaxM; e += kPThreads) {
      const int t = e >> 7, j = e & (kProdMaxM - 1);
      if (j >= m) continue;
      const float y = zy[t * kW1 + kY + j], tq = zy[t * kW1 + j];
      const float n16 = tk[t * 8 + kN16];
      const float s = fmaf(-n16, tq, y);
      const float tau = 1.02f * (gz * p.s_norm[j] * tk[t * 8 + kNB] +
                                 n16 * (gz + 2.f * kU) * p.sr_norm[j] * tk[t * 8 + kCN] +
                                 kU * n16 * fabsf(tq) + kU * fabsf(s)) + 1e-30f;
      uint8_t bit = s > 0.f ? 1 : 0;
      if (fabsf(s) <= tau && tk[t * 8 + kValid] != 0.f) {
        const int qi = atomicAdd(&queue[kTT * kProdMaxM], 1);
        queue[qi] = t * m + j;
      }
      sgn_s[t * kProdMaxM + j] = bit;
    }
    __syncthreads();

    // 9. exact sign decisions: per queued (token, j), the residual in
    //    double-float (r = x - n16 R c, every term split exactly), then S_j . r
    const int nq = queue[kTT * kProdMaxM];
    float* rh = fsm + AppSmem::rr + warp * 2 * kProdMaxD;
    float* rl = rh + kProdMaxD;
    int last_t = -1;
    for (int qi = warp; qi < nq; qi += kPThreads / 32) {
      const int e = queue[qi];
      const int t = e / m, j = e - t * m;
      const float n16 = tk[t * 8 + kN16];
      if (t != last_t) {
        __syncwarp();
        for (int i = lane; i < D; i += 32) {
          ff2 w{0.f, 0.f};
          for (int k = 0; k < D; ++k) w = ff_add(w, ff_mul(ff2{p.Vt[(size_t)k * D + i], 0.f}, ff2{cs[t * CS + k], 0.f}));
          const ff2 r = ff_add(ff2{xs[t * D + i], 0.f}, ff_mul(ff2{-n16, 0.f}, w));
          rh[i] = r.hi;
          rl[i] = r.lo;
        }
        __syncwarp();
        last_t = t;
      }
      ff2 acc{0.f, 0.f};
      for (int i = lane; i < D; i += 32)
        acc = ff_add(acc, ff_mul(ff2{p.W3[(size_t)(D + j) * D + i], 0.f}, ff2{rh[i], rl[i]}));
      acc = warp_sum_ff(acc);
      if (lane == 0) sgn_s[t * kProdMaxM + j] = (acc.hi > 0.f || (acc.hi == 0.f && acc.lo > 0.f)) ? 1 : 0;
    }
    if (lane == 0 && nq && warp == 0) atomicAdd(&p.counters[0], (unsigned long long)nq);
  }
  __syncthreads();

  // 10. rows: [codes | sign bits | outlier int8], staged, then copied out
  const int cbytes = p.code_bytes, sbytes = p.sign_bytes, bw = p.cb_bits;
  const int P = cbytes + sbytes + nout;
  for (int e = tid; e < nt * P; e += kPThreads) {
    const int t = e / P, c = e - t * P;
    uint32_t v = 0;
    if (c < cbytes) {
      // codes k with bits [k bw, k bw + bw) meeting [8 c, 8 c + 8)
      for (int k = (8 * c) / bw; k < D && k * bw < 8 * c + 8; ++k) {
        const int sh = k * bw - 8 * c;
        const uint32_t code = idx_s[t * kProdMaxD + k];
        v |= sh >= 0 ? code << sh : code >> -sh;
      }
      v &= 0xffu;
    } else if (c < cbytes + sbytes) {
      const int j0 = 8 * (c - cbytes);
      for (int q = 0; q < 8 && j0 + q < m; ++q) v |= (uint32_t)sgn_s[t * kProdMaxM + j0 + q] << q;
    } else {
      v = (uint8_t)o8_s[t * kProdMaxOut + (c - cbytes - sbytes)];
    }
    row_s[e] = (uint8_t)v;
  }
  __syncthreads();
  uint8_t* dst = p.store + p.pay_off[slot] + (a.t_base + t0) * (int64_t)P;
  for (int e = tid; e < nt * P; e += kPThreads) dst[e] = row_s[e];
  __half* side = reinterpret_cast<__half*>(p.store + p.side_off[slot]);
  const int nw = p.side_bytes / 2;
  for (int t = tid; t < nt; t += kPThreads) {
    const int64_t r = (a.t_base + t0 + t) * nw;
    int w = 0;
    side[r + w++] = __float2half_rn(tk[t * 8 + kN16]);
    if (m) side[r + w++] = __float2half_rn(tk[t * 8 + kG16]);
    if (nout) side[r + w++] = __float2half_rn(tk[t * 8 + kOS]);
  }
  n_ref_code = __reduce_add_sync(kFull, n_ref_code);
  n_ref_side = __reduce_add_sync(kFull, n_ref_side);
  if (lane == 0 && n_ref_code) atomicAdd(&p.counters[0], (unsigned long long)n_ref_code);
  if (lane == 0 && n_ref_side) atomicAdd(&p.counters[1], (unsigned long long)n_ref_side);
  if (tid == 0 && slot == 0) atomicAdd(&p.counters[2], (unsigned long long)nt);
}

// Fetch: A = [n16 c[idx] | sqrt(pi/2)/m ||r||16 (2 bits - 1)] per token,
// x_hat = A [R^T ; S] (+ the outlier channels' int8 decode).  Thread (ty, tx)
// takes tokens TM ty .., columns 8 tx ..; TX = D / 8 column groups.
template <int D>
__global__ void __launch_bounds__(kPThreads) fetch_prod_kernel(const Params p, const FetchArgs f) {
  constexpr int TX = D / 8, TY = kPThreads / TX, TM = kFT / TY;
  extern __shared__ __align__(16) unsigned char sm[];
  const int m = p.m, nout = p.n_out, K = D + m, KA = K + 4;  // KA: padded row stride of A
  float* A = reinterpret_cast<float*>(sm);           // [kFT][KA]
  float* osc = A + kFT * (D + kProdMaxM + 4);        // [kFT]
  float* Bs = osc + kFT;                             // [kBlk][D] staged rows of W3
  uint8_t* rows = reinterpret_cast<uint8_t*>(Bs + kBlk * D);  // [kFT][P]
  const int tid = threadIdx.x;
  const int slot = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kFT;
  const int nt = (int)min((int64_t)kFT, f.S - t0);
  const int cbytes = p.code_bytes, bw = p.cb_bits, nw = p.side_bytes / 2;
  const int P = cbytes + p.sign_bytes + nout;
  const uint8_t* src = p.store + p.pay_off[slot] + t0 * (int64_t)P;
  for (int e = tid; e < nt * P; e += kPThreads) rows[e] = src[e];
  __syncthreads();
  const __half* side = reinterpret_cast<const __half*>(p.store + p.side_off[slot]);
  const float coef = m ? kQjlCoef / (float)m : 0.f;
  for (int e = tid; e < kFT * K; e += kPThreads) {
    const int t = e / K, k = e - t * K;
    float v = 0.f;
    if (t < nt) {
      const uint8_t* row = rows + t * P;
      if (k < D) {
        const int pos = k * bw;
        uint32_t bits = row[pos >> 3] | ((pos >> 3) + 1 < cbytes ? (uint32_t)row[(pos >> 3) + 1] << 8 : 0u);
        const int idx = (int)((bits >> (pos & 7)) & ((1u << bw) - 1u));
        v = __half2float(side[(t0 + t) * nw]) * p.codebook[idx];
      } else {
        const int j = k - D;
        const int bit = (row[cbytes + (j >> 3)] >> (j & 7)) & 1;
        v = coef * __half2float(side[(t0 + t) * nw + 1]) * (bit ? 1.f : -1.f);
      }
    }
    A[t * KA + k] = v;
  }
  if (nout)
    for (int t = tid; t < kFT; t += kPThreads)
      osc[t] = t < nt ? __half2float(side[(t0 + t) * nw + nw - 1]) : 0.f;
  __syncthreads();
  const int tx = tid % TX, ty = tid / TX;
  float acc[TM][8];
  gemm_staged<TM, D>(A, KA, p.W3, D, K, Bs, TM * ty, 4 * tx, acc);
  const int b = slot / p.H, h = slot - b * p.H;
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int t = TM * ty + i;
    if (t >= nt) continue;
    float v[8];  // columns 4 tx .. 4 tx + 3 and D/2 + 4 tx .. D/2 + 4 tx + 3
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = acc[i][j];
    if (nout) {
      const int8_t* o8 = reinterpret_cast<const int8_t*>(rows + t * P + cbytes + p.sign_bytes);
      const int32_t* ch = p.channels + (size_t)slot * nout;
      for (int l = 0; l < nout; ++l) {
        const int c = ch[l];
        const int j = c - 4 * tx >= 0 && c - 4 * tx < 4 ? c - 4 * tx
                      : (c - D / 2 - 4 * tx >= 0 && c - D / 2 - 4 * tx < 4 ? 4 + c - D / 2 - 4 * tx : -1);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q == j) v[q] += (float)o8[l] * osc[t];
      }
    }
    const int64_t row0 = (((int64_t)b * p.H + h) * f.ld_s + t0 + t) * D;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int64_t base = row0 + half * (D / 2) + 4 * tx;
      if (p.out_dtype == KVC_F16) {
        __align__(8) __half o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __float2half_rn(v[4 * half + j]);
        *reinterpret_cast<uint2*>(static_cast<__half*>(f.out) + base) = *reinterpret_cast<const uint2*>(o);
      } else {
        __align__(8) __nv_bfloat16 o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = __float2bfloat16_rn(v[4 * half + j]);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(f.out) + base) =
            *reinterpret_cast<const uint2*>(o);
      }
    }
  }
}

// Outlier channels of a slot: the n_out largest mean |x_c| over the first n
// rows (float64 sums in row order, then / n), the lower channel first among
// equals, written in ascending channel order.
__global__ void __launch_bounds__(kPThreads) fit_outliers_kernel(const void* x, int dt, int H, int D,
                                                                 int64_t n, int64_t sb, int64_t sh,
                                                                 int64_t st, int n_out,
                                                                 int32_t* channels) {
  __shared__ double score[256];
  __shared__ int sel[256];
  const int slot = blockIdx.x, tid = threadIdx.x;
  const int b = slot / H, h = slot - b * H;
  const int64_t base = (int64_t)b * sb + (int64_t)h * sh;
  for (int c = tid; c < D; c += kPThreads) {
    double s = 0.0;
    for (int64_t t = 0; t < n; ++t) s += fabs((double)load_in(x, dt, base + t * st + c));
    score[c] = s / (double)n;
  }
  __syncthreads();
  for (int c = tid; c < D; c += kPThreads) {
    int rank = 0;
    for (int o = 0; o < D; ++o) rank += score[o] > score[c] || (score[o] == score[c] && o < c);
    sel[c] = rank < n_out;
  }
  __syncthreads();
  for (int c = tid; c < D; c += kPThreads)
    if (sel[c]) {
      int pos = 0;
      for (int o = 0; o < c; ++o) pos += sel[o];
      channels[(size_t)slot * n_out + pos] = c;
    }
}

}  // namespace

cudaError_t launch_fit_outliers(const void* x, int dt, int B, int H, int D, int64_t n, int64_t sb,
                                int64_t sh, int64_t st, int n_out, int32_t* channels,
                                cudaStream_t s) {
  fit_outliers_kernel<<<B * H, kPThreads, 0, s>>>(x, dt, H, D, n, sb, sh, st, n_out, channels);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_append_prod_d(const Params& p, const AppendArgs& a, cudaStream_t s) {
  const int P = p.code_bytes + p.sign_bytes + p.n_out;
  const size_t smem = (size_t)AppSmem::bytes(P);
  cudaError_t e = cudaFuncSetAttribute(append_prod_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((a.T + kTT - 1) / kTT), (unsigned)p.n_slots);
  append_prod_kernel<D><<<grid, kPThreads, smem, s>>>(p, a);
  return cudaGetLastError();
}

cudaError_t launch_append_prod(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk) {
  ++*nk;
  switch (p.D) {
    case 32: return launch_append_prod_d<32>(p, a, s);
    case 64: return launch_append_prod_d<64>(p, a, s);
    case 128: return launch_append_prod_d<128>(p, a, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int D>
static cudaError_t launch_fetch_prod_d(const Params& p, const FetchArgs& f, cudaStream_t s) {
  const int P = p.code_bytes + p.sign_bytes + p.n_out;
  const size_t smem = (size_t)kFT * (D + kProdMaxM + 4) * 4 + kFT * 4 + (size_t)kBlk * D * 4 +
                      (size_t)kFT * P + 16;
  cudaError_t e = cudaFuncSetAttribute(fetch_prod_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((f.S + kFT - 1) / kFT), (unsigned)p.n_slots);
  fetch_prod_kernel<D><<<grid, kPThreads, smem, s>>>(p, f);
  return cudaGetLastError();
}

cudaError_t launch_fetch_prod(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk) {
  ++*nk;
  switch (p.D) {
    case 32: return launch_fetch_prod_d<32>(p, f, s);
    case 64: return launch_fetch_prod_d<64>(p, f, s);
    case 128: return launch_fetch_prod_d<128>(p, f, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvc
