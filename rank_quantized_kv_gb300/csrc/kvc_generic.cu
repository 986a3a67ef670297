// CUDA-core kernels of the KV cache hot path: any shape, any input dtype.
//
// Append: each CTA takes TT tokens of one slot.  The projection runs in fp32
// on the CUDA cores (sequential FMA over the input dimension, so the
// textbook bound |z32 - z| <= gamma_{n} * sum_i |x_i - m_i| |V_ik| holds with
// gamma_n = n u / (1 - n u), u = 2^-24).  Every code whose fp32 value lies
// within that bound (carried through the quantiser's own roundings) of a
// rounding boundary is re-decided in double precision by one warp, so the
// stored codes are the ones exact arithmetic gives (and float64 with it,
// except at ties closer than float64's own error).
//
// Fetch: each CTA takes TT tokens of one slot, unpacks and dequantises into
// shared memory, then reconstructs x_hat = z_hat V^T + mean in fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_ff.cuh"
#include "kvc_internal.h"
#include "kvc_tc.h"

namespace kvc {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kU = 5.9604644775390625e-08f;  // 2^-24

__device__ __forceinline__ float load_in(const void* x, int dt, int64_t off) {
  if (dt == KVC_F32) return static_cast<const float*>(x)[off];
  if (dt == KVC_F16) return __half2float(static_cast<const __half*>(x)[off]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(x)[off]);
}

__device__ __forceinline__ void store_out(void* out, int dt, int64_t off, float v) {
  if (dt == KVC_F16)
    static_cast<__half*>(out)[off] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// q / d for 0 <= q < 2^21 without an integer division: (q + 1/2) / d lies at
// least 1/(2d) from an integer, and the two float roundings move it by less.
__device__ __forceinline__ int small_div(int q, float inv_d) {
  return __float2int_rd(((float)q + 0.5f) * inv_d);
}

// gamma_n = n u / (1 - n u)
__device__ __forceinline__ float gamma_n(int n) {
  const float nu = n * kU;
  return nu / (1.f - nu);
}

// The projection sums d_in products in blocks of kProjBlk (fp32 fma), then
// adds the block sums: every term passes through at most kProjBlk + (number
// of blocks) roundings, plus one for x - mean, so the error is at most
// gamma_{that + 1} sum |(x_i - m_i) V_ik| <= gamma ||x - m|| ||V_k||.
constexpr int kProjBlk = 32;
__device__ __forceinline__ float proj_gamma(int d_in) {
  return gamma_n(kProjBlk + (d_in + kProjBlk - 1) / kProjBlk + 2);
}

// sum_i (x_i - m_i) * w_i in double precision, one warp, result on every lane.
__device__ __forceinline__ double dot64(const float* x, const float* m, const float* w, int n,
                                        int lane) {
  double acc = 0.0;
  for (int i = lane; i < n; i += 32) acc = fma((double)x[i] - (double)m[i], (double)w[i], acc);
  return warp_sum(acc);
}

// sum_i (x_i - m_i) * w_i as a double-float (compensated fp32: x - m and each
// product split exactly, TwoSum accumulation), one warp, on every lane.
__device__ __forceinline__ void dot_ff_term(float xi, float mi, float wi, float& S, float& C) {
  float dh, dl;
  two_sum(xi, -mi, dh, dl);
  const float pr = dh * wi;
  const float pe = fmaf(dh, wi, -pr);
  float s, e;
  two_sum(S, pr, s, e);
  S = s;
  C += pe + e + dl * wi;
}

__device__ __forceinline__ ff2 dot_ff(const float* x, const float* m, const float* w, int n,
                                      int lane) {
  float S = 0.f, C = 0.f;
  if ((n & 3) == 0) {  // 4 consecutive terms per lane and load (16-byte aligned rows)
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* m4 = reinterpret_cast<const float4*>(m);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int n4 = n >> 2;
    int j = lane;
    for (; j + 96 < n4; j += 128) {  // four loads of w in flight per lane
      float4 wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) wv[u] = __ldg(w4 + j + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float4 xv = x4[j + 32 * u], mv = m4[j + 32 * u];
        dot_ff_term(xv.x, mv.x, wv[u].x, S, C);
        dot_ff_term(xv.y, mv.y, wv[u].y, S, C);
        dot_ff_term(xv.z, mv.z, wv[u].z, S, C);
        dot_ff_term(xv.w, mv.w, wv[u].w, S, C);
      }
    }
    for (; j < n4; j += 32) {
      const float4 xv = x4[j], mv = m4[j], wv = __ldg(w4 + j);
      dot_ff_term(xv.x, mv.x, wv.x, S, C);
      dot_ff_term(xv.y, mv.y, wv.y, S, C);
      dot_ff_term(xv.z, mv.z, wv.z, S, C);
      dot_ff_term(xv.w, mv.w, wv.w, S, C);
    }
  } else {
    for (int i = lane; i < n; i += 32) dot_ff_term(x[i], m[i], w[i], S, C);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float So = __shfl_xor_sync(kFull, S, o);
    const float Co = __shfl_xor_sync(kFull, C, o);
    float s, e;
    two_sum(S, So, s, e);
    S = s;
    C = C + Co + e;
  }
  float s, e;
  two_sum(S, C, s, e);
  return ff2{s, e};
}

// sum_i (x_i - m_i) * w_i in fp32, one warp, on every lane: each lane keeps
// four fma chains (one per component of its 16-byte loads), so no chain is
// longer than L = ceil(n / 128) terms (ceil(n / 32) for rows that are not
// 16-byte multiples); the chains and the lanes are then added with TwoSum
// into a double-float.  Error bound, u = 2^-24:
//   |result - sum (x_i - m_i) w_i| <= (gamma_L (1 + u) + u + 2^-40) sum |x_i - m_i| |w_i|
// (gamma_L for the chains, u for the rounding of x - m, 2^-40 for the
// compensated sums).  mid_gamma(n) is that factor.
__device__ __forceinline__ float mid_gamma(int n) {
  const int L = (n & 3) == 0 ? (n + 127) / 128 : (n + 31) / 32;
  return gamma_n(L) * (1.f + kU) + kU + 1e-12f;
}

__device__ __forceinline__ ff2 dot_mid(const float* x, const float* m, const float* w, int n,
                                       int lane) {
  float c0 = 0.f, c1 = 0.f, c2 = 0.f, c3 = 0.f;
  if ((n & 3) == 0) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const float4* m4 = reinterpret_cast<const float4*>(m);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int n4 = n >> 2;
#pragma unroll 4
    for (int j = lane; j < n4; j += 32) {
      const float4 xv = x4[j], mv = m4[j], wv = __ldg(w4 + j);
      c0 = fmaf(xv.x - mv.x, wv.x, c0);
      c1 = fmaf(xv.y - mv.y, wv.y, c1);
      c2 = fmaf(xv.z - mv.z, wv.z, c2);
      c3 = fmaf(xv.w - mv.w, wv.w, c3);
    }
  } else {
    for (int i = lane; i < n; i += 32) c0 = fmaf(x[i] - m[i], w[i], c0);
  }
  float S, C, e;
  two_sum(c0, c1, S, C);
  two_sum(S, c2, S, e);
  C += e;
  two_sum(S, c3, S, e);
  C += e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float So = __shfl_xor_sync(kFull, S, o);
    const float Co = __shfl_xor_sync(kFull, C, o);
    two_sum(S, So, S, e);
    C = C + Co + e;
  }
  two_sum(S, C, S, e);
  return ff2{S, e};
}

// sum_i x_i^2 in double precision, one warp.
__device__ __forceinline__ double sumsq64(const float* x, int n, int lane) {
  double acc = 0.0;
  for (int i = lane; i < n; i += 32) acc = fma((double)x[i], (double)x[i], acc);
  return warp_sum(acc);
}

// True when every value in [lo, hi] rounds to the same fp16.
__device__ __forceinline__ bool same_half(float lo, float hi) {
  return __half_as_ushort(__float2half_rn(lo)) == __half_as_ushort(__float2half_rn(hi));
}

// ---------------------------------------------------------------------------
// Quantisers: one warp per item, lane = component.
// ---------------------------------------------------------------------------

struct RowCtx {
  const float* xs;    // token row (fp32 copy of the input), d_in values
  const float* mean;  // basis mean, d_in values
  const float* zs;    // fp32 latents, r values
  float nrm;          // fp32 ||x - mean|| (||x|| in codebook mode)
  uint8_t* codes;     // r codes out
  __half* side;       // side words out
};

// Uniform: code = clip(rint((z - lo) / step), 0, 2^b - 1).
__device__ void quant_uniform(const Params& p, int beta, const float* vnorm, const RowCtx& c,
                              int chunk, int lane, unsigned* nref) {
  const int k = chunk * 32 + lane;
  const bool valid = k < p.r;
  const int w = valid ? p.bits[beta * p.r + k] : 0;
  const float gam = proj_gamma(p.d_in);
  int code = 0;
  bool near = false;
  float lo = 0.f, step = 1.f;
  int qmax = 0;
  if (w > 0) {
    lo = p.lo[beta * p.r + k];
    step = p.step[beta * p.r + k];
    const float inv = p.inv_step[beta * p.r + k];
    const float z = c.zs[k];
    const float u = (z - lo) * inv;
    const float tau_z = gam * c.nrm * vnorm[k] * (1.f + 1e-3f);
    const float tau_u = tau_z * inv * (1.f + 1e-6f) + 4.f * kU * (fabsf(u) + 1.f);
    qmax = (1 << w) - 1;
    // the interior boundary nearest u (0.5 .. qmax - 0.5): with a wide tau
    // the one below a clamped u counts too
    const float hb = fminf(fmaxf(floorf(u) + 0.5f, 0.5f), (float)qmax - 0.5f);
    near = fabsf(u - hb) <= tau_u;
    code = (int)fminf(fmaxf(rintf(u), 0.f), (float)qmax);
  }
  unsigned m = __ballot_sync(kFull, near);
  if (lane == 0 && m) atomicAdd(nref, (unsigned)__popc(m));
  while (m) {
    const int f = __ffs(m) - 1;
    m &= m - 1;
    const int kf = chunk * 32 + f;
    const double z64 =
        dot64(c.xs, c.mean, p.Vt + ((int64_t)beta * p.r + kf) * p.d_in, p.d_in, lane);
    if (lane == f) {
      const double u64 = (z64 - (double)lo) / (double)step;
      code = (int)fmin(fmax(rint(u64), 0.0), (double)qmax);
    }
  }
  if (valid && w > 0) c.codes[k] = (uint8_t)code;
}

// Error bound of the fp32 latents: |z32 - z| <= gamma n ||V_k|| + ex ||V_k|| + en n,
// n = ||x - mean||.
struct QBound {
  float gamma, ex, en;
};

// Group: per token and group, s = max(absmax / qmax, 1e-8); q = clip(rint(z / s)).
__device__ void quant_group(const Params& p, int beta, const float* vnorm, const RowCtx& c,
                            int gi, int lane, unsigned* nref, unsigned* nside, const QBound& qb) {
  const int first = p.groups[gi * 3 + 0];
  const int cnt = p.groups[gi * 3 + 1];
  const int w = p.groups[gi * 3 + 2];
  const int qmax = (1 << (w - 1)) - 1;
  const int off = 1 << (w - 1);
  const int k = first + lane;
  const bool valid = lane < cnt;
  const float z = valid ? c.zs[k] : 0.f;
  const float az = fabsf(z);
  const float tz =
      valid ? (qb.gamma * c.nrm * vnorm[k] + qb.ex * vnorm[k] + qb.en * c.nrm) * (1.f + 1e-3f) : 0.f;
  const float a32 = warp_maxf(valid ? az : 0.f);
  const float tzm = warp_maxf(tz);
  // Too close to zero (or to the 1e-8 floor) to trust the fp32 maximum.
  const bool full = a32 <= 2.f * tzm + (float)qmax * 4e-8f;
  const float s32 = a32 / (float)qmax;
  const float eps = full ? 0.f : tzm / a32 + 4.f * kU;
  const bool s_unsure = !full && !same_half(s32 * (1.f - eps), s32 * (1.f + eps));
  float u = full ? 0.f : z / s32;
  const float au = fabsf(u);
  const float tau_u = full ? 0.f : (tz / s32 + au * eps) * (1.f + 1e-6f) + 4.f * kU * (au + 1.f);
  // the interior boundary nearest |u| (0.5 .. qmax - 0.5)
  const float hb = fminf(floorf(au) + 0.5f, (float)qmax - 0.5f);
  const bool near = valid && !full && (fabsf(au - hb) <= tau_u);
  int q = (int)fminf(fmaxf(rintf(u), -(float)qmax), (float)qmax);
  __half s16 = __float2half_rn(s32);

  const unsigned vmask = __ballot_sync(kFull, valid);
  const unsigned nmask = full ? vmask : __ballot_sync(kFull, near);
  const bool flagged = full || s_unsure || nmask;
  bool decided = false;
  if (flagged) {
    // The scale needs the exact maximum: recompute every component that could hold it.
    const bool cand = valid && (full || az + tz >= a32 - tzm);
    const unsigned todo0 = __ballot_sync(kFull, cand) | nmask;
    if (lane == 0) {
      atomicAdd(nref, (unsigned)__popc(nmask));
      atomicAdd(nside, 1u);
    }
    // First those components again in fp32 with short fma chains (a bound
    // about 30 times tighter than the tensor-core one): that decides the
    // scale's fp16 rounding and the near codes in most groups.
    if (!full) {
      float zm = z, tm = tz;
      const float gm = mid_gamma(p.d_in);
      for (unsigned f_m = todo0; f_m; f_m &= f_m - 1) {
        const int f = __ffs(f_m) - 1;
        const ff2 z2 =
            dot_mid(c.xs, c.mean, p.Vt + ((int64_t)beta * p.r + first + f) * p.d_in, p.d_in, lane);
        if (lane == f) {
          zm = z2.hi + z2.lo;
          tm = gm * c.nrm * vnorm[k] * (1.f + 1e-3f) + kU * fabsf(zm);
        }
      }
      // the maximum is one of the candidates: a in [a_lo, a_hi], so
      // s = max(a / qmax, 1e-8) in [s_lo, s_hi]
      const float a_lo = warp_maxf(cand ? fabsf(zm) - tm : 0.f);
      const float a_hi = warp_maxf(cand ? fabsf(zm) + tm : 0.f);
      const float s_lo = a_lo / (float)qmax * (1.f - 4.f * kU);
      const float s_hi = a_hi / (float)qmax * (1.f + 4.f * kU);
      if (s_lo > 2e-8f && same_half(s_lo, s_hi)) {
        // u = z / s against sm, the middle of the range: |s / sm - 1| <= e2
        const float sm = 0.5f * (s_lo + s_hi);
        const float e2 = (s_hi - s_lo) / (s_hi + s_lo) * (1.f + 1e-5f) + 4.f * kU;
        bool bad = false;
        int q2 = q;
        if ((nmask >> lane) & 1u) {
          const float u2 = zm / sm;
          const float au2 = fabsf(u2);
          const float tau2 = (tm / sm + au2 * e2) * (1.f + 2.f * e2) * (1.f + 1e-6f) +
                             4.f * kU * (au2 + 1.f);
          const float hb2 = fminf(floorf(au2) + 0.5f, (float)qmax - 0.5f);
          bad = fabsf(au2 - hb2) <= tau2;
          q2 = (int)fminf(fmaxf(rintf(u2), -(float)qmax), (float)qmax);
        }
        if (!__any_sync(kFull, bad)) {
          q = q2;
          s16 = __float2half_rn(s_lo);
          decided = true;
        }
      }
    }
  }
  if (flagged && !decided) {  // else in double-float, exactly
    const bool cand = valid && (full || az + tz >= a32 - tzm);
    unsigned todo = __ballot_sync(kFull, cand) | nmask;
    const bool redone = (todo >> lane) & 1u;
    // double-float throughout (fp64 throughput is very low here)
    ff2 zmine{0.f, 0.f};
    while (todo) {
      const int f = __ffs(todo) - 1;
      todo &= todo - 1;
      const ff2 z2 =
          dot_ff(c.xs, c.mean, p.Vt + ((int64_t)beta * p.r + first + f) * p.d_in, p.d_in, lane);
      if (lane == f) zmine = z2;
    }
    if (redone && tz > 0.f) {  // the bound in use against the observed error
      const float ratio = fabsf((z - zmine.hi) - zmine.lo) / tz;
      atomicMax(&p.counters[3], (unsigned long long)__float_as_uint(ratio));
    }
    ff2 a2 = cand ? ff_abs(zmine) : ff2{0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const ff2 b2{__shfl_xor_sync(kFull, a2.hi, o), __shfl_xor_sync(kFull, a2.lo, o)};
      if (ff_less(a2, b2)) a2 = b2;
    }
    // s = max(a / qmax, 1e-8), the floor as the double 1e-8 in two floats
    ff2 s2 = ff_div_f(a2, (float)qmax);
    const ff2 floor2{1e-8f, (float)(1e-8 - (double)1e-8f)};  // folded at compile time
    if (ff_less(s2, floor2)) s2 = floor2;
    s16 = ff_to_half(s2);
    if ((nmask >> lane) & 1u)
      q = (int)fminf(fmaxf(ff_rint(ff_div(zmine, s2)), -(float)qmax), (float)qmax);
  }
  if (valid) c.codes[k] = (uint8_t)(q + off);
  if (lane == 0) c.side[gi] = s16;
}

// Codebook: u = (x R) / ||x||; idx = argmin_j |u - c_j| (first on ties); norm fp16.
__device__ void quant_codebook(const Params& p, int beta, const float* vnorm, const RowCtx& c,
                               int chunk, int lane, unsigned* nref, unsigned* nside) {
  const int k = chunk * 32 + lane;
  const bool valid = k < p.r;
  const int L = p.cb_levels;
  const float nrm = c.nrm;
  const bool tiny = nrm < 1e-18f;
  const float z = valid ? c.zs[k] : 0.f;
  const float u = tiny ? 0.f : z / nrm;
  // idx = number of midpoints strictly below u
  int lo_i = 0, hi_i = L - 1;
  while (lo_i < hi_i) {
    const int mid = (lo_i + hi_i) >> 1;
    if (p.mids[mid] < u) lo_i = mid + 1; else hi_i = mid;
  }
  int idx = lo_i;
  float dmin = 3.4e38f;
  if (idx > 0) dmin = fminf(dmin, fabsf(u - p.mids[idx - 1]));
  if (idx < L - 1) dmin = fminf(dmin, fabsf(u - p.mids[idx]));
  const float gam = proj_gamma(p.d_in);
  const float eps_n = 0.5f * gam + 2.f * kU;
  const float cmax = fmaxf(fabsf(p.codebook[0]), fabsf(p.codebook[L - 1]));
  const float tau_u = tiny ? 0.f
                           : (gam * vnorm[valid ? k : 0] * (1.f + 1e-3f) + fabsf(u) * eps_n) *
                                     (1.f + 1e-6f) +
                                 4.f * kU * (fabsf(u) + cmax);
  const bool near = valid && (tiny || dmin <= tau_u);
  const bool norm_unsure =
      chunk == 0 && (tiny || !same_half(nrm * (1.f - eps_n), nrm * (1.f + eps_n)));
  unsigned m = __ballot_sync(kFull, near);
  double n64 = -1.0;
  if (m || norm_unsure) n64 = sqrt(sumsq64(c.xs, p.d_in, lane));
  if (lane == 0 && m) atomicAdd(nref, (unsigned)__popc(m));
  while (m) {
    const int f = __ffs(m) - 1;
    m &= m - 1;
    const int kf = chunk * 32 + f;
    const double z64 =
        dot64(c.xs, c.mean, p.Vt + ((int64_t)beta * p.r + kf) * p.d_in, p.d_in, lane);
    if (lane == f) {
      const double u64 = n64 > 0.0 ? z64 / n64 : 0.0;
      double best = fabs(u64 - (double)p.codebook[0]);
      int bi = 0;
      for (int j = 1; j < L; ++j) {
        const double d = fabs(u64 - (double)p.codebook[j]);
        if (d < best) { best = d; bi = j; }
      }
      idx = bi;
    }
  }
  if (valid) c.codes[k] = (uint8_t)idx;
  if (chunk == 0 && lane == 0) {
    if (norm_unsure) {
      c.side[0] = __double2half(n64);
      atomicAdd(nside, 1u);
    } else {
      c.side[0] = __float2half_rn(nrm);
    }
  }
}

// ---------------------------------------------------------------------------
// Append
// ---------------------------------------------------------------------------

constexpr int kAppTT = 8;
constexpr int kAppThreads = 256;

__global__ void __launch_bounds__(kAppThreads, 4)
append_generic_kernel(Params p, AppendArgs a, ZIn zin) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int slot = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kAppTT;
  const int n = (int)min((int64_t)kAppTT, a.T - t0);
  const int beta = p.basis_of[slot];
  const int d_in = p.d_in, r = p.r;
  const int b = slot / p.Hg, g = slot % p.Hg;

  // With latents from the tensor-core projection the centred rows are not
  // kept (they are recomputed where needed: the same fp32 subtraction), so
  // the block needs half the shared memory and more of them fit on an SM.
  const bool has_xc = zin.z == nullptr;
  float* xs = reinterpret_cast<float*>(smem);      // [TT][d_in]
  float* xc = has_xc ? xs + kAppTT * d_in : nullptr;  // [TT][d_in] fl(x - mean)
  float* zs = xs + (has_xc ? 2 : 1) * kAppTT * d_in;  // [TT][r]
  float* nrm = zs + kAppTT * r;                    // [TT]
  __half* side = reinterpret_cast<__half*>(nrm + kAppTT);  // [TT][n_side]
  const int n_side = p.side_bytes / 2;
  uint8_t* codes = reinterpret_cast<uint8_t*>(side + kAppTT * (n_side > 0 ? n_side : 1));
  __shared__ unsigned s_nref, s_nside;

  const float* mean = p.mean + (int64_t)beta * d_in;
  const float* vnorm = p.vnorm + (int64_t)beta * r;
  if (threadIdx.x == 0) { s_nref = 0; s_nside = 0; }

  // 1. token rows -> fp32 (exact for f32 / f16 / bf16 inputs); 16-bit inputs
  // with 16-byte aligned rows and head slices load 8 values at a time
  const bool vec8 = p.in_dtype != KVC_F32 && p.D % 8 == 0 &&
                    (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
                    ((a.sb | a.sh | a.st) & 7) == 0;
  const float inv_din = 1.f / (float)d_in, inv_D = 1.f / (float)p.D;
  if (vec8) {
    for (int e = threadIdx.x * 8; e < kAppTT * d_in; e += blockDim.x * 8) {
      const int t = small_div(e, inv_din), i = e - t * d_in;
      float v[8];
      if (t < n) {
        const int hh = small_div(i, inv_D);
        const int h = g * p.hpg + hh, dd = i - hh * p.D;
        const uint4 raw = *reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(a.x) + (int64_t)b * a.sb + (int64_t)h * a.sh +
            (t0 + t) * a.st + dd);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint16_t bits = (uint16_t)(w[q >> 1] >> (16 * (q & 1)));
          v[q] = p.in_dtype == KVC_F16 ? __half2float(__ushort_as_half(bits))
                                        : __uint_as_float((uint32_t)bits << 16);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      *reinterpret_cast<float4*>(xs + e) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(xs + e + 4) = make_float4(v[4], v[5], v[6], v[7]);
      if (has_xc) {
#pragma unroll
        for (int q = 0; q < 8; ++q) xc[e + q] = t < n ? v[q] - mean[i + q] : 0.f;
      }
    }
  } else {
    for (int idx = threadIdx.x; idx < kAppTT * d_in; idx += blockDim.x) {
      const int t = idx / d_in, i = idx - t * d_in;
      float v = 0.f;
      if (t < n) {
        const int h = g * p.hpg + i / p.D, dd = i % p.D;
        v = load_in(a.x, p.in_dtype, (int64_t)b * a.sb + (int64_t)h * a.sh + (t0 + t) * a.st + dd);
      }
      xs[idx] = v;
      if (has_xc) xc[idx] = t < n ? v - mean[i] : 0.f;  // the projection's one rounding of x - mean
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  // 2. fp32 norms of the centred rows (the error bound's scale)
  for (int t = warp; t < kAppTT; t += nwarps) {
    float acc = 0.f;
    for (int i = lane; i < d_in; i += 32) {
      const float d = has_xc ? xc[t * d_in + i] : xs[t * d_in + i] - mean[i];
      acc = fmaf(d, d, acc);
    }
    acc = warp_sumf(acc);
    if (lane == 0) nrm[t] = sqrtf(acc);  // the bounds below carry their own margin
  }
  // 3. projection: fp32 fma in blocks of kProjBlk terms, then the block sums;
  // or the latents the tensor-core projection wrote for this tile
  const bool from_z = zin.z != nullptr && zin.ovf[(int64_t)slot * zin.tps + (t0 >> 7)] == 0;
  const QBound qb = from_z ? QBound{zin.gamma, zin.ex, zin.en} : QBound{proj_gamma(d_in), 0.f, 0.f};
  const float* V = p.V + (int64_t)beta * d_in * r;
  if (from_z) {
    const float* zsrc = zin.z + ((int64_t)slot * zin.Tc + t0) * r;
    for (int idx = threadIdx.x; idx < n * r; idx += blockDim.x) zs[idx] = zsrc[idx];
  }
  for (int k = from_z ? r : threadIdx.x; k < r; k += blockDim.x) {
    float acc[kAppTT];
#pragma unroll
    for (int t = 0; t < kAppTT; ++t) acc[t] = 0.f;
    for (int i0 = 0; i0 < d_in; i0 += kProjBlk) {
      float blk[kAppTT];
#pragma unroll
      for (int t = 0; t < kAppTT; ++t) blk[t] = 0.f;
      if (i0 + kProjBlk > d_in || d_in % 4) {  // a partial block or unaligned rows
        for (int i = i0; i < min(i0 + kProjBlk, d_in); ++i) {
          const float v = V[(int64_t)i * r + k];
#pragma unroll
          for (int t = 0; t < kAppTT; ++t)
            blk[t] = fmaf(has_xc ? xc[t * d_in + i] : xs[t * d_in + i] - mean[i], v, blk[t]);
        }
      } else {  // whole block, 4 columns per 128-bit load
#pragma unroll 2
      for (int i = i0; i < i0 + kProjBlk; i += 4) {
        const float v0 = V[(int64_t)i * r + k], v1 = V[(int64_t)(i + 1) * r + k];
        const float v2 = V[(int64_t)(i + 2) * r + k], v3 = V[(int64_t)(i + 3) * r + k];
#pragma unroll
        for (int t = 0; t < kAppTT; ++t) {
          float4 c4;
          if (has_xc) {
            c4 = *reinterpret_cast<const float4*>(xc + t * d_in + i);
          } else {
            const float4 x4 = *reinterpret_cast<const float4*>(xs + t * d_in + i);
            const float4 m4 = *reinterpret_cast<const float4*>(mean + i);
            c4 = make_float4(x4.x - m4.x, x4.y - m4.y, x4.z - m4.z, x4.w - m4.w);
          }
          blk[t] = fmaf(c4.x, v0, blk[t]);
          blk[t] = fmaf(c4.y, v1, blk[t]);
          blk[t] = fmaf(c4.z, v2, blk[t]);
          blk[t] = fmaf(c4.w, v3, blk[t]);
        }
      }
      }
#pragma unroll
      for (int t = 0; t < kAppTT; ++t) acc[t] += blk[t];
    }
#pragma unroll
    for (int t = 0; t < kAppTT; ++t) zs[t * r + k] = acc[t];
  }
  __syncthreads();

  // 4. quantise (+ exact re-decision near boundaries), one warp per item
  if (p.mode == KVC_MODE_GROUP) {
    for (int item = warp; item < n * p.n_groups; item += nwarps) {
      const int t = item / p.n_groups, gi = item - t * p.n_groups;
      RowCtx c{xs + t * d_in, mean, zs + t * r, nrm[t], codes + t * r, side + t * n_side};
      quant_group(p, beta, vnorm, c, gi, lane, &s_nref, &s_nside, qb);
    }
  } else {
    const int nchunk = (r + 31) / 32;
    for (int item = warp; item < n * nchunk; item += nwarps) {
      const int t = item / nchunk, ch = item - t * nchunk;
      RowCtx c{xs + t * d_in, mean, zs + t * r, nrm[t], codes + t * r, side + t * n_side};
      if (p.mode == KVC_MODE_UNIFORM)
        quant_uniform(p, beta, vnorm, c, ch, lane, &s_nref);
      else
        quant_codebook(p, beta, vnorm, c, ch, lane, &s_nref, &s_nside);
    }
  }
  __syncthreads();

  // 5. pack: one thread per output byte
  const int P = p.P[beta];
  const int16_t* order = p.order + (int64_t)beta * r;
  const int32_t* seg = p.seg + (int64_t)beta * kMaxSeg * 4;
  uint8_t* dst = p.store + p.pay_off[slot] + (a.t_base + t0) * P;
  const float inv_P = 1.f / (float)P;
  for (int idx = threadIdx.x; idx < n * P; idx += blockDim.x) {
    const int t = small_div(idx, inv_P), j = idx - t * P;
    int s = 0;
    while (s + 1 < kMaxSeg && seg[(s + 1) * 4 + 3] > 0 && seg[(s + 1) * 4 + 0] <= j) ++s;
    const int start = seg[s * 4 + 0], w = seg[s * 4 + 1], m0 = seg[s * 4 + 2], cntm = seg[s * 4 + 3];
    const int q0 = 8 * (j - start);
    const float inv_w = 1.f / (float)w;  // w in {1, 2, 3, 4, 8}
    int mlo = small_div(q0, inv_w), mhi = small_div(q0 + 7, inv_w);
    if (mhi > cntm - 1) mhi = cntm - 1;
    unsigned v = 0;
    for (int mm = mlo; mm <= mhi; ++mm) {
      const unsigned code = codes[t * r + order[m0 + mm]];
      const int sh = mm * w - q0;
      v |= sh >= 0 ? (code << sh) : (code >> (-sh));
    }
    dst[idx] = (uint8_t)(v & 0xffu);
  }
  if (n_side > 0) {
    __half* sdst = reinterpret_cast<__half*>(p.store + p.side_off[slot]) + (a.t_base + t0) * n_side;
    for (int idx = threadIdx.x; idx < n * n_side; idx += blockDim.x) sdst[idx] = side[idx];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_nref) atomicAdd(&p.counters[0], (unsigned long long)s_nref);
    if (s_nside) atomicAdd(&p.counters[1], (unsigned long long)s_nside);
    if (blockIdx.y == 0) atomicAdd(&p.counters[2], (unsigned long long)n);
  }
}

// ---------------------------------------------------------------------------
// Fetch
// ---------------------------------------------------------------------------

constexpr int kFetTT = 16;
constexpr int kFetThreads = 256;

__global__ void __launch_bounds__(kFetThreads) fetch_generic_kernel(Params p, FetchArgs f) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int slot = blockIdx.y;
  const int64_t t0 = (int64_t)blockIdx.x * kFetTT;
  const int n = (int)min((int64_t)kFetTT, f.S - t0);
  const int beta = p.basis_of[slot];
  const int d_in = p.d_in, r = p.r;
  const int b = slot / p.Hg, g = slot % p.Hg;
  float* zh = reinterpret_cast<float*>(smem);  // [TT][r]

  for (int idx = threadIdx.x; idx < kFetTT * r; idx += blockDim.x) zh[idx] = 0.f;
  __syncthreads();

  const int P = p.P[beta];
  const int nk = p.n_kept[beta];
  const int16_t* order = p.order + (int64_t)beta * r;
  const int32_t* seg = p.seg + (int64_t)beta * kMaxSeg * 4;
  const uint8_t* src = p.store + p.pay_off[slot] + t0 * P;
  const int n_side = p.side_bytes / 2;
  const __half* sside =
      reinterpret_cast<const __half*>(p.store + p.side_off[slot]) + t0 * (int64_t)n_side;

  for (int idx = threadIdx.x; idx < n * nk; idx += blockDim.x) {
    const int t = idx / nk, m = idx - t * nk;
    int s = 0;
    while (s + 1 < kMaxSeg && seg[(s + 1) * 4 + 3] > 0 && seg[(s + 1) * 4 + 2] <= m) ++s;
    const int start = seg[s * 4 + 0], w = seg[s * 4 + 1], m0 = seg[s * 4 + 2];
    const int bit = 8 * start + (m - m0) * w;
    const uint8_t* row = src + (int64_t)t * P;
    unsigned v = row[bit >> 3];
    if ((bit & 7) + w > 8) v |= (unsigned)row[(bit >> 3) + 1] << 8;
    const int code = (int)((v >> (bit & 7)) & ((1u << w) - 1u));
    const int k = order[m];
    float zv;
    if (p.mode == KVC_MODE_UNIFORM) {
      zv = fmaf((float)code, p.step[beta * r + k], p.lo[beta * r + k]);
    } else if (p.mode == KVC_MODE_GROUP) {
      int gi = 0;
      while (gi + 1 < p.n_groups && p.groups[(gi + 1) * 3] <= k) ++gi;
      zv = (float)(code - (1 << (w - 1))) * __half2float(sside[(int64_t)t * n_side + gi]);
    } else {
      zv = __half2float(sside[t]) * p.codebook[code];
    }
    zh[t * r + k] = zv;
  }
  __syncthreads();

  const float* Vt = p.Vt + (int64_t)beta * r * d_in;
  const float* mean = p.mean + (int64_t)beta * d_in;
  for (int i = threadIdx.x; i < d_in; i += blockDim.x) {
    float acc[kFetTT];
    const float m = mean[i];
#pragma unroll
    for (int t = 0; t < kFetTT; ++t) acc[t] = m;
    for (int k = 0; k < r; ++k) {
      const float v = Vt[(int64_t)k * d_in + i];
#pragma unroll
      for (int t = 0; t < kFetTT; ++t) acc[t] = fmaf(zh[t * r + k], v, acc[t]);
    }
    const int h = g * p.hpg + i / p.D, dd = i % p.D;
    const int64_t base = (((int64_t)b * p.H + h) * f.ld_s + t0) * p.D + dd;
    for (int t = 0; t < n; ++t) store_out(f.out, p.out_dtype, base + (int64_t)t * p.D, acc[t]);
  }
}

// ---------------------------------------------------------------------------
// int8 values: one warp per token
// ---------------------------------------------------------------------------

constexpr int kI8Warps = 8;

__global__ void __launch_bounds__(kI8Warps * 32) append_int8_kernel(Params p, AppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t tok = (int64_t)blockIdx.x * kI8Warps + (threadIdx.x >> 5);  // over n_slots * T
  if (tok >= (int64_t)p.n_slots * a.T) return;
  const int slot = (int)(tok / a.T);
  const int64_t t = tok - (int64_t)slot * a.T;
  const int b = slot / p.H, h = slot % p.H;
  const int64_t xoff = (int64_t)b * a.sb + (int64_t)h * a.sh + t * a.st;
  float amax = 0.f;
  for (int i = lane; i < p.D; i += 32) amax = fmaxf(amax, fabsf(load_in(a.x, p.in_dtype, xoff + i)));
  amax = warp_maxf(amax);
  // exactly the double-precision scale of the reference arithmetic
  const double s64 = fmax((double)amax / 127.0, 1e-8);
  const float inv = (float)(1.0 / s64);
  int8_t* dst = reinterpret_cast<int8_t*>(p.store + p.pay_off[slot]) + (a.t_base + t) * p.D;
  unsigned nref = 0;
  for (int i = lane; i < p.D; i += 32) {
    const float v = load_in(a.x, p.in_dtype, xoff + i);
    const float u = v * inv;  // |u - v / s| <= 3 * 2^-24 * 127.5 < 2.5e-5
    const float au = fabsf(u);
    float q;
    if (fabsf(au - floorf(au) - 0.5f) < 1e-4f) {
      q = (float)rint((double)v / s64);
      ++nref;
    } else {
      q = rintf(u);
    }
    dst[i] = (int8_t)fminf(fmaxf(q, -127.f), 127.f);
  }
  if (lane == 0) {
    reinterpret_cast<__half*>(p.store + p.side_off[slot])[a.t_base + t] = __double2half(s64);
  }
  nref = __reduce_add_sync(kFull, nref);
  if (lane == 0 && nref) atomicAdd(&p.counters[0], (unsigned long long)nref);
  if (lane == 0 && slot == 0) atomicAdd(&p.counters[2], 1ull);
}

__global__ void __launch_bounds__(kI8Warps * 32) fetch_int8_kernel(Params p, FetchArgs f) {
  const int lane = threadIdx.x & 31;
  const int64_t tok = (int64_t)blockIdx.x * kI8Warps + (threadIdx.x >> 5);
  if (tok >= (int64_t)p.n_slots * f.S) return;
  const int slot = (int)(tok / f.S);
  const int64_t t = tok - (int64_t)slot * f.S;
  const int b = slot / p.H, h = slot % p.H;
  const int8_t* src = reinterpret_cast<const int8_t*>(p.store + p.pay_off[slot]) + t * p.D;
  const float s = __half2float(reinterpret_cast<const __half*>(p.store + p.side_off[slot])[t]);
  const int64_t base = (((int64_t)b * p.H + h) * f.ld_s + t) * p.D;
  for (int i = lane; i < p.D; i += 32) store_out(f.out, p.out_dtype, base + i, (float)src[i] * s);
}

// ---------------------------------------------------------------------------
// int8 values, vectorised: one thread per 8 values, TPR = D / 8 threads per row
// (8, 16 or 32, always inside one warp).  Exact without a double division per
// row: the fast path is u = v * fl32(127 / a), within 1.5e-5 of v / s (s the
// double-precision scale), so only values within 1e-4 of a half-integer, rows
// with a <= 2e-6 (zero rows and the 1e-8 scale floor) and scales near an fp16
// rounding boundary are decided in double precision.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void load8(const void* x, int dt, int64_t off, float (&v)[8]) {
  if (dt == KVC_F32) {
    const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
    const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 q = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t lo = (uint16_t)(w[i] & 0xffffu), hi = (uint16_t)(w[i] >> 16);
      if (dt == KVC_F16) {
        v[2 * i] = __half2float(__ushort_as_half(lo));
        v[2 * i + 1] = __half2float(__ushort_as_half(hi));
      } else {
        v[2 * i] = __bfloat162float(__ushort_as_bfloat16(lo));
        v[2 * i + 1] = __bfloat162float(__ushort_as_bfloat16(hi));
      }
    }
  }
}

// One token row, NV = 32 values per thread: its absmax over the TPR threads,
// the int8 codes q = rint(v / s), s = max(a / 127, 1e-8), and fp16(s).
// Returns the number of codes re-decided.  The fast u = v fl(127 / a) is
// within 1.5e-5 of 127 v / a (two roundings, |u| <= 127, so no clamp is
// needed); a code within 3e-5 of a half is decided exactly: for 16-bit inputs
// 254 |v| and (2k + 1) a are exact in fp32 (at most 19 significant bits
// each), so the sign of their difference decides it; an exact tie, fp32
// inputs, a < 2e-6 and a >= 1e30 take the float64 path.
constexpr int kI8NV = 32;
template <int TPR, bool IL = false>
__device__ __forceinline__ unsigned append_int8_vals(const Params& p, const AppendArgs& a, int slot,
                                                     int64_t t, int j, bool valid,
                                                     float (&v)[kI8NV]);

template <int TPR>
__device__ __forceinline__ unsigned append_int8_row(const Params& p, const AppendArgs& a, int slot,
                                                    int64_t t, int j) {
  const bool valid = t < a.T;
  float v[kI8NV];
#pragma unroll
  for (int i = 0; i < kI8NV; ++i) v[i] = 0.f;
  if (valid) {
    const int b = slot / p.H, h = slot - b * p.H;
    const int64_t off = (int64_t)b * a.sb + (int64_t)h * a.sh + t * a.st + kI8NV * j;
#pragma unroll
    for (int c = 0; c < kI8NV / 8; ++c)
      load8(a.x, p.in_dtype, off + 8 * c, *reinterpret_cast<float(*)[8]>(&v[8 * c]));
  }
  return append_int8_vals<TPR>(p, a, slot, t, j, valid, v);
}

// IL (interleaved): the thread's values are the row's 8-value groups
// j, j + TPR, j + 2 TPR, j + 3 TPR instead of 32 consecutive values.
template <int TPR, bool IL>
__device__ __forceinline__ unsigned append_int8_vals(const Params& p, const AppendArgs& a, int slot,
                                                     int64_t t, int j, bool valid,
                                                     float (&v)[kI8NV]) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < kI8NV; ++i) am = fmaxf(am, fabsf(v[i]));
#pragma unroll
  for (int o = TPR / 2; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(kFull, am, o));
  unsigned nref = 0;
  if (valid) {
    const bool slow = !(am > 2e-6f);
    const bool exact16 = p.in_dtype != KVC_F32 && am < 1e30f;  // no overflow in 254 v
    const float inv = slow ? 0.f : 127.f / am;
    // Rounding by adding 1.5 2^23 (half to even for |u| < 2^22) leaves the
    // code in the low byte of the sum, two's complement, so four codes are
    // packed by byte permutes: no float-to-int conversions on this path.
    // Two values at a time with the packed fp32 fma (each lane rounds as the
    // scalar one): t = v inv + M, -q = M - t (exact: t lies within a factor
    // 2 of M), and the remainder v inv - q for the near test.
    constexpr float kMagic = 12582912.f;
    const float2 inv2 = make_float2(inv, inv), m2 = make_float2(kMagic, kMagic),
                 neg2 = make_float2(-1.f, -1.f);
    uint32_t packed[kI8NV / 4];
    bool any_near = slow;  // a value within 3e-5 of a half, a NaN, or a tiny row
#pragma unroll
    for (int i = 0; i < kI8NV; i += 4) {
      uint32_t tb[4];
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        // q = rint(v inv) of the exact product (within 127 2^-24 of 127 v / a)
        const float2 vv = make_float2(v[i + e], v[i + e + 1]);
        const float2 t = __ffma2_rn(vv, inv2, m2);
        const float2 nq = __ffma2_rn(t, neg2, m2);
        const float2 rm = __ffma2_rn(vv, inv2, nq);
        any_near |= !(fabsf(rm.x) <= 0.5f - 3e-5f) || !(fabsf(rm.y) <= 0.5f - 3e-5f);
        tb[e] = __float_as_uint(t.x);
        tb[e + 1] = __float_as_uint(t.y);
      }
      packed[i >> 2] =
          __byte_perm(__byte_perm(tb[0], tb[1], 0x0040), __byte_perm(tb[2], tb[3], 0x0040), 0x5410);
    }
    // the fast codes go out first; the rare re-decisions below overwrite
    // single bytes of them (same thread, so in program order), which keeps
    // the packed words out of the rare path's registers
    uint8_t* dst = p.store + p.pay_off[slot] + (a.t_base + t) * p.D + (IL ? 8 * j : kI8NV * j);
    if (IL) {
#pragma unroll
      for (int g = 0; g < kI8NV / 8; ++g)
        reinterpret_cast<uint2*>(dst + 8 * TPR * g)[0] = make_uint2(packed[2 * g], packed[2 * g + 1]);
    } else {
#pragma unroll
      for (int w = 0; w < kI8NV / 16; ++w)
        reinterpret_cast<uint4*>(dst)[w] =
            make_uint4(packed[4 * w], packed[4 * w + 1], packed[4 * w + 2], packed[4 * w + 3]);
    }
    uint32_t flag = 0;
    if (any_near) {
#pragma unroll
      for (int i = 0; i < kI8NV; ++i) {
        const float u = v[i] * inv;
        flag |= (uint32_t)!(fabsf(u - rintf(u)) <= 0.5f - 3e-5f) << i;
      }
      if (slow) flag = 0xffffffffu;
    }
    if (flag) {  // rare: re-decide those exactly, then patch their bytes
      double s64 = fmax((double)am / 127.0, 1e-8);
      for (uint32_t f = flag; f; f &= f - 1) {
        const int i = __ffs(f) - 1;
        float vi = 0.f;
#pragma unroll
        for (int e = 0; e < kI8NV; ++e) vi = e == i ? v[e] : vi;  // no local-memory indexing
        // the byte of value i: group i / 8 of the thread's groups when interleaved
        uint8_t* bp = dst + (IL ? 8 * TPR * (i >> 3) + (i & 7) : i);
        const float u = vi * inv;
        if (!slow && u != u) {  // a NaN (or an infinity times 0): code 0
          *bp = 0;
          continue;
        }
        ++nref;
        const float k = floorf(fabsf(u));
        const float d = exact16 && !slow ? 254.f * fabsf(vi) - (2.f * k + 1.f) * am : 0.f;
        float q;
        if (d != 0.f) {
          q = copysignf(d > 0.f ? k + 1.f : k, vi);
        } else {  // an exact tie, fp32 input or a tiny row: as float64 decides it
          q = (float)fmin(fmax(rint((double)vi / s64), -127.0), 127.0);
        }
        *bp = (uint8_t)(__float2int_rn(q) & 0xff);
      }
    }
    if (j == 0) {
      const float s32 = am / 127.f;
      __half s16;
      if (!slow && same_half(s32 * (1.f - 4.f * kU), s32 * (1.f + 4.f * kU))) {
        s16 = __float2half_rn(s32);
      } else {
        s16 = __double2half(fmax((double)am / 127.0, 1e-8));
      }
      reinterpret_cast<__half*>(p.store + p.side_off[slot])[a.t_base + t] = s16;
    }
  }
  return nref;
}

// Grid: x over blocks of 256 / TPR tokens, y over slots (strided when there
// are more than 65535), so no thread divides by a runtime value.  Counters:
// a warp adds its re-decisions (rarely any); the tokens appended are added
// once per block of the first slot.
template <int TPR>
__global__ void __launch_bounds__(256) append_int8_vec(Params p, AppendArgs a) {
  const int j = (int)(threadIdx.x % TPR);
  const int64_t t = (int64_t)blockIdx.x * (256 / TPR) + threadIdx.x / TPR;
  unsigned nref = 0;
  for (int slot = blockIdx.y; slot < p.n_slots; slot += gridDim.y)
    nref += append_int8_row<TPR>(p, a, slot, t, j);
  nref = __reduce_add_sync(kFull, nref);
  if ((threadIdx.x & 31) == 0 && nref) atomicAdd(&p.counters[0], (unsigned long long)nref);
  if (threadIdx.x == 0 && blockIdx.y == 0) {
    const int64_t rows = min((int64_t)(256 / TPR), a.T - (int64_t)blockIdx.x * (256 / TPR));
    if (rows > 0) atomicAdd(&p.counters[2], (unsigned long long)rows);
  }
}

// Pipelined int8 append: a persistent grid walks the rows (slot-major, 256 /
// TPR rows per block step); each thread copies its own 32 values of the rows
// kI8Stages - 1 steps ahead into shared memory with cp.async (16 bytes each,
// one commit group per step) and waits for its oldest group with
// cp.async.wait_group, so HBM sees kI8Stages - 1 rows per thread in flight.
// A thread reads back only what it copied: no barrier is needed.  ESZ: the
// input element bytes (2 or 4).  Two stages (one row ahead) measured faster
// than three or four: three blocks of 256 threads per SM already keep far
// more bytes in flight than HBM needs, and fewer blocks per SM with deeper
// stages were slower still.
constexpr int kI8Stages = 2;
template <int TPR, int ESZ, bool F16>
__global__ void __launch_bounds__(256, 3) append_int8_pipe(Params p, AppendArgs a) {
  constexpr int Q = kI8NV * ESZ / 16;  // 16-byte pieces of a thread's values
  constexpr bool IL = ESZ == 2;
  constexpr int RPB = 256 / TPR;       // rows per block step
  extern __shared__ uint4 stage_buf[];  // [kI8Stages][Q][256]
  const int tid = threadIdx.x, j = tid % TPR;
  const int64_t total = (int64_t)p.n_slots * a.T;
  const int64_t step = (int64_t)gridDim.x * RPB;
  const int64_t r0 = (int64_t)blockIdx.x * RPB + tid / TPR;
  // (slot, token) of a row, advanced by one step without dividing: a step is
  // sq slots and st_rem tokens
  const int64_t sq = step / a.T, st_rem = step - sq * a.T;
  struct Pos {
    int64_t slot, t;
  };
  auto advance = [&](Pos q) {
    q.slot += sq;
    q.t += st_rem;
    if (q.t >= a.T) {
      q.t -= a.T;
      ++q.slot;
    }
    return q;
  };
  Pos pi{r0 / a.T, 0}, pp;
  pi.t = r0 - pi.slot * a.T;
  pp = pi;
  auto issue = [&](const Pos q, int st) {
    if (q.slot < p.n_slots) {
      const int slot = (int)q.slot;
      const int b = slot / p.H, h = slot - b * p.H;
      // 16-bit inputs: piece qq is the row's 16-byte piece TPR qq + j, so
      // each copy instruction of a warp reads whole 32-byte sectors
      const char* src = static_cast<const char*>(a.x) +
                        ((int64_t)b * a.sb + (int64_t)h * a.sh + q.t * a.st +
                         (IL ? 8 * j : kI8NV * j)) * ESZ;
#pragma unroll
      for (int qq = 0; qq < Q; ++qq) {
        const uint32_t dst =
            (uint32_t)__cvta_generic_to_shared(&stage_buf[((size_t)st * Q + qq) * 256 + tid]);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst),
                     "l"(src + 16 * (IL ? TPR * qq : qq))
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
#pragma unroll
  for (int s0 = 0; s0 < kI8Stages - 1; ++s0) {
    issue(pi, s0);
    pi = advance(pi);
  }
  unsigned nref = 0, rows0 = 0;
  int64_t rb = (int64_t)blockIdx.x * RPB;  // the block's first row of the step
  for (int k = 0; rb < total; ++k, rb += step) {
    issue(pi, (k + kI8Stages - 1) % kI8Stages);
    pi = advance(pi);
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kI8Stages - 1) : "memory");
    const int st = k % kI8Stages;
    float v[kI8NV];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      const uint4 w = stage_buf[((size_t)st * Q + q) * 256 + tid];
      if (ESZ == 4) {
        v[4 * q] = __uint_as_float(w.x);
        v[4 * q + 1] = __uint_as_float(w.y);
        v[4 * q + 2] = __uint_as_float(w.z);
        v[4 * q + 3] = __uint_as_float(w.w);
      } else {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint16_t lo = (uint16_t)(ww[e] & 0xffffu), hi = (uint16_t)(ww[e] >> 16);
          if (F16) {
            v[8 * q + 2 * e] = __half2float(__ushort_as_half(lo));
            v[8 * q + 2 * e + 1] = __half2float(__ushort_as_half(hi));
          } else {
            v[8 * q + 2 * e] = __uint_as_float(ww[e] << 16);
            v[8 * q + 2 * e + 1] = __uint_as_float(ww[e] & 0xffff0000u);
          }
        }
      }
    }
    const bool valid = pp.slot < p.n_slots;
    const int slot = valid ? (int)pp.slot : 0;
    nref += append_int8_vals<TPR, IL>(p, a, slot, valid ? pp.t : a.T, j, valid, v);
    rows0 += (valid && slot == 0 && j == 0) ? 1u : 0u;
    pp = advance(pp);
  }
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  nref = __reduce_add_sync(kFull, nref);
  rows0 = __reduce_add_sync(kFull, rows0);
  if ((tid & 31) == 0 && nref) atomicAdd(&p.counters[0], (unsigned long long)nref);
  if ((tid & 31) == 0 && rows0) atomicAdd(&p.counters[2], (unsigned long long)rows0);
}

// Grid: x over blocks of R (256 / TPR) tokens, y over slots (strided when
// there are more than 65535).  A thread takes R token rows 256 / TPR apart
// (a warp's rows stay contiguous), with all R loads issued before any decode.
template <int TPR, int R>
__global__ void __launch_bounds__(256) fetch_int8_vec(Params p, FetchArgs f) {
  constexpr int RPB = 256 / TPR;  // rows per block step
  const int j = (int)(threadIdx.x % TPR);
  const int64_t t0 = (int64_t)blockIdx.x * RPB * R + threadIdx.x / TPR;
  if (t0 >= f.S) return;
  // Code byte b + 128 placed in the low mantissa bits of fp16 1024 gives
  // 1024 + 128 + b exactly; subtracting 1152 leaves b as an fp16 integer.  No
  // int-to-float conversions.  b s is exact in fp32 (8 by 11 significant
  // bits), so one fp16 product rounds exactly as fp16(float(b) s) does.
  const __half2 bias = __float2half2_rn(-1152.f);
  for (int slot = blockIdx.y; slot < p.n_slots; slot += gridDim.y) {
    const int b = slot / p.H, h = slot - b * p.H;
    const uint8_t* pay = p.store + p.pay_off[slot];
    const __half* side = reinterpret_cast<const __half*>(p.store + p.side_off[slot]);
    uint2 q[R];
    __half sh[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t t = t0 + (int64_t)r * RPB;
      if (t < f.S) {
        q[r] = *reinterpret_cast<const uint2*>(pay + t * p.D + 8 * j);
        sh[r] = side[t];
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int64_t t = t0 + (int64_t)r * RPB;
      if (t >= f.S) break;
      const uint32_t w[2] = {q[r].x ^ 0x80808080u, q[r].y ^ 0x80808080u};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t hb = __byte_perm(w[i >> 1], 0x64646464u, (i & 1) ? 0x4342 : 0x4140);
        const __half2 b2 = __hadd2(*reinterpret_cast<const __half2*>(&hb), bias);
        if (p.out_dtype == KVC_F16) {
          const __half2 hv = __hmul2(b2, __half2half2(sh[r]));
          o[i] = *reinterpret_cast<const uint32_t*>(&hv);
        } else {
          const float2 fv = __half22float2(b2);
          const float s = __half2float(sh[r]);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(fv.x * s, fv.y * s);
          o[i] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
      uint16_t* out =
          static_cast<uint16_t*>(f.out) + (((int64_t)b * p.H + h) * f.ld_s + t) * p.D + 8 * j;
      *reinterpret_cast<uint4*>(out) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_append_generic(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk,
                                  const ZIn* zin) {
  if (a.T <= 0) return cudaSuccess;
  const int n_side = p.side_bytes / 2;
  const size_t smem = sizeof(float) * ((zin ? 1 : 2) * kAppTT * p.d_in + kAppTT * p.r + kAppTT) +
                      sizeof(__half) * kAppTT * (n_side > 0 ? n_side : 1) + kAppTT * p.r + 16;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(append_generic_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)((a.T + kAppTT - 1) / kAppTT), (unsigned)p.n_slots);
  append_generic_kernel<<<grid, kAppThreads, smem, s>>>(p, a, zin ? *zin : ZIn{});
  ++*nk;
  return cudaGetLastError();
}

cudaError_t launch_fetch_generic(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk) {
  if (f.S <= 0) return cudaSuccess;
  const size_t smem = sizeof(float) * kFetTT * p.r;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fetch_generic_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)((f.S + kFetTT - 1) / kFetTT), (unsigned)p.n_slots);
  fetch_generic_kernel<<<grid, kFetThreads, smem, s>>>(p, f);
  ++*nk;
  return cudaGetLastError();
}

cudaError_t launch_append_int8(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk) {
  const int64_t toks = (int64_t)p.n_slots * a.T;
  if (toks <= 0) return cudaSuccess;
  const int esz = p.in_dtype == KVC_F32 ? 4 : 2;
  const bool vec = (p.D == 64 || p.D == 128 || p.D == 256) &&
                   reinterpret_cast<uintptr_t>(a.x) % 16 == 0 && (a.st * esz) % 16 == 0 &&
                   (a.sh * esz) % 16 == 0 && (a.sb * esz) % 16 == 0;
  if (vec && toks >= 4096) {
    // persistent, pipelined: three blocks per SM, or fewer for a small call
    const int tpr = p.D / kI8NV;
    const int rpb = 256 / tpr;
    const int64_t steps = (toks + rpb - 1) / rpb;
    const unsigned grid = (unsigned)std::min<int64_t>(steps, 3 * (int64_t)sm_count());
    const size_t smem = (size_t)kI8Stages * kI8NV * esz * 256;
    cudaError_t e = cudaSuccess;
#define KVC_I8_PIPE(T, E, H)                                                                 \
  e = cudaFuncSetAttribute(append_int8_pipe<T, E, H>,                                          \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);            \
  if (e == cudaSuccess) append_int8_pipe<T, E, H><<<grid, 256, smem, s>>>(p, a);
    if (esz == 2 && p.in_dtype == KVC_F16) {
      if (tpr == 2) { KVC_I8_PIPE(2, 2, true) } else if (tpr == 4) { KVC_I8_PIPE(4, 2, true) } else { KVC_I8_PIPE(8, 2, true) }
    } else if (esz == 2) {
      if (tpr == 2) { KVC_I8_PIPE(2, 2, false) } else if (tpr == 4) { KVC_I8_PIPE(4, 2, false) } else { KVC_I8_PIPE(8, 2, false) }
    } else {
      if (tpr == 2) { KVC_I8_PIPE(2, 4, false) } else if (tpr == 4) { KVC_I8_PIPE(4, 4, false) } else { KVC_I8_PIPE(8, 4, false) }
    }
#undef KVC_I8_PIPE
    if (e != cudaSuccess) return e;
  } else if (vec) {
    const int tpr = p.D / kI8NV;  // 32 values per thread
    const dim3 grid((unsigned)((a.T * tpr + 255) / 256), (unsigned)std::min(p.n_slots, 65535));
    if (tpr == 2) append_int8_vec<2><<<grid, 256, 0, s>>>(p, a);
    else if (tpr == 4) append_int8_vec<4><<<grid, 256, 0, s>>>(p, a);
    else append_int8_vec<8><<<grid, 256, 0, s>>>(p, a);
  } else {
    append_int8_kernel<<<(unsigned)((toks + kI8Warps - 1) / kI8Warps), kI8Warps * 32, 0, s>>>(p, a);
  }
  ++*nk;
  return cudaGetLastError();
}

cudaError_t launch_fetch_int8(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk) {
  const int64_t toks = (int64_t)p.n_slots * f.S;
  if (toks <= 0) return cudaSuccess;
  const bool vec = (p.D == 64 || p.D == 128 || p.D == 256) &&
                   reinterpret_cast<uintptr_t>(f.out) % 16 == 0;
  if (vec) {
    constexpr int R = 4;  // token rows per thread
    const int tpr = p.D / 8;
    const int64_t rows_per_block = (int64_t)(256 / tpr) * R;
    const dim3 grid((unsigned)((f.S + rows_per_block - 1) / rows_per_block),
                    (unsigned)std::min(p.n_slots, 65535));
    if (tpr == 8) fetch_int8_vec<8, R><<<grid, 256, 0, s>>>(p, f);
    else if (tpr == 16) fetch_int8_vec<16, R><<<grid, 256, 0, s>>>(p, f);
    else fetch_int8_vec<32, R><<<grid, 256, 0, s>>>(p, f);
  } else {
    fetch_int8_kernel<<<(unsigned)((toks + kI8Warps - 1) / kI8Warps), kI8Warps * 32, 0, s>>>(p, f);
  }
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
