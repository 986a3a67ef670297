// Exact re-decision of quantiser outputs near a rounding boundary, shared by
// the tensor-core append kernels (sm_103a).
//
// The tensor-core projection z32 carries an accumulation error bounded by
//   |z32 - z| <= gamma * ||x|| * ||V_k|| + 2^-21 (|z| + |mean . V_k|)
// (gamma from a model of aligned, truncated fp32 accumulation; see the host
// plan).  Codes whose fast-path value lies within that bound (through the
// quantiser's own roundings) of a rounding boundary are queued and re-decided
// here by one warp with a compensated fp32 dot product (error ~1e-13
// relative) finished in double precision.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvc_ff.cuh"
#include "kvc_internal.h"

namespace kvc {
namespace {

__device__ __forceinline__ void set_err(int* err, int code) { atomicCAS(err, 0, code); }

// True when every value in [lo, hi] rounds to the same fp16.
__device__ __forceinline__ bool same_half(float lo, float hi) {
  return __half_as_ushort(__float2half_rn(lo)) == __half_as_ushort(__float2half_rn(hi));
}

constexpr int kQueue = 512;
constexpr uint32_t kNormEntry = 0xFFFFu;

struct AppendTc {
  const uint16_t* B;    // [nb][3][rpad][D]
  const double* c64;    // [nb][r]
  int rpad, cols;
  float inv_scale, gamma;
};


// x_t . w with x_t a row of the swizzled x tile (w == nullptr: x_t . x_t),
// compensated fp32 (TwoProd / TwoSum) finished in double.  WARP: the 32 lanes
// split the row and the result is on every lane; else one thread does it all.
template <bool BF16, bool WARP>
__device__ ff2 dot2_ff(const unsigned char* xs, int t, int D, const float* w, int lane) {
  float S = 0.f, C = 0.f;
  auto term = [&](int i, float wv, bool self) {
    const unsigned char* src =
        xs + (i >> 6) * 16384 + t * 128 + ((((i & 63) >> 3) ^ (t & 7)) << 4) + (i & 7) * 2;
    const uint16_t raw = *reinterpret_cast<const uint16_t*>(src);
    const float xv = BF16 ? __bfloat162float(__ushort_as_bfloat16(raw))
                          : __half2float(__ushort_as_half(raw));
    const float wx = self ? xv : wv;
    const float pr = xv * wx;
    const float pe = fmaf(xv, wx, -pr);
    float s, e;
    two_sum(S, pr, s, e);
    S = s;
    C += pe + e;
  };
  if (WARP) {
    // the lane's (at most 8) entries of w are loaded before the arithmetic:
    // one memory latency instead of one per entry
    float wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = lane + 32 * j;
      wv[j] = (w && i < D) ? w[i] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = lane + 32 * j;
      if (i < D) term(i, wv[j], w == nullptr);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float So = __shfl_xor_sync(0xffffffffu, S, o);
      const float Co = __shfl_xor_sync(0xffffffffu, C, o);
      float s, e;
      two_sum(S, So, s, e);
      S = s;
      C = C + Co + e;
    }
  } else {
    for (int i = 0; i < D; ++i) term(i, w ? w[i] : 0.f, w == nullptr);
  }
  float s, e;
  two_sum(S, C, s, e);
  return ff2{s, e};
}

// The same dots by a group of GL lanes (GL divides 32; the shuffles stay
// inside the group): x_t . x_t and, when w is not null, x_t . w in one pass
// over the row.  Every lane of the warp must call it; the results are on every
// lane of the group.
template <bool BF16, int GL>
__device__ __forceinline__ void dot2_ff_group(const unsigned char* xs, int t, int D,
                                              const float* w, int sub, ff2& xx, ff2& xw) {
  float S1 = 0.f, C1 = 0.f, S2 = 0.f, C2 = 0.f;
  for (int i = sub; i < D; i += GL) {
    const unsigned char* src =
        xs + (i >> 6) * 16384 + t * 128 + ((((i & 63) >> 3) ^ (t & 7)) << 4) + (i & 7) * 2;
    const uint16_t raw = *reinterpret_cast<const uint16_t*>(src);
    const float xv = BF16 ? __bfloat162float(__ushort_as_bfloat16(raw))
                          : __half2float(__ushort_as_half(raw));
    float s, e;
    const float p1 = xv * xv, e1 = fmaf(xv, xv, -p1);
    two_sum(S1, p1, s, e);
    S1 = s;
    C1 += e1 + e;
    if (w) {
      const float wv = w[i];
      const float p2 = xv * wv, e2 = fmaf(xv, wv, -p2);
      two_sum(S2, p2, s, e);
      S2 = s;
      C2 += e2 + e;
    }
  }
#pragma unroll
  for (int o = GL / 2; o > 0; o >>= 1) {
    float s, e;
    const float So1 = __shfl_xor_sync(0xffffffffu, S1, o), Co1 = __shfl_xor_sync(0xffffffffu, C1, o);
    two_sum(S1, So1, s, e);
    S1 = s;
    C1 = C1 + Co1 + e;
    const float So2 = __shfl_xor_sync(0xffffffffu, S2, o), Co2 = __shfl_xor_sync(0xffffffffu, C2, o);
    two_sum(S2, So2, s, e);
    S2 = s;
    C2 = C2 + Co2 + e;
  }
  float s, e;
  two_sum(S1, C1, s, e);
  xx = ff2{s, e};
  two_sum(S2, C2, s, e);
  xw = ff2{s, e};
}

template <bool BF16, bool WARP>
__device__ double dot2_row(const unsigned char* xs, int t, int D, const float* w, int lane) {
  const ff2 v = dot2_ff<BF16, WARP>(xs, t, D, w, lane);
  return (double)v.hi + (double)v.lo;
}

// Decide code k of token tt exactly (or, k == kNormEntry, the fp16 norm of a
// codebook token).  Lane 0 (or the lone thread) writes the result.
// The largest |u_fast - u_exact| / bound seen (float bits; all non-negative)
// is kept in counters[3]: evidence of how much margin the bound carries.
__device__ __forceinline__ void note_ratio(const Params& p, double uf, double u, float tau) {
  if (tau > 0.f) {
    const float ratio = (float)(fabs(uf - u) / (double)tau);
    atomicMax(&p.counters[3], (unsigned long long)__float_as_uint(ratio));
  }
}

template <int MODE, bool BF16, bool WARP>
__device__ void refine_entry(const Params& p, const AppendTc& t, int beta, const unsigned char* xs,
                             unsigned char* codes_s, __half* side_s, unsigned* nside, int tt, int k,
                             int lane, float uf = 0.f, float tau = 0.f) {
  const int D = p.D, r = p.r;
  const float* Vt = p.Vt + (size_t)beta * r * D;
  if (MODE == KVC_MODE_UNIFORM) {
    const double z64 = dot2_row<BF16, WARP>(xs, tt, D, Vt + (size_t)k * D, lane) -
                       t.c64[(size_t)beta * r + k];
    if (lane == 0) {
      const int qmax = (1 << p.bits[(size_t)beta * r + k]) - 1;
      const double u64 =
          (z64 - (double)p.lo[(size_t)beta * r + k]) / (double)p.step[(size_t)beta * r + k];
      codes_s[tt * r + k] = (uint8_t)(int)fmin(fmax(rint(u64), 0.0), (double)qmax);
      note_ratio(p, uf, u64, tau);
    }
  } else {
    const double n64 = sqrt(dot2_row<BF16, WARP>(xs, tt, D, nullptr, lane));
    if (k == (int)kNormEntry) {
      if (lane == 0) {
        side_s[tt] = __double2half(n64);
        atomicAdd(nside, 1u);
      }
    } else {
      const double z64 = dot2_row<BF16, WARP>(xs, tt, D, Vt + (size_t)k * D, lane);
      if (lane == 0) {
        const double u64 = n64 > 0.0 ? z64 / n64 : 0.0;
        note_ratio(p, uf, u64, tau);
        double best = fabs(u64 - (double)p.codebook[0]);
        int bi = 0;
        for (int j = 1; j < p.cb_levels; ++j) {
          const double d = fabs(u64 - (double)p.codebook[j]);
          if (d < best) {
            best = d;
            bi = j;
          }
        }
        codes_s[tt * r + k] = (uint8_t)bi;
      }
    }
  }
}

}  // namespace
}  // namespace kvc
