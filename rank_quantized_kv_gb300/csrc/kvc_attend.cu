// Decode attention on the stored codes: one query per (batch, query head)
// over every stored token of a key layer and a value layer, without
// reconstructing keys or values (turboquant_cache page,
// TurboQuantKVCache.attend: scores from the packed keys, softmax of the
// scaled scores, weighted sum of the decoded values; palu_cache page: the
// latents are reconstructed only at attend time).
//
//   scores   uniform keys   k_hat = (lo + code step) V^T + mean, so
//                           q . k_hat = sum_j w_j code_j + c1 with
//                           w_j = (V^T q)_k step_k and c1 = (V^T q) . lo + q . mean;
//            codebook keys  k_hat = n R c[idx], so q . k_hat = n sum_k (R^T q)_k c[idx_k];
//                           with a residual sketch (turboquant_cache page,
//                           estimate_inner_product) plus
//                           sqrt(pi/2)/m ||r|| sum_j (S q)_j (2 bit_j - 1), and
//                           with an outlier stream plus s sum_l q_{ch_l} o8_l;
//   weights  softmax over the tokens, online and in base 2 (scale log2(e)
//            folded into w and c1);
//   output   int8 values    sum_t p_t s_t q8_t;
//            uniform values (sum_t p_t z_hat_t) V^T + mean, z_hat = lo + code step
//            (the weights sum to one).
//
// Three launches: prep (per query: w and c1), main (the tokens split across
// CTAs; each warp keeps a running maximum, sum and weighted accumulator per
// query head over 32-token blocks; the CTA merges its warps into one partial
// per query head), combine (the partials of a query merged, the output
// written).  Query head hq reads key/value head hq / rep.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "kvc_internal.h"

namespace kvc {

namespace {

constexpr int kMainThreads = 128;  // 4 warps
constexpr unsigned kFull = 0xffffffffu;

// Chunk-aligned packed positions of basis b (every width segment starts on a
// chunk of 8): entry c = first byte | width << 16 | (codes - 1) << 20 | valid << 31;
// the chunk's positions are 8 c .. 8 c + 7.
__device__ uint32_t chunk_entry(const Params& p, int beta, int c) {
  int nch = 0;
  for (int s = 0; s < kMaxSeg; ++s) {
    const int32_t* e = p.seg + ((size_t)beta * kMaxSeg + s) * 4;
    if (!e[3]) break;
    const int n = (e[3] + 7) / 8;
    if (c < nch + n) {
      const int ci = c - nch;
      const int nc = min(8, e[3] - ci * 8);
      return (uint32_t)(e[0] + e[1] * ci) | ((uint32_t)e[1] << 16) | ((uint32_t)(nc - 1) << 20) |
             (1u << 31);
    }
    nch += n;
  }
  return 0u;
}

// Component of packed position j of basis b (-1: padding).
__device__ int position_component(const Params& p, int beta, int j) {
  int nch = 0;
  for (int s = 0; s < kMaxSeg; ++s) {
    const int32_t* e = p.seg + ((size_t)beta * kMaxSeg + s) * 4;
    if (!e[3]) break;
    const int n = (e[3] + 7) / 8;
    if (j < (nch + n) * 8) {
      const int m = j - nch * 8;
      return m < e[3] ? p.order[(size_t)beta * p.r + e[2] + m] : -1;
    }
    nch += n;
  }
  return -1;
}

// The 64 bits of a packed row from byte a of a 4-byte aligned buffer.
__device__ __forceinline__ uint2 bits_at(const unsigned char* base, int a) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(base) + (a >> 2);
  const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
  const uint32_t sh = 8 * (a & 3);
  return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// Code e (0..7) of a chunk of width w starting at bit 0 of b.
__device__ __forceinline__ uint32_t chunk_code(uint2 b, int w, int e) {
  if (w == 8) return ((e < 4 ? b.x : b.y) >> (8 * (e & 3))) & 0xffu;
  return (b.x >> (w * e)) & ((1u << w) - 1u);
}

// REP consecutive fp32 weights from shared memory in as few vector loads as
// possible (16-byte aligned for REP >= 4).
template <int REP>
__device__ __forceinline__ void load_w(const float* src, float (&w)[REP]) {
  if constexpr (REP >= 4) {
#pragma unroll
    for (int q = 0; q < REP / 4; ++q) {
      const float4 v = reinterpret_cast<const float4*>(src)[q];
      w[4 * q] = v.x; w[4 * q + 1] = v.y; w[4 * q + 2] = v.z; w[4 * q + 3] = v.w;
    }
  } else if constexpr (REP == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    w[0] = v.x; w[1] = v.y;
  } else {
    w[0] = src[0];
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---------------------------------------------------------------- prep

// One block per (batch, query head): w_j = scale log2(e) (V^T q)_k coef_k at
// every packed position j of the key basis (coef = step in uniform mode, 1 for
// a codebook), and c1 = scale log2(e) ((V^T q) . lo + q . mean).
__global__ void attend_prep_kernel(const Params kp, const AttendArgs a) {
  __shared__ float qs[256];
  __shared__ float red[32];
  const int bq = blockIdx.x;
  const int b = bq / a.Hq, hq = bq - b * a.Hq;
  const int slot = b * kp.H + hq / a.rep;
  const int beta = kp.basis_of[slot];
  const int D = kp.D, tid = threadIdx.x;
  for (int i = tid; i < D; i += blockDim.x) qs[i] = a.q[(size_t)bq * D + i];
  float* w = a.w + (size_t)bq * a.NCk;
  for (int j = tid; j < a.NCk; j += blockDim.x) w[j] = 0.f;
  __syncthreads();
  const bool uniform = kp.mode == KVC_MODE_UNIFORM;
  float part = 0.f;
  for (int j = tid; j < a.NCk; j += blockDim.x) {
    const int k = position_component(kp, beta, j);
    if (k < 0) continue;
    // (V^T q)_k: the threads of a warp read one row of V [D_in][r] at their
    // columns; four partial sums keep the dependent chain short
    const float* vc = kp.V + (size_t)beta * D * kp.r + k;
    float q4[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < D; i += 4) {
#pragma unroll
      for (int e = 0; e < 4; ++e) q4[e] = fmaf(qs[i + e], vc[(size_t)(i + e) * kp.r], q4[e]);
    }
    const float qv = (q4[0] + q4[1]) + (q4[2] + q4[3]);
    const size_t bk = (size_t)beta * kp.r + k;
    w[j] = a.scale_log2 * qv * (uniform ? kp.step[bk] : 1.f);
    if (uniform) part = fmaf(qv, kp.lo[bk], part);
  }
  if (a.prod) {  // sketch weights sqrt(pi/2)/m (S q)_j, outlier weights q[ch_l]
    float* wx = a.wx + (size_t)bq * (a.m + a.n_out);
    const float coef = a.m ? 1.2533141373155003f / (float)a.m : 0.f;
    for (int j = tid; j < a.m; j += blockDim.x) {
      const float* srow = kp.W3 + (size_t)(D + j) * D;
      float sq = 0.f;
      for (int i = 0; i < D; ++i) sq = fmaf(srow[i], qs[i], sq);
      wx[j] = a.scale_log2 * coef * sq;
    }
    for (int l = tid; l < a.n_out; l += blockDim.x)
      wx[a.m + l] = a.scale_log2 * qs[kp.channels[(size_t)slot * a.n_out + l]];
  }
  if (uniform)
    for (int i = tid; i < D; i += blockDim.x) part = fmaf(qs[i], kp.mean[(size_t)beta * D + i], part);
  part = warp_sum(part);
  if ((tid & 31) == 0) red[tid >> 5] = part;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
    a.c1[bq] = a.scale_log2 * s;
  }
}

// ---------------------------------------------------------------- main

// Shared memory of the main kernel (dynamic), in order:
//   ws    [REP][NCk] fp32 key weights of the CTA's query heads
//   per warp: krow [32 Pk + 16], vrow [32 Pv + 16] (uniform values), ps [32][REP]
//   merge [4][REP][2 + Dv]
template <int KMODE, int VMODE, int REP, int DPL>
__global__ void __launch_bounds__(kMainThreads)
    attend_main_kernel(const Params kp, const Params vp, const AttendArgs a, int kstage,
                       int vstage) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ uint32_t kch[32], vch[32];
  __shared__ float cbv[256];
  __shared__ float c1s[REP];
  __shared__ float wxs[(kProdMaxM + kProdMaxOut) * REP];  // sketch, outlier weights [j][g]
  constexpr bool VU = VMODE == KVC_MODE_UNIFORM;
  constexpr int ACC = VU ? 8 : DPL;  // accumulator values per lane and query head
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slot = blockIdx.y, split = blockIdx.x;
  const int b = slot / kp.H;
  const int bq0 = b * a.Hq + (slot - b * kp.H) * REP;  // first query head of the slot
  const int kbeta = kp.basis_of[slot];
  const int vbeta = VU ? vp.basis_of[slot] : 0;
  const int NCk = a.NCk, Dv = a.Dv;
  const int Pk = kp.P[kbeta];
  const int Pv = VU ? vp.P[vbeta] : vp.D;
  float* ws = reinterpret_cast<float*>(sm);
  unsigned char* wbase = sm + (size_t)REP * NCk * 4 + (size_t)warp * (kstage + vstage + 32 * REP * 4);
  unsigned char* krow = wbase;
  unsigned char* vrow = wbase + kstage;
  float* ps = reinterpret_cast<float*>(wbase + kstage + vstage);
  float* merge = reinterpret_cast<float*>(sm + (size_t)REP * NCk * 4 +
                                          4 * (size_t)(kstage + vstage + 32 * REP * 4));
  if (tid < 32) {
    kch[tid] = chunk_entry(kp, kbeta, tid);
    vch[tid] = VU ? chunk_entry(vp, vbeta, tid) : 0u;
  }
  if (KMODE == KVC_MODE_CODEBOOK)
    for (int j = tid; j < kp.cb_levels; j += kMainThreads) cbv[j] = kp.codebook[j];
  for (int e = tid; e < REP * NCk; e += kMainThreads) {  // ws[j][g]: one vector load per position
    const int j = e / REP, g = e - j * REP;
    ws[e] = a.w[(size_t)(bq0 + g) * NCk + j];
  }
  if (tid < REP) c1s[tid] = KMODE == KVC_MODE_UNIFORM ? a.c1[bq0 + tid] : 0.f;
  const int nx = a.m + a.n_out;
  if (KMODE == KVC_MODE_CODEBOOK && a.prod)
    for (int e = tid; e < REP * nx; e += kMainThreads) {
      const int j = e / REP, g = e - j * REP;
      wxs[e] = a.wx[(size_t)(bq0 + g) * nx + j];
    }
  __syncthreads();
  int nchk = 0, nchv = 0;
  while (nchk < 32 && (kch[nchk] >> 31)) ++nchk;
  if (VU)
    while (nchv < 32 && (vch[nchv] >> 31)) ++nchv;
  // uniform values: lanes split as LG chunk lanes x (32 / LG) token groups
  int LG = 1;
  while (LG < nchv) LG *= 2;
  const int vc = lane & (LG - 1), tg = lane / LG, TG = 32 / LG;

  const int64_t t0 = (int64_t)split * a.span, t1 = min(a.S, t0 + a.span);
  const unsigned char* kbase = kp.store + kp.pay_off[slot];
  const __half* knorm = reinterpret_cast<const __half*>(kp.store + kp.side_off[slot]);
  const unsigned char* vbase = vp.store + vp.pay_off[slot];
  const __half* vscale = reinterpret_cast<const __half*>(vp.store + vp.side_off[slot]);

  float m[REP], l[REP], acc[REP][ACC];
#pragma unroll
  for (int g = 0; g < REP; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < ACC; ++e) acc[g][e] = 0.f;
  }

  for (int64_t tb = t0 + 32 * warp; tb < t1; tb += 128) {
    const int nrow = (int)min((int64_t)32, t1 - tb);
    // the block's packed key rows (and value rows): 16-byte copies (32 Pk is a
    // multiple of 16 and the block starts at a multiple of 32 tokens)
    {
      const uint4* src = reinterpret_cast<const uint4*>(kbase + tb * Pk);
      const int nv = (nrow * Pk + 15) >> 4;
      for (int i = lane; i < nv; i += 32) reinterpret_cast<uint4*>(krow)[i] = src[i];
      if (VU) {
        const uint4* vs = reinterpret_cast<const uint4*>(vbase + tb * Pv);
        const int nvv = (nrow * Pv + 15) >> 4;
        for (int i = lane; i < nvv; i += 32) reinterpret_cast<uint4*>(vrow)[i] = vs[i];
      }
    }
    __syncwarp();
    // scores of this lane's token, one per query head (base 2, scaled)
    float sc[REP];
    const bool live = lane < nrow;
#pragma unroll
    for (int g = 0; g < REP; ++g) sc[g] = c1s[g];
    if (live) {
      const int row = lane * Pk;  // byte offset of the lane's row in the staging
      for (int c = 0; c < nchk; ++c) {
        const uint32_t ent = kch[c];
        const int w = (int)((ent >> 16) & 0xfu);
        const uint2 bits = bits_at(krow, row + (int)(ent & 0xffffu));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t code = chunk_code(bits, w, e);
          const float v = KMODE == KVC_MODE_CODEBOOK ? cbv[code] : (float)code;
          float wv[REP];
          load_w<REP>(ws + (8 * c + e) * REP, wv);
#pragma unroll
          for (int g = 0; g < REP; ++g) sc[g] = fmaf(wv[g], v, sc[g]);
        }
      }
      if (KMODE == KVC_MODE_CODEBOOK) {
        const int64_t sw = (tb + lane) * a.knw;  // the key's side words
        const float n = __half2float(knorm[sw]);
#pragma unroll
        for (int g = 0; g < REP; ++g) sc[g] *= n;
        if (a.prod) {
          if (a.m) {  // + ||r|| sum_j w_j (2 bit_j - 1)
            const unsigned char* sb = krow + row + a.kcode;
            float qj[REP];
#pragma unroll
            for (int g = 0; g < REP; ++g) qj[g] = 0.f;
            for (int j8 = 0; j8 < (a.m >> 3); ++j8) {
              const uint32_t byte = sb[j8];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float f = (byte >> e) & 1u ? 1.f : -1.f;
#pragma unroll
                for (int g = 0; g < REP; ++g) qj[g] = fmaf(wxs[(8 * j8 + e) * REP + g], f, qj[g]);
              }
            }
            const float gam = __half2float(knorm[sw + 1]);
#pragma unroll
            for (int g = 0; g < REP; ++g) sc[g] = fmaf(gam, qj[g], sc[g]);
          }
          if (a.n_out) {  // + s sum_l q[ch_l] o8_l
            const int8_t* o8 = reinterpret_cast<const int8_t*>(krow + row + a.kcode + (a.m >> 3));
            float qo[REP];
#pragma unroll
            for (int g = 0; g < REP; ++g) qo[g] = 0.f;
            for (int l = 0; l < a.n_out; ++l) {
              const float v = (float)o8[l];
#pragma unroll
              for (int g = 0; g < REP; ++g) qo[g] = fmaf(wxs[(a.m + l) * REP + g], v, qo[g]);
            }
            const float os = __half2float(knorm[sw + a.knw - 1]);
#pragma unroll
            for (int g = 0; g < REP; ++g) sc[g] = fmaf(os, qo[g], sc[g]);
          }
        }
      }
    } else {
#pragma unroll
      for (int g = 0; g < REP; ++g) sc[g] = -INFINITY;
    }
    // online softmax: rescale the running state to the block's new maximum
    const float s_t = (!VU && live) ? __half2float(vscale[tb + lane]) : 1.f;
#pragma unroll
    for (int g = 0; g < REP; ++g) {
      const float mn = fmaxf(m[g], warp_max(sc[g]));
      const float corr = exp2f(m[g] - mn);
      const float pt = live ? exp2f(sc[g] - mn) : 0.f;
      l[g] = l[g] * corr + warp_sum(pt);
      m[g] = mn;
#pragma unroll
      for (int e = 0; e < ACC; ++e) acc[g][e] *= corr;
      ps[lane * REP + g] = pt * s_t;
    }
    __syncwarp();
    if (!VU) {
      // int8 values: lane owns DPL consecutive channels, token rows read whole
      for (int tt = 0; tt < nrow; ++tt) {
        const unsigned char* vr = vbase + (tb + tt) * (int64_t)Pv + lane * DPL;
        int8_t q8[DPL];
        if (DPL == 8) {
          const uint2 u = *reinterpret_cast<const uint2*>(vr);
          *reinterpret_cast<uint2*>(q8) = u;
        } else if (DPL == 4) {
          *reinterpret_cast<uint32_t*>(q8) = *reinterpret_cast<const uint32_t*>(vr);
        } else {
          *reinterpret_cast<uint16_t*>(q8) = *reinterpret_cast<const uint16_t*>(vr);
        }
        float pv[REP];
#pragma unroll
        for (int g = 0; g < REP; ++g) pv[g] = ps[tt * REP + g];
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          const float v = (float)q8[e];
#pragma unroll
          for (int g = 0; g < REP; ++g) acc[g][e] = fmaf(pv[g], v, acc[g][e]);
        }
      }
    } else if (vc < nchv) {
      // uniform values: lane (chunk vc, token group tg) sums p_t code_t
      const uint32_t ent = vch[vc];
      const int w = (int)((ent >> 16) & 0xfu), off = (int)(ent & 0xffffu);
      for (int tt = tg; tt < nrow; tt += TG) {
        const uint2 bits = bits_at(vrow, tt * Pv + off);
        float pv[REP];
#pragma unroll
        for (int g = 0; g < REP; ++g) pv[g] = ps[tt * REP + g];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float v = (float)chunk_code(bits, w, e);
#pragma unroll
          for (int g = 0; g < REP; ++g) acc[g][e] = fmaf(pv[g], v, acc[g][e]);
        }
      }
    }
    __syncwarp();  // staging and ps are rewritten by the next block
  }
  if (VU) {  // sum the token groups of each chunk lane
    for (int o = LG; o < 32; o <<= 1)
#pragma unroll
      for (int g = 0; g < REP; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(kFull, acc[g][e], o);
  }
  // merge the 4 warps: merge[w][g] = {m, l, acc[Dv]}
  const int stride = 2 + Dv;
  for (int e = tid; e < 4 * REP * stride; e += kMainThreads) merge[e] = 0.f;
  __syncthreads();
#pragma unroll
  for (int g = 0; g < REP; ++g) {
    float* mg = merge + ((size_t)warp * REP + g) * stride;
    if (lane == 0) {
      mg[0] = m[g];
      mg[1] = l[g];
    }
    if (!VU) {
#pragma unroll
      for (int e = 0; e < DPL; ++e) mg[2 + lane * DPL + e] = acc[g][e];
    } else if (tg == 0 && vc < nchv) {
#pragma unroll
      for (int e = 0; e < 8; ++e) mg[2 + vc * 8 + e] = acc[g][e];
    }
  }
  __syncthreads();
  float* out = a.part + (((size_t)slot * a.splits + split) * REP) * stride;
  for (int e = tid; e < REP * stride; e += kMainThreads) {
    const int g = e / stride, d = e - g * stride;
    float M = -INFINITY;
    for (int w4 = 0; w4 < 4; ++w4) M = fmaxf(M, merge[((size_t)w4 * REP + g) * stride]);
    float v = 0.f;
    if (d == 0) {
      v = M;
    } else {
      for (int w4 = 0; w4 < 4; ++w4) {
        const float* mg = merge + ((size_t)w4 * REP + g) * stride;
        if (mg[0] == -INFINITY) continue;  // a warp without tokens
        v = fmaf(exp2f(mg[0] - M), mg[d], v);
      }
    }
    out[(size_t)g * stride + d] = v;
  }
}

// ---------------------------------------------------------------- combine

// One block per (batch, query head): merge the splits' partials, normalise,
// and write the output row (uniform values: project the mean latent).
__global__ void attend_combine_kernel(const Params kp, const Params vp, const AttendArgs a) {
  __shared__ float zbar[256];
  __shared__ int comp[256];
  const int bq = blockIdx.x;
  const int b = bq / a.Hq, hq = bq - b * a.Hq;
  const int h = hq / a.rep, g = hq - h * a.rep;
  const int slot = b * kp.H + h;
  const int stride = 2 + a.Dv, tid = threadIdx.x;
  const float* part = a.part + ((size_t)slot * a.splits * a.rep + g) * stride;
  const size_t sstride = (size_t)a.rep * stride;  // next split
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, part[s * sstride]);
  float L = 0.f;
  for (int s = 0; s < a.splits; ++s) L = fmaf(exp2f(part[s * sstride] - M), part[s * sstride + 1], L);
  const float invL = 1.f / L;
  const int D = vp.D;
  const bool vu = vp.mode == KVC_MODE_UNIFORM;
  float* zb = zbar;
  for (int d = tid; d < a.Dv; d += blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < a.splits; ++s)
      v = fmaf(exp2f(part[s * sstride] - M), part[s * sstride + 2 + d], v);
    v *= invL;
    if (!vu) {
      const size_t o = (size_t)bq * D + d;
      if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v);
      else reinterpret_cast<__half*>(a.out)[o] = __float2half_rn(v);
    } else {
      zb[d] = v;
    }
  }
  if (!vu) return;
  const int beta = vp.basis_of[slot];
  for (int j = tid; j < a.Dv; j += blockDim.x) {
    const int k = position_component(vp, beta, j);
    comp[j] = k;
    if (k >= 0) {
      const size_t bk = (size_t)beta * vp.r + k;
      zb[j] = vp.lo[bk] + vp.step[bk] * zb[j];  // the weighted mean latent
    }
  }
  __syncthreads();
  for (int i = tid; i < D; i += blockDim.x) {
    float v = vp.mean[(size_t)beta * D + i];
    const float* Vrow = vp.V + ((size_t)beta * D + i) * vp.r;
    for (int j = 0; j < a.Dv; ++j) {
      const int k = comp[j];
      if (k >= 0) v = fmaf(zb[j], Vrow[k], v);
    }
    const size_t o = (size_t)bq * D + i;
    if (a.out_bf16) reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(v);
    else reinterpret_cast<__half*>(a.out)[o] = __float2half_rn(v);
  }
}

using MainKernel = void (*)(const Params, const Params, const AttendArgs, int, int);

template <int KMODE, int VMODE, int REP>
MainKernel main_for_dpl(int dpl) {
  if (VMODE == KVC_MODE_UNIFORM) return attend_main_kernel<KMODE, VMODE, REP, 8>;
  switch (dpl) {
    case 2: return attend_main_kernel<KMODE, VMODE, REP, 2>;
    case 4: return attend_main_kernel<KMODE, VMODE, REP, 4>;
    default: return attend_main_kernel<KMODE, VMODE, REP, 8>;
  }
}

template <int KMODE, int VMODE>
MainKernel main_for_rep(int rep, int dpl) {
  switch (rep) {
    case 1: return main_for_dpl<KMODE, VMODE, 1>(dpl);
    case 2: return main_for_dpl<KMODE, VMODE, 2>(dpl);
    case 4: return main_for_dpl<KMODE, VMODE, 4>(dpl);
    default: return main_for_dpl<KMODE, VMODE, 8>(dpl);
  }
}

MainKernel main_kernel_for(int kmode, int vmode, int rep, int dpl) {
  if (kmode == KVC_MODE_UNIFORM)
    return vmode == KVC_MODE_UNIFORM ? main_for_rep<KVC_MODE_UNIFORM, KVC_MODE_UNIFORM>(rep, dpl)
                                     : main_for_rep<KVC_MODE_UNIFORM, KVC_MODE_INT8>(rep, dpl);
  return vmode == KVC_MODE_UNIFORM ? main_for_rep<KVC_MODE_CODEBOOK, KVC_MODE_UNIFORM>(rep, dpl)
                                   : main_for_rep<KVC_MODE_CODEBOOK, KVC_MODE_INT8>(rep, dpl);
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

size_t attend_plan(int B, int Hq, int n_slots, int rep, int64_t S, int NCk, int Dv, int sms,
                   int extra, int* splits, int64_t* span) {
  // enough CTAs for about twelve per SM (the main kernel is bound by load
  // latency; more resident warps hide more of it), at least 128 tokens each (a
  // multiple of 128 so that every warp's 32-token blocks start at a multiple
  // of 32)
  const int64_t max_splits = std::max<int64_t>(1, (S + 127) / 128);
  int64_t sp = std::min<int64_t>(max_splits, std::max<int64_t>(1, (12 * sms + n_slots - 1) / n_slots));
  int64_t sn = (S + sp - 1) / sp;
  sn = (sn + 127) / 128 * 128;
  sp = (S + sn - 1) / sn;
  *splits = (int)std::max<int64_t>(sp, 1);
  *span = sn;
  const size_t w = align256((size_t)B * Hq * NCk * 4);
  const size_t c1 = align256((size_t)B * Hq * 4);
  const size_t part = align256((size_t)n_slots * (*splits) * rep * (2 + Dv) * 4);
  const size_t wx = align256((size_t)B * Hq * extra * 4);
  return w + c1 + part + wx;
}

cudaError_t launch_attend(const Params& kp, const Params& vp, AttendArgs a, void* workspace,
                          cudaStream_t s, int* nk) {
  const size_t wbytes = align256((size_t)kp.B * a.Hq * a.NCk * 4);
  const size_t cbytes = align256((size_t)kp.B * a.Hq * 4);
  a.w = static_cast<float*>(workspace);
  a.c1 = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + wbytes);
  a.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + wbytes + cbytes);
  const size_t pbytes = align256((size_t)kp.n_slots * a.splits * a.rep * (2 + a.Dv) * 4);
  a.wx = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + wbytes + cbytes + pbytes);
  attend_prep_kernel<<<(unsigned)(kp.B * a.Hq), 128, 0, s>>>(kp, a);
  ++*nk;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int kstage = (32 * a.Pk_max + 16 + 15) / 16 * 16;
  const int vstage = vp.mode == KVC_MODE_UNIFORM ? (32 * a.Pv_max + 16 + 15) / 16 * 16 : 0;
  const size_t smem = (size_t)a.rep * a.NCk * 4 + 4 * (size_t)(kstage + vstage + 32 * a.rep * 4) +
                      4 * (size_t)a.rep * (2 + a.Dv) * 4;
  MainKernel k = main_kernel_for(kp.mode, vp.mode, a.rep, kp.D / 32);
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<dim3((unsigned)a.splits, (unsigned)kp.n_slots), kMainThreads, smem, s>>>(kp, vp, a, kstage,
                                                                                vstage);
  ++*nk;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attend_combine_kernel<<<(unsigned)(kp.B * a.Hq), 128, 0, s>>>(kp, vp, a);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
