// Tensor-core kernels of the hot path (sm_103a): fetch as a tcgen05 contraction.
//
// Fetch of one 128-token tile of one slot, one CTA of 128 threads (thread t
// owns token t of the tile, i.e. TMEM lane t):
//   1. copy the tile's packed rows (and fp16 side words) to shared memory;
//   2. thread t decodes its row into the fp16 A operand (UMMA K-major, no
//      swizzle), K = kept components in packed order:
//        uniform   A = code - 2^(b-1)            (exact; B = fp16(step * V^T))
//        group     A = fp16((code - 2^(b-1)) * s) (B = fp16(V^T))
//        codebook  A = fp16(c[code])             (B = fp16(R^T), norm in the epilogue)
//   3. one thread issues K/16 tcgen05.mma (M = 128, N = D) into TMEM;
//   4. the epilogue reads TMEM (tcgen05.ld 32x32b), adds the per-basis bias
//      mean + sum_k (lo_k + 2^(b_k-1) step_k) V_k (uniform), mean (group) or
//      scales by the fp16 norm (codebook), converts to fp16/bf16 into a
//      128-byte-swizzled staging tile and TMA-stores it to [B, H, S, D];
//      rows past the length are clipped by the tensor map.
// In group mode the tile is decoded once and contracted against each head's
// slice of the group basis in turn.  Several CTAs per SM overlap the phases.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "kvc_append_exact.cuh"
#include "kvc_sm100.cuh"
#include "kvc_tc.h"

namespace kvc {

using namespace sm100;

namespace {

constexpr int kTile = 128;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait

struct FetchTc {
  const uint16_t* B;  // fp16 bits, [nb][D_in][K] UMMA order
  const float* bias;  // [nb][D_in]
  int K;
  int cols;
};

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Accumulates fp16 values of one A row and stores them 8 at a time (16 bytes)
// at the row's place in the UMMA no-swizzle K-major layout.
struct RowWriter {
  unsigned char* row_base;  // A + (t / 8) * sbo + (t % 8) * 16
  uint64_t lo = 0, hi = 0;  // values 0-3 and 4-7 of the current chunk
  int n = 0;                // values in the current chunk
  int kc = 0;               // chunk index along K
  __device__ __forceinline__ void push(__half v) {
    const uint64_t bits = __half_as_ushort(v);
    if (n < 4)
      lo |= bits << (16 * n);
    else
      hi |= bits << (16 * (n - 4));
    if (++n == 8) {
      *reinterpret_cast<uint4*>(row_base + kc * 128) =
          make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
      lo = hi = 0;
      n = 0;
      ++kc;
    }
  }
  __device__ __forceinline__ void pad_to(int K) {
    while (kc * 8 + n < K) push(__ushort_as_half(0));
  }
};

template <int MODE, bool OUT_BF16>
__global__ void __launch_bounds__(kTile) fetch_tc_kernel(const Params p, const FetchTc t,
                                                         const __grid_constant__ CUtensorMap omap,
                                                         int64_t S, int tiles_per_slot) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int D = p.D, K = t.K, nbox = D / 64;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int slot = blockIdx.x / tiles_per_slot;
  const int64_t t0 = (int64_t)(blockIdx.x % tiles_per_slot) * kTile;
  const int n = (int)min((int64_t)kTile, S - t0);
  const int beta = p.basis_of[slot];
  const int P = p.P[beta];
  const int sbytes = p.side_bytes;
  const int b = slot / p.Hg, g = slot % p.Hg;

  unsigned char* stage = smem;                               // nbox x [128 rows x 128 B]
  unsigned char* As = stage + nbox * 16384;                  // [128 x K] fp16
  unsigned char* Bs = As + kTile * K * 2;                    // [D x K] fp16
  float* bias_s = reinterpret_cast<float*>(Bs + D * K * 2);  // [D]
  float* cb_s = bias_s + D;                                  // [256]
  unsigned char* codes_s = reinterpret_cast<unsigned char*>(cb_s + 256);
  unsigned char* side_s = codes_s + ((kTile * P + 16 + 15) & ~15);

  if (warp == 0) tmem_alloc(&tmem_base, t.cols);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  {  // packed rows and side words of the tile (16-byte aligned, over-read <= 15 bytes)
    const uint4* src = reinterpret_cast<const uint4*>(p.store + p.pay_off[slot] + t0 * P);
    const int nv = (n * P + 15) >> 4;
    for (int i = tid; i < nv; i += kTile) reinterpret_cast<uint4*>(codes_s)[i] = src[i];
    if (sbytes) {
      const uint4* ss = reinterpret_cast<const uint4*>(p.store + p.side_off[slot] + t0 * sbytes);
      const int ns = (n * sbytes + 15) >> 4;
      for (int i = tid; i < ns; i += kTile) reinterpret_cast<uint4*>(side_s)[i] = ss[i];
    }
    if (MODE == KVC_MODE_CODEBOOK)
      for (int j = tid; j < p.cb_levels; j += kTile) cb_s[j] = p.codebook[j];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_base;

  // ---- decode row tid into A
  const uint32_t sbo = (uint32_t)(K / 8) * 128;
  RowWriter w{As + (tid >> 3) * sbo + (tid & 7) * 16};
  if (tid < n) {
    const unsigned char* row = codes_s + tid * P;
    const int32_t* seg = p.seg + (int64_t)beta * kMaxSeg * 4;
    int kk = 0, gi = 0, gend = 0;
    float gscale = 0.f;
    if (MODE == KVC_MODE_GROUP) {
      gend = p.groups[1];
      gscale = __half2float(reinterpret_cast<const __half*>(side_s + tid * sbytes)[0]);
    }
    for (int s = 0; s < kMaxSeg; ++s) {
      const int cnt = seg[s * 4 + 3];
      if (!cnt) break;
      const int start = seg[s * 4 + 0], wd = seg[s * 4 + 1];
      const int off = 1 << (wd - 1);
      const unsigned mask = (1u << wd) - 1u;
      for (int m = 0; m < cnt; ++m, ++kk) {
        const int bit = start * 8 + m * wd;
        unsigned v = row[bit >> 3];
        if ((bit & 7) + wd > 8) v |= (unsigned)row[(bit >> 3) + 1] << 8;
        const int code = (int)((v >> (bit & 7)) & mask);
        if (MODE == KVC_MODE_UNIFORM) {
          w.push(__int2half_rn(code - off));
        } else if (MODE == KVC_MODE_GROUP) {
          if (kk == gend) {
            ++gi;
            gend += p.groups[gi * 3 + 1];
            gscale = __half2float(reinterpret_cast<const __half*>(side_s + tid * sbytes)[gi]);
          }
          w.push(__float2half_rn((float)(code - off) * gscale));
        } else {
          w.push(__float2half_rn(cb_s[code]));
        }
      }
      w.pad_to((w.kc * 8 + w.n + 7) & ~7);  // the next segment starts a new chunk
    }
  }
  w.pad_to(K);
  fence_proxy_async_smem();

  float nrm = 1.f;
  if (MODE == KVC_MODE_CODEBOOK && tid < n)
    nrm = __half2float(reinterpret_cast<const __half*>(side_s)[tid]);

  const uint32_t idesc = idesc_f16(kTile, D, 0);
  uint32_t phase = 0;
  for (int j = 0; j < p.hpg; ++j) {
    {  // this head's slice of B and of the bias
      const uint4* bsrc = reinterpret_cast<const uint4*>(
          t.B + ((size_t)beta * p.d_in + (size_t)j * D) * (size_t)K);
      const int nv = D * K * 2 / 16;
      for (int i = tid; i < nv; i += kTile) reinterpret_cast<uint4*>(Bs)[i] = bsrc[i];
      for (int c = tid; c < D; c += kTile) bias_s[c] = t.bias[(size_t)beta * p.d_in + j * D + c];
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      for (int ks = 0; ks < K / 16; ++ks) {
        const uint64_t ad = desc_kmajor_noswizzle(smem_u32(As) + ks * 256, 128, sbo);
        const uint64_t bd = desc_kmajor_noswizzle(smem_u32(Bs) + ks * 256, 128, sbo);
        umma_f16(taddr, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
      umma_commit(&bar);
    }
    const bool ok = mbar_wait_bounded(&bar, phase, kWaitNs);
    phase ^= 1;
    tc_fence_after();
    if (!ok) abort_flag = 1;
    if (tid == 0) bulk_wait_read0();  // the previous head's stores have left the staging tile
    __syncthreads();
    if (abort_flag) {
      if (tid == 0) set_err(p.err, kErrTimeout);
      break;
    }
    // ---- epilogue: TMEM -> registers -> fp16/bf16 -> swizzled staging
    const uint32_t lane_addr = taddr + ((uint32_t)(warp * 32) << 16);
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t r[32];
      tmem_ld32(lane_addr + cc * 32, r);
      tmem_wait_ld();
      unsigned char* dst = stage + (cc >> 1) * 16384 + tid * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c0 = q * 8 + 2 * e;
          float v0 = __uint_as_float(r[c0]), v1 = __uint_as_float(r[c0 + 1]);
          if (MODE == KVC_MODE_CODEBOOK) {
            v0 *= nrm;
            v1 *= nrm;
          } else {
            v0 += bias_s[cc * 32 + c0];
            v1 += bias_s[cc * 32 + c0 + 1];
          }
          h[e] = OUT_BF16 ? pack_bf162(v0, v1) : pack_half2(v0, v1);
        }
        const int c16 = (cc & 1) * 4 + q;
        *reinterpret_cast<uint4*>(dst + ((c16 ^ (tid & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const int z = b * p.H + g * p.hpg + j;
      for (int bx = 0; bx < nbox; ++bx) tma_store_3d(&omap, stage + bx * 16384, bx * 64, (int)t0, z);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait0();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(taddr, t.cols);
  }
}

// ---------------------------------------------------------------- append
//
// One CTA per 128-token tile of one slot (thread t = token t = TMEM lane t).
// The x tile arrives by TMA (128-byte swizzle) and is the A operand as is
// (bf16 or fp16 values are exact).  B holds the fp32 basis as three exact
// 16-bit pieces, each accumulated in its own TMEM region, so z = hi + mid + lo.
// Error bound of the tensor-core accumulation (a model of aligned, truncated
// fp32 accumulation, per K = 16 block at most 17 ulp of the running magnitude,
// itself <= sum_i |x_i V_ik| <= ||x|| ||V_k||):
//   |z32 - z| <= gamma * ||x|| * ||V_k|| + 2^-21 (|z| + |mean . V_k|),
//   gamma = (17 D/16 + 2) 2^-23 (1 + 2^-7).
// Codes closer than that (through the quantiser's own roundings) to a rounding
// boundary are queued and re-decided by a warp with a compensated fp32 dot
// product (error ~ 1e-13 relative) finished in double precision.

// ---------------------------------------------------------------- append, 512 threads
//
// Same arithmetic as above with the tile's work spread over 16 warps: warp w
// reads TMEM lanes 32 (w % 4) .. +31 (its tokens) and column block w / 4 (a
// quarter of the components).  Accumulators: the hi piece alone, the smaller
// pieces together (their accumulation error is <= 2^-8 of the hi piece's).

constexpr int kV3 = 512;

template <int MODE, bool BF16, int CW>
__global__ void __launch_bounds__(kV3) append_tc_v3(const Params p, const AppendTc t,
                                                    const __grid_constant__ CUtensorMap xmap,
                                                    const AppendArgs a, int tiles_per_slot,
                                                    int npieces) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t tma_bar, mma_bar;
  __shared__ uint32_t tmem_base;
  __shared__ unsigned qcount, nside;
  __shared__ int abort_flag;
  __shared__ int32_t seg_s[kMaxSeg * 4];

  constexpr int rpad = 4 * CW;
  const int D = p.D, r = p.r, nbox = D / 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, cblk = warp >> 2;
  const int row = quarter * 32 + lane;  // token of this thread within the tile
  const int slot = blockIdx.x / tiles_per_slot;
  const int64_t t0 = (int64_t)(blockIdx.x % tiles_per_slot) * kTile;
  const int n = (int)min((int64_t)kTile, a.T - t0);
  const int beta = p.basis_of[slot];
  const int P = p.P[beta];
  const int b = slot / p.H, h = slot % p.H;

  unsigned char* xs = smem;                                           // nbox x 16 KB
  unsigned char* Bs = xs + nbox * 16384;                              // npieces x rpad x D
  unsigned char* codes_s = Bs + npieces * rpad * D * 2;               // [128][r]
  uint32_t* queue = reinterpret_cast<uint32_t*>(codes_s + ((kTile * r + 15) & ~15));
  float2* aux = reinterpret_cast<float2*>(queue + kQueue);
  float* nsq_s = reinterpret_cast<float*>(aux + kQueue);              // [4][128]
  float* lo_s = nsq_s + 4 * kTile;                                     // [rpad] each
  float* inv_s = lo_s + rpad;
  float* ck_s = inv_s + rpad;
  float* vn_s = ck_s + rpad;
  float* mids_s = vn_s + rpad;                                         // [256]
  __half* side_s = reinterpret_cast<__half*>(mids_s + 256);           // [128]
  int16_t* order_s = reinterpret_cast<int16_t*>(side_s + kTile);      // [rpad]
  uint8_t* bits_s = reinterpret_cast<uint8_t*>(order_s + rpad);       // [rpad]

  if (warp == 0) tmem_alloc(&tmem_base, t.cols);
  if (tid == 0) {
    mbar_init(&tma_bar, 1);
    mbar_init(&mma_bar, 1);
    fence_mbar_init();
    qcount = 0;
    nside = 0;
    abort_flag = 0;
    mbar_arrive_expect_tx(&tma_bar, nbox * 16384);
    for (int bx = 0; bx < nbox; ++bx) tma_load_4d(xs + bx * 16384, &xmap, &tma_bar, bx * 64, (int)t0, h, b);
  }
  {
    const uint4* src = reinterpret_cast<const uint4*>(t.B + (size_t)beta * npieces * rpad * D);
    const int nv = npieces * rpad * D * 2 / 16;
    for (int i = tid; i < nv; i += kV3) reinterpret_cast<uint4*>(Bs)[i] = src[i];
    for (int k = tid; k < rpad; k += kV3) {
      const bool in = k < r;
      const size_t bk = (size_t)beta * r + k;
      lo_s[k] = in && MODE == KVC_MODE_UNIFORM ? p.lo[bk] : 0.f;
      inv_s[k] = in && MODE == KVC_MODE_UNIFORM ? p.inv_step[bk] : 0.f;
      ck_s[k] = in ? (float)t.c64[bk] : 0.f;
      vn_s[k] = in ? p.vnorm[bk] : 0.f;
      bits_s[k] = in ? p.bits[bk] : 0;
      order_s[k] = in ? p.order[bk] : 0;
    }
    if (MODE == KVC_MODE_CODEBOOK)
      for (int j = tid; j < p.cb_levels - 1; j += kV3) mids_s[j] = p.mids[j];
    if (tid < kMaxSeg * 4) seg_s[tid] = p.seg[(int64_t)beta * kMaxSeg * 4 + tid];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tmem_base;

  if (!mbar_wait_bounded(&tma_bar, 0, kWaitNs)) abort_flag = 1;
  __syncthreads();
  if (!abort_flag && tid == 0) {
    const uint32_t idesc = idesc_f16(kTile, rpad, BF16 ? 1 : 0);
    const uint32_t sbo = (uint32_t)(D / 8) * 128;
    for (int pc = 0; pc < npieces; ++pc)
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t ad = desc_kmajor_sw128(smem_u32(xs) + (ks >> 2) * 16384 + (ks & 3) * 32);
        const uint64_t bd =
            desc_kmajor_noswizzle(smem_u32(Bs) + pc * rpad * D * 2 + ks * 256, 128, sbo);
        umma_f16(taddr + (pc ? rpad : 0), ad, bd, idesc, (pc > 1 || ks > 0) ? 1u : 0u);
      }
    umma_commit(&mma_bar);
  }
  {  // partial ||x||^2 over this warp's quarter of the row
    float acc = 0.f;
    const int c0 = cblk * (D / 4);
    for (int c = c0; c < c0 + D / 4; c += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(
          xs + (c >> 6) * 16384 + row * 128 + (((((c & 63) >> 3)) ^ (row & 7)) << 4));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float e0, e1;
        if (BF16) {
          e0 = __bfloat162float(__ushort_as_bfloat16((uint16_t)(w4[q] & 0xffff)));
          e1 = __bfloat162float(__ushort_as_bfloat16((uint16_t)(w4[q] >> 16)));
        } else {
          e0 = __half2float(__ushort_as_half((uint16_t)(w4[q] & 0xffff)));
          e1 = __half2float(__ushort_as_half((uint16_t)(w4[q] >> 16)));
        }
        acc = fmaf(e0, e0, acc);
        acc = fmaf(e1, e1, acc);
      }
    }
    nsq_s[cblk * kTile + row] = acc;
  }
  if (!abort_flag && !mbar_wait_bounded(&mma_bar, 0, kWaitNs)) abort_flag = 1;
  tc_fence_after();
  __syncthreads();
  if (abort_flag) {
    if (tid == 0) set_err(p.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(taddr, t.cols);
    }
    return;
  }
  const float nx = sqrtf(((nsq_s[row] + nsq_s[kTile + row]) + nsq_s[2 * kTile + row]) +
                         nsq_s[3 * kTile + row]);

  // ---- fast path: components cblk*CW .. +CW of token `row`
  const float kU = 5.9604644775390625e-08f;
  const float nxb = nx * (1.f + 1e-3f);
  const float eps_n = 0.5f * ((D + 2) * kU) / (1.f - (D + 2) * kU) + 2.f * kU;
  float z[CW];
  {
    uint32_t rr[CW];
    const uint32_t la = taddr + ((uint32_t)(quarter * 32) << 16) + cblk * CW;
    tmem_ld_n<CW>(la, rr);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < CW; ++i) z[i] = __uint_as_float(rr[i]);
    tmem_ld_n<CW>(la + rpad, rr);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < CW; ++i) z[i] += __uint_as_float(rr[i]);
  }
  tc_fence_before();
  const bool tiny = MODE == KVC_MODE_CODEBOOK && nx < 1e-18f;
  float cmax = 0.f;
  if (MODE == KVC_MODE_CODEBOOK) cmax = fmaxf(fabsf(p.codebook[0]), fabsf(p.codebook[p.cb_levels - 1]));
  if (row < n) {
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      const int k = cblk * CW + i;
      if (k >= r) continue;
      bool near = false;
      int code = 0;
      float uf = 0.f, tf = 0.f;
      if (MODE == KVC_MODE_UNIFORM) {
        const int w = bits_s[k];
        if (w == 0) continue;
        const float ck = ck_s[k];
        const float zc = z[i] * t.inv_scale - ck;
        const float inv = inv_s[k];
        const float u = (zc - lo_s[k]) * inv;
        const float tz = t.gamma * nxb * vn_s[k] + 4.f * kU * (fabsf(zc) + fabsf(ck));
        const float tau = tz * inv * (1.f + 1e-6f) + 4.f * kU * (fabsf(u) + 1.f);
        const int qmax = (1 << w) - 1;
        const float hb = fminf(fmaxf(floorf(u) + 0.5f, 0.5f), (float)qmax - 0.5f);
        near = fabsf(u - hb) <= tau;
        code = (int)fminf(fmaxf(rintf(u), 0.f), (float)qmax);
        uf = u;
        tf = tau;
      } else {
        const int L = p.cb_levels;
        const float u = tiny ? 0.f : z[i] * t.inv_scale / nx;
        int lo_i = 0, hi_i = L - 1;
        while (lo_i < hi_i) {
          const int mid = (lo_i + hi_i) >> 1;
          if (mids_s[mid] < u) lo_i = mid + 1; else hi_i = mid;
        }
        code = lo_i;
        float dmin = 3.4e38f;
        if (code > 0) dmin = fminf(dmin, fabsf(u - mids_s[code - 1]));
        if (code < L - 1) dmin = fminf(dmin, fabsf(u - mids_s[code]));
        const float tau = (t.gamma * vn_s[k] * (1.f + 1e-3f) + fabsf(u) * eps_n) * (1.f + 1e-6f) +
                          4.f * kU * (fabsf(u) + cmax);
        near = tiny || dmin <= tau;
        uf = u;
        tf = tiny ? 0.f : tau;
      }
      codes_s[row * r + k] = (uint8_t)code;
      if (near) {
        const unsigned q = atomicAdd(&qcount, 1u);
        if (q < kQueue) {
          queue[q] = ((uint32_t)row << 16) | (uint32_t)k;
          aux[q] = make_float2(uf, tf);
        } else {  // queue full: decide it here, alone
          refine_entry<MODE, BF16, false>(p, t, beta, xs, codes_s, side_s, &nside, row, k, 0);
        }
      }
    }
    if (MODE == KVC_MODE_CODEBOOK && cblk == 0) {
      if (tiny || !same_half(nx * (1.f - eps_n), nx * (1.f + eps_n))) {
        const unsigned q = atomicAdd(&qcount, 1u);
        if (q < kQueue) {
          queue[q] = ((uint32_t)row << 16) | kNormEntry;
          aux[q] = make_float2(0.f, 0.f);
        } else {
          refine_entry<MODE, BF16, false>(p, t, beta, xs, codes_s, side_s, &nside, row,
                                          (int)kNormEntry, 0);
        }
      } else {
        side_s[row] = __float2half_rn(nx);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(taddr, t.cols);
  }

  // ---- exact re-decision of the queued codes, one warp per entry
  const unsigned nq = qcount;
  for (unsigned e = warp; e < min(nq, (unsigned)kQueue); e += kV3 / 32) {
    const uint32_t ent = queue[e];
    const float2 ax = aux[e];
    refine_entry<MODE, BF16, true>(p, t, beta, xs, codes_s, side_s, &nside, (int)(ent >> 16),
                                   (int)(ent & 0xffffu), lane, ax.x, ax.y);
  }
  __syncthreads();

  // ---- pack: one thread per output byte, written straight to the store
  unsigned char* dst = p.store + p.pay_off[slot] + (a.t_base + t0) * P;
  for (int idx = tid; idx < n * P; idx += kV3) {
    const int tt = idx / P, j = idx - tt * P;
    int s = 0;
    while (s + 1 < kMaxSeg && seg_s[(s + 1) * 4 + 3] > 0 && seg_s[(s + 1) * 4 + 0] <= j) ++s;
    const int start = seg_s[s * 4 + 0], wd = seg_s[s * 4 + 1], m0 = seg_s[s * 4 + 2];
    const int cntm = seg_s[s * 4 + 3];
    const int q0 = 8 * (j - start);
    const int mlo = q0 / wd;
    const int mhi = min((q0 + 7) / wd, cntm - 1);
    unsigned v = 0;
    for (int mm = mlo; mm <= mhi; ++mm) {
      const unsigned code = codes_s[tt * r + order_s[m0 + mm]];
      const int sh = mm * wd - q0;
      v |= sh >= 0 ? (code << sh) : (code >> (-sh));
    }
    dst[idx] = (unsigned char)(v & 0xffu);
  }
  if (MODE == KVC_MODE_CODEBOOK && tid < n) {
    __half* sdst = reinterpret_cast<__half*>(p.store + p.side_off[slot]) + a.t_base + t0;
    sdst[tid] = side_s[tid];
  }
  if (tid == 0) {
    if (nq > nside) atomicAdd(&p.counters[0], (unsigned long long)(nq - nside));
    if (nside) atomicAdd(&p.counters[1], (unsigned long long)nside);
    if (slot == 0) atomicAdd(&p.counters[2], (unsigned long long)n);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

template <class T>
size_t put(std::vector<uint8_t>& im, const T* src, size_t n) {
  const size_t off = align_up(im.size(), 256);
  im.resize(off + sizeof(T) * std::max<size_t>(n, 1), 0);
  if (n) std::memcpy(im.data() + off, src, sizeof(T) * n);
  return off;
}

uint16_t half_bits(float v) {
  const __half h = __float2half_rn(v);
  return __half_as_ushort(h);
}

using FetchKernel = void (*)(const Params, const FetchTc, const CUtensorMap, int64_t, int);

FetchKernel fetch_kernel_for(int mode, int out_dtype) {
  const bool bf = out_dtype == KVC_BF16;
  switch (mode) {
    case KVC_MODE_UNIFORM:
      return bf ? fetch_tc_kernel<KVC_MODE_UNIFORM, true> : fetch_tc_kernel<KVC_MODE_UNIFORM, false>;
    case KVC_MODE_GROUP:
      return bf ? fetch_tc_kernel<KVC_MODE_GROUP, true> : fetch_tc_kernel<KVC_MODE_GROUP, false>;
    default:
      return bf ? fetch_tc_kernel<KVC_MODE_CODEBOOK, true>
                : fetch_tc_kernel<KVC_MODE_CODEBOOK, false>;
  }
}

uint16_t bf16_bits(float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  return __bfloat16_as_ushort(h);
}

// Tensor-core append tables: three exact 16-bit pieces of V (scaled by
// 2^scale_exp for fp16 so that no piece is subnormal) and c = mean . V in double.
void prepare_append(const kvc_layer_desc& d, const Geo& g, std::vector<uint8_t>& image,
                    TcPlan& plan) {
  const int D = d.D, r = g.r, nb = g.nb;
  if (!(d.mode == KVC_MODE_UNIFORM || d.mode == KVC_MODE_CODEBOOK)) return;
  if (!(d.in_dtype == KVC_BF16 || d.in_dtype == KVC_F16) || d.heads_per_group != 1) return;
  int rpad = 16;
  while (rpad < r) rpad *= 2;
  if (!(D % 64 == 0 && D <= 256 && rpad <= 128)) return;
  const bool bf = d.in_dtype == KVC_BF16;
  const int npieces = bf ? 3 : 2;  // bf16: 3 x 8 bits; fp16 (scaled): 2 x 11 bits
  const int cols = std::max(32, 2 * rpad);
  size_t smem = 1024 + (size_t)(D / 64) * 16384 + (size_t)npieces * rpad * D * 2 +
                align_up((size_t)kTile * r, 16) + (size_t)kQueue * 12 + 4 * kTile * 4 +
                4 * (size_t)rpad * 4 + 256 * 4 + kTile * 2 + (size_t)rpad * 3 + 64;
  smem = std::max(smem, (size_t)(228 * 1024) / (512 / cols + 1) + 1024);
  if (smem > 226 * 1024) return;
  int scale_exp = 0;
  if (!bf) {
    float vmax = 0.f;
    for (size_t i = 0; i < (size_t)nb * D * r; ++i) vmax = std::max(vmax, std::fabs(d.V[i]));
    if (!(vmax > 0.f)) return;
    scale_exp = 14 - (int)std::ceil(std::log2((double)vmax));
  }
  const float scale = std::ldexp(1.f, scale_exp);
  std::vector<uint16_t> Bop((size_t)nb * npieces * rpad * D, 0);
  std::vector<double> c64((size_t)nb * r, 0.0);
  for (int b = 0; b < nb; ++b) {
    const float* V = d.V + (size_t)b * D * r;
    for (int k = 0; k < r; ++k) {
      double c = 0.0;
      for (int i = 0; i < D; ++i) {
        const float v = V[(size_t)i * r + k];
        if (d.mean) c += (double)d.mean[(size_t)b * D + i] * (double)v;
        float rest = v * scale;  // exact
        for (int pc = 0; pc < npieces; ++pc) {
          uint16_t bits;
          float got;
          if (bf) {
            bits = bf16_bits(rest);
            got = __bfloat162float(__ushort_as_bfloat16(bits));
          } else {
            bits = half_bits(rest);
            got = __half2float(__ushort_as_half(bits));
          }
          rest -= got;  // exact: the rounding error of a 16-bit rounding of an fp32 value
          const size_t idx = ((size_t)(pc * (rpad / 8) + k / 8) * (D / 8) + i / 8) * 64 +
                             (k % 8) * 8 + (i % 8);
          Bop[(size_t)b * npieces * rpad * D + idx] = bits;
        }
      }
      c64[(size_t)b * r + k] = c;
    }
  }
  plan.oAppB = put(image, Bop.data(), Bop.size());
  plan.oC64 = put(image, c64.data(), c64.size());
  plan.app_rpad = rpad;
  plan.app_cols = cols;
  plan.app_smem = smem;
  plan.app_bf16 = bf ? 1 : 0;
  plan.app_inv_scale = std::ldexp(1.f, -scale_exp);
  // Bound of the tensor-core accumulation per unit of ||x|| ||V_k||, from a
  // model of the accumulator: each K = 16 step adds 16 exact products and the
  // running sum after aligning them to the largest exponent and truncating,
  // at most one unit in the 24th bit of the running magnitude per addend
  // (17 per step, <= sum_i |x_i V_ik| <= ||x|| ||V_k||).  The PTX ISA states
  // no rounding rule for tcgen05.mma accumulation, so this is a model, held
  // against measurement: counters[3] reports the largest observed error over
  // the re-decided codes as a fraction of it.  fp16 pieces add their 2^-22
  // representation error.
  plan.app_gamma = (float)((17.0 * D / 16.0 + 2.0) * std::ldexp(1.0, -23) *
                               (1.0 + std::ldexp(1.0, -7)) +
                           (bf ? 0.0 : std::ldexp(1.0, -21)));
  plan.app_pieces = npieces;
  plan.append_ready = encoder() != nullptr;
  // the persistent warp-specialised kernel, where its tables and rings fit
  int pmax = 0;
  for (int b = 0; b < nb; ++b) pmax = std::max(pmax, g.P[b]);
  const size_t tab_bytes = append_ws_tab_bytes(rpad);
  std::vector<unsigned char> tab((size_t)nb * tab_bytes, 0);
  int max_chunks = 0;
  for (int b = 0; b < nb; ++b) max_chunks = std::max(max_chunks, append_ws_chunks(g, b));
  if (max_chunks > 32) max_chunks = -1;
  // the code staging row (append_ws_plan's)
  const int ks = std::max(max_chunks * 8, d.mode == KVC_MODE_CODEBOOK ? rpad : 0) + 8;
  for (int b = 0; b < nb && max_chunks > 0; ++b)
    if (append_ws_table(g, d, rpad, c64.data(), (double)plan.app_inv_scale, (double)plan.app_gamma,
                        ks, b, tab.data() + (size_t)b * tab_bytes) < 0)
      max_chunks = -1;
  AppendWsShape ws;
  const size_t wsm = max_chunks > 0 ? append_ws_plan(D, r, rpad, npieces, pmax, max_chunks, nb,
                                                    d.mode == KVC_MODE_CODEBOOK, &ws)
                                     : 0;
  if (wsm > 0 && plan.append_ready) {
    plan.oWsTab = put(image, tab.data(), tab.size());
    plan.ws = ws;
    plan.ws_smem = wsm;
    plan.ws_ready = true;
  }
}

// Group mode: tables of the tensor-core projection (kvc_group_proj.cu).  V is
// scaled by 2^se (largest entry near 2^14) and split into fp16 hi + lo, cut
// into [rpad][64] slices per head and 64-column box, each in core-matrix order.
// The latents' error bound, per unit of ||x - mean|| ||V_k|| (gamma):
//   the hi accumulator's chain of D terms per head, the accumulator model of
//   the uniform append (17 units in the 24th bit per K = 16 step), plus 2^-9
//   of it for the rest
//   accumulator (its terms are <= 2^-10 of the hi terms, twice as many);
//   the epilogue's fp32 sums, gamma_{hpg+2}; the pieces' representation
//   errors, 2^-22 each for x and V, and the dropped x_lo V_lo, 2^-22;
//   the rounding of x - mean, 2^-24;
// absolute parts where a piece is subnormal in fp16 (residual <= 2^-25 in
// scaled units): ex = 2^-24-sx sqrt(d_in) (times ||V_k||) and
// en = 2^-24-se sqrt(d_in) (times ||x - mean||).
constexpr size_t kZScratchBytes = size_t(32) << 20;

void prepare_group(const kvc_layer_desc& d, const Geo& g, std::vector<uint8_t>& image,
                   TcPlan& plan) {
  if (d.mode != KVC_MODE_GROUP || !(d.in_dtype == KVC_BF16 || d.in_dtype == KVC_F16)) return;
  const int D = d.D, hpg = d.heads_per_group, din = g.d_in, r = g.r, nb = g.nb;
  int rpad = 32;
  while (rpad < r) rpad *= 2;
  if (!(D % 64 == 0 && rpad <= 256) || encoder() == nullptr) return;
  int n_b = 0;
  const size_t smem = group_proj_smem(rpad, &n_b);
  if (smem == 0) return;
  float vmax = 0.f;
  for (size_t i = 0; i < (size_t)nb * din * r; ++i) vmax = std::max(vmax, std::fabs(d.V[i]));
  if (!(vmax > 0.f) || !std::isfinite(vmax)) return;
  const int se = 14 - (int)std::ceil(std::log2((double)vmax));
  const int sx = 6;  // x - mean up to 1023 in magnitude; larger tiles fall back
  const float vscale = std::ldexp(1.f, se);
  const int nbx = D / 64;
  std::vector<uint16_t> Bop((size_t)nb * din * 2 * rpad, 0);
  for (int b = 0; b < nb; ++b) {
    const float* V = d.V + (size_t)b * din * r;
    for (int i = 0; i < din; ++i) {
      const int h = i / D, bx = (i % D) / 64, kk = i % 64;
      for (int k = 0; k < r; ++k) {
        const float v = V[(size_t)i * r + k] * vscale;  // exact
        const uint16_t hi = half_bits(v);
        const uint16_t lo = half_bits(v - __half2float(__ushort_as_half(hi)));
        const size_t in_slice = ((size_t)(k / 8) * 8 + kk / 8) * 64 + (k % 8) * 8 + (kk % 8);
        for (int pc = 0; pc < 2; ++pc) {
          const size_t slice = (((size_t)b * hpg + h) * nbx + bx) * 2 + pc;
          Bop[slice * rpad * 64 + in_slice] = pc == 0 ? hi : lo;
        }
      }
    }
  }
  const double u = std::ldexp(1.0, -24);
  const double g_tc =
      (17.0 * D / 16.0 + 2.0) * std::ldexp(1.0, -23) * (1.0 + std::ldexp(1.0, -7));
  const double n_ep = hpg + 2;
  const double gamma = g_tc * (1.0 + std::ldexp(1.0, -9)) + n_ep * u / (1.0 - n_ep * u) +
                       3.0 * std::ldexp(1.0, -22) + u;
  const double root = std::sqrt((double)din);
  const int64_t per_tok = (int64_t)g.n_slots * r * 4;
  int64_t Tc = (int64_t)kZScratchBytes / per_tok / kTile * kTile;
  Tc = std::max<int64_t>(Tc, kTile);
  Tc = std::min<int64_t>(Tc, (d.capacity + kTile - 1) / kTile * kTile);
  plan.oGpB = put(image, Bop.data(), Bop.size());
  plan.gp_bf16 = d.in_dtype == KVC_BF16 ? 1 : 0;
  plan.gp_rpad = rpad;
  plan.gp_nb = n_b;
  plan.gp_smem = smem;
  plan.gp_xscale = std::ldexp(1.f, sx);
  plan.gp_zscale = std::ldexp(1.f, -(sx + se));
  plan.gp_gamma = (float)gamma;
  plan.gp_ex = (float)(std::ldexp(1.0, -24 - sx) * root);
  plan.gp_en = (float)(std::ldexp(1.0, -24 - se) * root);
  plan.gp_Tc = Tc;
  plan.gp_ready = true;
}

using AppendKernel = void (*)(const Params, const AppendTc, const CUtensorMap, const AppendArgs, int,
                              int);

template <int MODE, bool BF16>
AppendKernel append_v3_for(int rpad) {
  switch (rpad) {
    case 16: return append_tc_v3<MODE, BF16, 4>;
    case 32: return append_tc_v3<MODE, BF16, 8>;
    case 64: return append_tc_v3<MODE, BF16, 16>;
    default: return append_tc_v3<MODE, BF16, 32>;
  }
}

AppendKernel append_kernel_for(int mode, int bf16, int rpad) {
  if (mode == KVC_MODE_UNIFORM)
    return bf16 ? append_v3_for<KVC_MODE_UNIFORM, true>(rpad) : append_v3_for<KVC_MODE_UNIFORM, false>(rpad);
  return bf16 ? append_v3_for<KVC_MODE_CODEBOOK, true>(rpad) : append_v3_for<KVC_MODE_CODEBOOK, false>(rpad);
}

}  // namespace

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 1;
  return n;
}

kvc_status tc_prepare(const kvc_layer_desc& d, const Geo& g, std::vector<uint8_t>& image,
                      TcPlan& plan) {
  plan = TcPlan{};
  if (d.mode == KVC_MODE_INT8) return KVC_OK;
  prepare_append(d, g, image, plan);
  prepare_group(d, g, image, plan);
  const int D = d.D, din = g.d_in, r = g.r, nb = g.nb;
  // K layout: every packed segment starts on an 8-value chunk boundary, so a
  // chunk of A is decoded from consecutive bytes of one segment; the gaps are
  // zero columns of B.  koff[b][s] is segment s's first K position.
  int ktot = 0, pmax = 0;
  std::vector<int> koff((size_t)nb * kMaxSeg, 0);
  for (int b = 0; b < nb; ++b) {
    int k = 0;
    for (int s = 0; s < kMaxSeg; ++s) {
      koff[(size_t)b * kMaxSeg + s] = k;
      k += (g.seg[((size_t)b * kMaxSeg + s) * 4 + 3] + 7) / 8 * 8;
    }
    ktot = std::max(ktot, k);
    pmax = std::max(pmax, g.P[b]);
  }
  // Uniform mode folds the bias into the contraction: one more chunk of A
  // holds (1, 1, 0 ...) and the matching B columns hold the bias as fp16 hi + lo.
  const bool fold_bias = d.mode == KVC_MODE_UNIFORM;
  const int kones = ktot;
  if (fold_bias) ktot += 8;
  const int K = (ktot + 15) / 16 * 16;
  const int cols = D <= 64 ? 64 : (D <= 128 ? 128 : 256);
  size_t smem = 1024 + (size_t)(D / 64) * 16384 + (size_t)kTile * K * 2 + (size_t)D * K * 2 +
                (size_t)D * 4 + 256 * 4 + align_up((size_t)kTile * pmax + 16, 16) +
                align_up((size_t)kTile * g.side_bytes + 16, 16);
  // No more CTAs per SM than TMEM holds (512 columns), so allocation never waits.
  smem = std::max(smem, (size_t)(228 * 1024) / (512 / cols + 1) + 1024);
  if (!(D % 64 == 0 && D <= 256 && K >= 16 && K <= 256 && smem <= 226 * 1024 &&
        (d.mode != KVC_MODE_GROUP || d.group_size <= 32)))
    return KVC_OK;  // the CUDA-core kernels serve this shape

  // B = coef_k * V[:, k] at k's K position, coef = step (uniform) or 1; bias in fp64.
  // Chunk table: for each 8-value chunk of K, its first byte in the packed row,
  // its width and a valid bit (zero chunks are padding).
  std::vector<uint16_t> Bop((size_t)nb * din * K, 0);
  std::vector<float> bias((size_t)nb * din, 0.f);
  std::vector<uint32_t> chunks((size_t)nb * (K / 8), 0u);
  for (int b = 0; b < nb; ++b) {
    const float* V = d.V + (size_t)b * din * r;
    const int16_t* order = g.order.data() + (size_t)b * r;
    std::vector<int> kpos(g.n_kept[b]);
    int gbase = 0;  // group mode: groups of the earlier segments
    for (int s = 0; s < kMaxSeg; ++s) {
      const int32_t* e = &g.seg[((size_t)b * kMaxSeg + s) * 4];
      for (int m = 0; m < e[3]; ++m) kpos[e[2] + m] = koff[(size_t)b * kMaxSeg + s] + m;
      for (int ci = 0; ci * 8 < e[3]; ++ci) {
        const uint32_t gi =
            d.mode == KVC_MODE_GROUP ? (uint32_t)(gbase + (8 * ci) / d.group_size) : 0u;
        chunks[(size_t)b * (K / 8) + koff[(size_t)b * kMaxSeg + s] / 8 + ci] =
            (uint32_t)(e[0] + e[1] * ci) | ((uint32_t)e[1] << 16) | (gi << 20) | (1u << 31);
      }
      if (d.mode == KVC_MODE_GROUP) gbase += (e[3] + d.group_size - 1) / d.group_size;
    }
    for (int nrow = 0; nrow < din; ++nrow) {
      double acc = d.mean && d.mode != KVC_MODE_CODEBOOK ? (double)d.mean[(size_t)b * din + nrow] : 0.0;
      for (int kk = 0; kk < g.n_kept[b]; ++kk) {
        const int k = order[kk];
        const double v = V[(size_t)nrow * r + k];
        double coef = 1.0;
        if (d.mode == KVC_MODE_UNIFORM) {
          const int wdt = g.bits[(size_t)b * r + k];
          coef = d.qstep[(size_t)b * r + k];
          acc += ((double)d.qmin[(size_t)b * r + k] + (double)(1 << (wdt - 1)) * coef) * v;
        }
        const int kp = kpos[kk];
        const size_t idx = ((size_t)(nrow / 8) * (K / 8) + kp / 8) * 64 + (nrow % 8) * 8 + (kp % 8);
        Bop[(size_t)b * din * K + idx] = half_bits((float)(coef * v));
      }
      bias[(size_t)b * din + nrow] = (float)acc;
      if (fold_bias) {
        const uint16_t hi = half_bits((float)acc);
        const double rest = acc - (double)__half2float(__ushort_as_half(hi));
        for (int e = 0; e < 2; ++e) {
          const int kp = kones + e;
          const size_t idx = ((size_t)(nrow / 8) * (K / 8) + kp / 8) * 64 + (nrow % 8) * 8 + (kp % 8);
          Bop[(size_t)b * din * K + idx] = e == 0 ? hi : half_bits((float)rest);
        }
      }
    }
    if (fold_bias) chunks[(size_t)b * (K / 8) + kones / 8] = 1u << 30;  // the ones chunk
  }
  plan.bias_folded = fold_bias;
  {  // packed row bytes per slot (one load instead of basis_of -> P)
    std::vector<int32_t> slotP(g.n_slots);
    for (int sl = 0; sl < g.n_slots; ++sl) slotP[sl] = g.P[g.basis[sl]];
    plan.oSlotP = put(image, slotP.data(), slotP.size());
  }
  plan.oChunks = put(image, chunks.data(), chunks.size());
  plan.oFetchB = put(image, Bop.data(), Bop.size());
  plan.oBias = put(image, bias.data(), bias.size());
  plan.fetch_K = K;
  plan.fetch_cols = cols;
  plan.fetch_smem = smem;
  plan.fetch_ready = encoder() != nullptr;
  const bool grp = d.mode == KVC_MODE_GROUP;
  // group mode: chunks lie inside one group (group size a multiple of 8), at
  // most 256 groups (8 bits of the chunk entry)
  if ((d.heads_per_group == 1 || (grp && d.group_size % 8 == 0 && g.n_groups <= 256)) && K <= 256) {
    // the chunk table again, padded to 32 entries: one 128-byte bulk copy per tile
    std::vector<uint32_t> c32((size_t)nb * 32, 0u);
    for (int b = 0; b < nb; ++b)
      for (int c = 0; c < K / 8; ++c) c32[(size_t)b * 32 + c] = chunks[(size_t)b * (K / 8) + c];
    plan.oChunks32 = put(image, c32.data(), c32.size());
    FetchPipeShape sh;
    // group mode streams the heads' slices of B through two buffers
    const size_t ps = fetch_pipe_smem(d.mode, D, d.heads_per_group, K, g.side_bytes, pmax,
                                      grp ? 2 : nb, grp ? 2 : 3,
                                      d.mode == KVC_MODE_CODEBOOK ? d.cb_bits : 0, &sh);
    if (ps > 0 && d.mode == KVC_MODE_UNIFORM) {
      // every basis one segment of one width w in {1, 2, 4, 8}, whole 8-code
      // chunks from byte 0 and K position 0: chunk c is w bytes at c w
      int w0 = -1, n0 = -1;
      bool one = true;
      for (int b = 0; b < nb && one; ++b) {
        const int32_t* e = &g.seg[(size_t)b * kMaxSeg * 4];
        for (int s2 = 1; s2 < kMaxSeg; ++s2) one = one && g.seg[((size_t)b * kMaxSeg + s2) * 4 + 3] == 0;
        one = one && e[0] == 0 && e[3] > 0 && e[3] % 8 == 0 &&
              (e[1] == 1 || e[1] == 2 || e[1] == 4 || e[1] == 8) && (w0 < 0 || (e[1] == w0 && e[3] == n0));
        w0 = e[1];
        n0 = e[3];
      }
      if (one && n0 / 8 < K / 8) {
        sh.uni_w = w0;
        sh.uni_chunks = n0 / 8;
      }
    }
    if (ps > 0) {
      plan.pipe_ready = plan.fetch_ready;
      int cols_alloc = 32;  // TMEM allocations are powers of two
      while (cols_alloc < sh.a_col0 + sh.n_a * sh.a_cols) cols_alloc *= 2;
      plan.pipe_cols = cols_alloc;
      plan.pipe = sh;
      plan.pipe_smem = ps;
    }
  }
  return KVC_OK;
}

void tc_bind(TcPlan& plan, uint8_t* base) {
  if (plan.fetch_ready) {
    plan.fetchB = reinterpret_cast<const uint16_t*>(base + plan.oFetchB);
    plan.bias = reinterpret_cast<const float*>(base + plan.oBias);
    plan.chunks = reinterpret_cast<const uint32_t*>(base + plan.oChunks);
    plan.slotP = reinterpret_cast<const int32_t*>(base + plan.oSlotP);
    if (plan.pipe_ready) plan.chunks32 = reinterpret_cast<const uint32_t*>(base + plan.oChunks32);
  }
  if (plan.append_ready) {
    plan.appB = reinterpret_cast<const uint16_t*>(base + plan.oAppB);
    plan.c64 = reinterpret_cast<const double*>(base + plan.oC64);
    if (plan.ws_ready) plan.wsTab = reinterpret_cast<const unsigned char*>(base + plan.oWsTab);
  }
  if (plan.gp_ready) plan.gpB = reinterpret_cast<const uint16_t*>(base + plan.oGpB);
}

kvc_status tc_alloc(TcPlan& plan, int n_slots, int r) {
  if (!plan.gp_ready) return KVC_OK;
  const size_t zb = align_up((size_t)n_slots * plan.gp_Tc * r * sizeof(float), 256);
  const size_t ob = (size_t)n_slots * (plan.gp_Tc / kTile) * sizeof(int);
  void* mem = nullptr;
  if (cudaMalloc(&mem, zb + ob) != cudaSuccess) {
    cudaGetLastError();
    return set_error(KVC_ECUDA, "cudaMalloc(group projection scratch) failed");
  }
  plan.zbuf = static_cast<float*>(mem);
  plan.zovf = reinterpret_cast<int*>(static_cast<uint8_t*>(mem) + zb);
  return KVC_OK;
}

void tc_release(TcPlan& plan) {
  if (plan.zbuf) cudaFree(plan.zbuf);
  plan.zbuf = nullptr;
  plan.zovf = nullptr;
}

bool tc_fetch_ok(const TcPlan& plan, const Params&, const FetchArgs& f) {
  return plan.fetch_ready && (reinterpret_cast<uintptr_t>(f.out) % 16 == 0) && f.S > 0 &&
         f.S < (int64_t(1) << 31);
}

cudaError_t launch_fetch_tc(const TcPlan& plan, const Params& p, const FetchArgs& f,
                            cudaStream_t s, int* nk) {
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)p.D, (cuuint64_t)f.S, (cuuint64_t)p.B * p.H};
  const cuuint64_t strides[2] = {(cuuint64_t)p.D * 2, (cuuint64_t)f.ld_s * p.D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kTile, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult cr = encoder()(
      &map, p.out_dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
      3, f.out, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (plan.pipe_ready) return launch_fetch_pipe(plan, p, f, map, s, nk);
  FetchKernel kern = fetch_kernel_for(p.mode, p.out_dtype);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.fetch_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((f.S + kTile - 1) / kTile);
  const FetchTc t{plan.fetchB, plan.bias, plan.fetch_K, plan.fetch_cols};
  kern<<<(unsigned)(tiles * p.n_slots), kTile, plan.fetch_smem, s>>>(p, t, map, f.S, tiles);
  ++*nk;
  return cudaGetLastError();
}

bool tc_append_ok(const TcPlan& plan, const Params& p, const AppendArgs& a) {
  // TMA needs a 16-byte aligned base and strides that are multiples of 16 bytes
  return plan.append_ready && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) && a.T > 0 &&
         a.T < (int64_t(1) << 31) && a.st % 8 == 0 && a.sh % 8 == 0 && a.sb % 8 == 0 &&
         a.st >= p.D && (p.H == 1 || a.sh > 0) && (p.B == 1 || a.sb > 0);
}

// x as a 4D tensor map (D, tokens, heads, batch), boxes of 64 x 128 x 1 x 1
// with 128-byte swizzle.
CUresult encode_x_map(CUtensorMap* map, const Params& p, const AppendArgs& a, bool bf16) {
  const cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)a.T, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t strides[3] = {(cuuint64_t)a.st * 2,
                                 (cuuint64_t)(p.H > 1 ? a.sh : a.T * a.st) * 2,
                                 (cuuint64_t)(p.B > 1 ? a.sb : p.H * a.T * a.st) * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)kTile, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return encoder()(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   4, const_cast<void*>(a.x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool tc_group_ok(const TcPlan& plan, const Params& p, const AppendArgs& a) {
  // TMA needs a 16-byte aligned base and strides that are multiples of 16 bytes
  return plan.gp_ready && plan.zbuf && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) && a.T > 0 &&
         a.T < (int64_t(1) << 31) && a.st % 8 == 0 && a.sh % 8 == 0 && a.sb % 8 == 0 &&
         a.st >= p.D && (p.H == 1 || a.sh > 0) && (p.B == 1 || a.sb > 0);
}

// Chunks of gp_Tc tokens: the projection into the scratch, then the CUDA-core
// quantiser and packer reading it.
cudaError_t launch_append_group_tc(const TcPlan& plan, const Params& p, const AppendArgs& a,
                                   cudaStream_t s, int* nk) {
  for (int64_t c0 = 0; c0 < a.T; c0 += plan.gp_Tc) {
    AppendArgs ac = a;
    ac.x = static_cast<const uint16_t*>(a.x) + c0 * a.st;
    ac.T = std::min(plan.gp_Tc, a.T - c0);
    ac.t_base = a.t_base + c0;
    CUtensorMap map;
    if (encode_x_map(&map, p, ac, plan.gp_bf16 != 0) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    cudaError_t e = launch_group_proj(plan, p, ac, map, s, nk);
    if (e != cudaSuccess) return e;
    ZIn zin;
    zin.z = plan.zbuf;
    zin.ovf = plan.zovf;
    zin.Tc = plan.gp_Tc;
    zin.tps = (int)((ac.T + kTile - 1) / kTile);
    zin.gamma = plan.gp_gamma;
    zin.ex = plan.gp_ex;
    zin.en = plan.gp_en;
    e = launch_append_generic(p, ac, s, nk, &zin);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_append_tc(const TcPlan& plan, const Params& p, const AppendArgs& a,
                             uint64_t wait_ns, cudaStream_t s, int* nk) {
  CUtensorMap map;
  // dims: D, tokens, heads, batch (innermost first); strides of dims 1..3 in bytes
  const cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)a.T, (cuuint64_t)p.H, (cuuint64_t)p.B};
  const cuuint64_t strides[3] = {(cuuint64_t)a.st * 2,
                                 (cuuint64_t)(p.H > 1 ? a.sh : a.T * a.st) * 2,
                                 (cuuint64_t)(p.B > 1 ? a.sb : p.H * a.T * a.st) * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)kTile, 1, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult cr = encoder()(
      &map, plan.app_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
      const_cast<void*>(a.x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (plan.ws_ready) return launch_append_ws(plan, p, a, map, wait_ns, s, nk);
  AppendKernel kern = append_kernel_for(p.mode, plan.app_bf16, plan.app_rpad);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.app_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((a.T + kTile - 1) / kTile);
  const AppendTc t{plan.appB, plan.c64, plan.app_rpad, plan.app_cols, plan.app_inv_scale,
                   plan.app_gamma};
  kern<<<(unsigned)(tiles * p.n_slots), kV3, plan.app_smem, s>>>(p, t, map, a, tiles, plan.app_pieces);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
