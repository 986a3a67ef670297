// Pipelined persistent fetch for one head per slot (uniform and codebook modes).
//
// 512 threads per CTA, two CTAs per SM.  Each CTA owns a contiguous run of
// 128-token tiles (mostly of one slot, so the basis B stays in shared memory)
// and overlaps, in iteration i,
//   bulk prefetch of tile i+1's packed rows   |  decode of tile i into A[i%2]
//   tcgen05.mma of tile i into TMEM buffer i%2 |  epilogue of tile i-1 from the other
//   TMA store of tile i-1 from staging (i-1)%2, still draining during tile i.
//
// Decode works on 8-value chunks of K: every packed segment starts a chunk,
// so a chunk is w consecutive bytes of the row (w = the segment's width).
// A code c becomes fp16 through its bit pattern: 0x6400 | c is exactly
// 1024 + c, and one half2 subtraction of 1024 + 2^(w-1) gives c - 2^(w-1)
// exactly (uniform); codebook codes index an fp16 copy of the centroids.
// Epilogue: warp w reads TMEM lanes 32 (w % 4).. and a quarter of the columns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kvc_sm100.cuh"
#include "kvc_tc.h"

namespace kvc {

using namespace sm100;

namespace {

constexpr int kTile = 128;
constexpr int kThreads = 512;
constexpr uint64_t kWaitNs = 2000000000ull;

struct PipeArgs {
  const uint16_t* B;       // fp16 [nb][D][K] UMMA no-swizzle K-major
  const float* bias;       // [nb][D]
  const uint32_t* chunks;  // [nb][K/8]
  int K, cols, cbuf;
  int64_t S;
  int tiles_per_slot, total_tiles;
};

__device__ __forceinline__ uint32_t pack_out(float a, float b, bool bf) {
  if (bf) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Eight fp16 values of one A chunk from the packed row.
template <int MODE>
__device__ __forceinline__ uint4 decode_chunk(const unsigned char* row, uint32_t ent,
                                              const uint16_t* cbh) {
  if (!(ent >> 31)) return make_uint4(0u, 0u, 0u, 0u);
  const int off = (int)(ent & 0xffffu), w = (int)((ent >> 16) & 0xfu);
  uint64_t bits = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < w) bits |= (uint64_t)row[off + i] << (8 * i);
  const uint32_t mask = (1u << w) - 1u;
  uint32_t o[4];
  if (MODE == KVC_MODE_UNIFORM) {
    const uint32_t bias16 = 0x6400u | (1u << (w - 1));     // fp16(1024 + 2^(w-1))
    const __half2 sub = __halves2half2(__ushort_as_half((uint16_t)bias16),
                                       __ushort_as_half((uint16_t)bias16));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t c0 = (uint32_t)(bits >> (w * (2 * q))) & mask;
      const uint32_t c1 = (uint32_t)(bits >> (w * (2 * q + 1))) & mask;
      const uint32_t hv = (0x6400u | c0) | ((0x6400u | c1) << 16);
      const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&hv), sub);
      o[q] = *reinterpret_cast<const uint32_t*>(&v);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t c0 = (uint32_t)(bits >> (w * (2 * q))) & mask;
      const uint32_t c1 = (uint32_t)(bits >> (w * (2 * q + 1))) & mask;
      o[q] = (uint32_t)cbh[c0] | ((uint32_t)cbh[c1] << 16);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int MODE, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 2)
    fetch_pipe_kernel(const Params p, const PipeArgs t, const __grid_constant__ CUtensorMap omap) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[2], mma_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int D = p.D, K = t.K, KC = K / 8, nbox = D / 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int first = (int)((int64_t)t.total_tiles * blockIdx.x / G);
  const int last = (int)((int64_t)t.total_tiles * (blockIdx.x + 1) / G);
  const int m = last - first;

  unsigned char* stage = smem;                              // 2 x nbox x 16 KB
  unsigned char* As = stage + 2 * nbox * 16384;             // 2 x [128 x K] fp16
  unsigned char* Bs = As + 2 * kTile * K * 2;               // [D x K] fp16
  float* bias_s = reinterpret_cast<float*>(Bs + D * K * 2);   // 2 x [D]
  uint16_t* cbh = reinterpret_cast<uint16_t*>(bias_s + 2 * D);  // [256] fp16 centroids
  uint32_t* chunk_s = reinterpret_cast<uint32_t*>(cbh + 256);    // [KC <= 32]
  float* norm_s = reinterpret_cast<float*>(chunk_s + 32);        // 2 x [128] codebook norms
  unsigned char* cbuf = reinterpret_cast<unsigned char*>(norm_s + 2 * kTile);  // 2 x cbuf
  const int side_off = t.cbuf - kTile * 2 - 16;              // codebook norms in a buffer
  const uint32_t sbo = (uint32_t)KC * 128;
  const uint32_t idesc = idesc_f16(kTile, D, 0);

  if (warp == 0) tmem_alloc(&tmem_base, t.cols);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&mma_bar[i], 1);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  if (MODE == KVC_MODE_CODEBOOK)
    for (int j = tid; j < p.cb_levels; j += kThreads)
      cbh[j] = __half_as_ushort(__float2half_rn(p.codebook[j]));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr0 = tmem_base;

  auto prefetch = [&](int tile, int bi) {
    const int slot = tile / t.tiles_per_slot;
    const int64_t t0 = (int64_t)(tile % t.tiles_per_slot) * kTile;
    const int n = (int)min((int64_t)kTile, t.S - t0);
    const int P = p.P[p.basis_of[slot]];
    const uint32_t cb = (uint32_t)((n * P + 15) & ~15);
    const uint32_t sbb = (uint32_t)((n * p.side_bytes + 15) & ~15);
    unsigned char* dst = cbuf + bi * t.cbuf;
    mbar_arrive_expect_tx(&full_bar[bi], cb + sbb);
    if (cb) bulk_load(dst, p.store + p.pay_off[slot] + t0 * P, cb, &full_bar[bi]);
    if (sbb)
      bulk_load(dst + side_off, p.store + p.side_off[slot] + t0 * p.side_bytes, sbb, &full_bar[bi]);
  };

  if (tid == 0 && m > 0) prefetch(first, 0);
  int cur_beta = -1;
  for (int it = 0; it <= m; ++it) {
    const int buf = it & 1;
    if (it < m) {
      const int tile = first + it;
      const int slot = tile / t.tiles_per_slot;
      const int64_t t0 = (int64_t)(tile % t.tiles_per_slot) * kTile;
      const int n = (int)min((int64_t)kTile, t.S - t0);
      const int beta = p.basis_of[slot];
      const int P = p.P[beta];
      if (tid == 0 && it + 1 < m) prefetch(first + it + 1, buf ^ 1);
      if (beta != cur_beta) {  // the previous MMA must be done with B
        if (it > 0 && !mbar_wait_bounded(&mma_bar[buf ^ 1], ((it - 1) >> 1) & 1, kWaitNs))
          abort_flag = 1;
        const uint4* bsrc = reinterpret_cast<const uint4*>(t.B + (size_t)beta * D * K);
        for (int i = tid; i < D * K * 2 / 16; i += kThreads)
          reinterpret_cast<uint4*>(Bs)[i] = bsrc[i];
        if (tid < KC) chunk_s[tid] = t.chunks[(size_t)beta * KC + tid];
        cur_beta = beta;
        __syncthreads();  // chunk_s before decode
      }
      if (MODE != KVC_MODE_CODEBOOK)
        for (int c = tid; c < D; c += kThreads) bias_s[buf * D + c] = t.bias[(size_t)beta * D + c];
      if (!mbar_wait_bounded(&full_bar[buf], (it >> 1) & 1, kWaitNs)) abort_flag = 1;
      const unsigned char* rows = cbuf + buf * t.cbuf;
      unsigned char* A = As + buf * kTile * K * 2;
      for (int item = tid; item < kTile * KC; item += kThreads) {
        const int tt = item & (kTile - 1), c = item >> 7;
        const uint4 v = tt < n ? decode_chunk<MODE>(rows + tt * P, chunk_s[c], cbh)
                               : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(A + (tt >> 3) * sbo + c * 128 + (tt & 7) * 16) = v;
        if (MODE == KVC_MODE_CODEBOOK && c == 0)  // kept until this tile's epilogue
          norm_s[buf * kTile + tt] =
              tt < n ? __half2float(__ushort_as_half(
                           reinterpret_cast<const uint16_t*>(rows + side_off)[tt]))
                     : 0.f;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (abort_flag) break;
      if (tid == 0) {
        tc_fence_after();
        const uint32_t a0 = smem_u32(A), b0 = smem_u32(Bs);
        for (int ks = 0; ks < K / 16; ++ks)
          umma_f16(taddr0 + buf * D, desc_kmajor_noswizzle(a0 + ks * 256, 128, sbo),
                   desc_kmajor_noswizzle(b0 + ks * 256, 128, sbo), idesc, ks > 0 ? 1u : 0u);
        umma_commit(&mma_bar[buf]);
      }
    }
    if (it >= 1) {
      const int prev = it - 1, pb = prev & 1;
      const int tile = first + prev;
      const int slot = tile / t.tiles_per_slot;
      const int64_t t0 = (int64_t)(tile % t.tiles_per_slot) * kTile;
      const int b = slot / p.H, h = slot % p.H;
      if (!mbar_wait_bounded(&mma_bar[pb], (prev >> 1) & 1, kWaitNs)) abort_flag = 1;
      tc_fence_after();
      if (tid == 0) bulk_wait_read1();  // staging pb (two tiles ago) has been read
      __syncthreads();
      if (abort_flag) break;
      const int quarter = warp & 3, row = quarter * 32 + lane;
      const float nrm = MODE == KVC_MODE_CODEBOOK ? norm_s[pb * kTile + row] : 1.f;
      const uint32_t lane_addr = taddr0 + pb * D + ((uint32_t)(quarter * 32) << 16);
      unsigned char* stg = stage + pb * nbox * 16384;
      for (int c32 = warp >> 2; c32 < D / 32; c32 += kThreads / 128) {
        uint32_t r[32];
        tmem_ld32(lane_addr + c32 * 32, r);
        tmem_wait_ld();
        unsigned char* dst = stg + (c32 >> 1) * 16384 + row * 128;
        const float4* bv = reinterpret_cast<const float4*>(bias_s + pb * D + c32 * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(r[q * 8 + e]);
          if (MODE == KVC_MODE_CODEBOOK) {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= nrm;
          } else {
            const float4 b0 = bv[2 * q], b1 = bv[2 * q + 1];
            x[0] += b0.x; x[1] += b0.y; x[2] += b0.z; x[3] += b0.w;
            x[4] += b1.x; x[5] += b1.y; x[6] += b1.z; x[7] += b1.w;
          }
          const int c16 = (c32 & 1) * 4 + q;
          *reinterpret_cast<uint4*>(dst + ((c16 ^ (row & 7)) << 4)) =
              make_uint4(pack_out(x[0], x[1], OUT_BF16), pack_out(x[2], x[3], OUT_BF16),
                         pack_out(x[4], x[5], OUT_BF16), pack_out(x[6], x[7], OUT_BF16));
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        for (int bx = 0; bx < nbox; ++bx)
          tma_store_3d(&omap, stg + bx * 16384, bx * 64, (int)t0, b * p.H + h);
        bulk_commit();
      }
    }
  }
  if (abort_flag && tid == 0) atomicCAS(p.err, 0, kErrTimeout);
  if (tid == 0) bulk_wait0();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(taddr0, t.cols);
  }
}

using PipeKernel = void (*)(const Params, const PipeArgs, const CUtensorMap);

PipeKernel pipe_kernel_for(int mode, int out_dtype) {
  const bool bf = out_dtype == KVC_BF16;
  if (mode == KVC_MODE_UNIFORM)
    return bf ? fetch_pipe_kernel<KVC_MODE_UNIFORM, true> : fetch_pipe_kernel<KVC_MODE_UNIFORM, false>;
  return bf ? fetch_pipe_kernel<KVC_MODE_CODEBOOK, true> : fetch_pipe_kernel<KVC_MODE_CODEBOOK, false>;
}

}  // namespace

cudaError_t launch_fetch_pipe(const TcPlan& plan, const Params& p, const FetchArgs& f,
                              const CUtensorMap& map, cudaStream_t s, int* nk) {
  PipeKernel k = pipe_kernel_for(p.mode, p.out_dtype);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)plan.pipe_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((f.S + kTile - 1) / kTile);
  const int total = tiles * p.n_slots;
  const int grid = std::min(total, sm_count() * plan.pipe_ctas_per_sm);
  const PipeArgs t{plan.fetchB, plan.bias, plan.chunks, plan.fetch_K, plan.pipe_cols,
                   plan.pipe_cbuf, f.S, tiles, total};
  k<<<(unsigned)grid, kThreads, plan.pipe_smem, s>>>(p, t, map);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
