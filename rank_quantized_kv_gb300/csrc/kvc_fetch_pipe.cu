// Pipelined persistent fetch for one head per slot (uniform and codebook modes).
//
// 512 threads per CTA, two CTAs per SM.  Each CTA owns a contiguous run of
// 128-token tiles (mostly of one slot, so the basis B stays in shared memory).
// One barrier per iteration i separates two phases:
//   all threads:  decode of tile i (packed rows -> A[i%2]), then the epilogue
//                 of tile i-1 (TMEM buffer (i-1)%2 -> staging (i-1)%2);
//   one thread:   tcgen05.mma of tile i into TMEM buffer i%2, TMA store of
//                 tile i-1, bulk prefetch of tile i+3's packed rows (a ring of
//                 four buffers keeps three tiles of rows in flight).
// so the MMA, the store and the prefetch of one iteration run under the next
// iteration's arithmetic.
//
// Decode works on 8-value chunks of K: every packed segment starts a chunk,
// so a chunk is w consecutive bytes of the row (w = the segment's width).
// A code c becomes fp16 through its bit pattern: 0x6400 | c is exactly
// 1024 + c, and one half2 subtraction of 1024 + 2^(w-1) gives c - 2^(w-1)
// exactly (uniform; the bias enters the contraction through a chunk of ones);
// codebook codes index an fp16 copy of the centroids, the fp16 norm is applied
// in the epilogue.  Epilogue: warp w reads TMEM lanes 32 (w % 4).. and a
// quarter of the columns.
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
constexpr int kStages = 4;  // packed-row buffers: tile i+3 is fetched while tile i decodes
constexpr uint64_t kWaitNs = 2000000000ull;

struct PipeArgs {
  const uint16_t* B;       // fp16 [nb][D][K] UMMA no-swizzle K-major
  const uint32_t* chunks;  // [nb][K/8]
  const int32_t* slotP;    // [n_slots] packed row bytes
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

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// 32 bits of the packed stream starting at byte a of `base` (4-byte aligned).
__device__ __forceinline__ uint32_t bytes_at(const unsigned char* base, int a) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(base) + (a >> 2);
  return __funnelshift_r(wp[0], wp[1], 8 * (a & 3));
}

// Eight centred codes of width w (uniform mode) as fp16 pairs.
__device__ __forceinline__ uint4 decode_uniform(const unsigned char* base, int a, int w) {
  const uint32_t lo = bytes_at(base, a);
  const uint32_t sub = 0x64006400u | ((1u << (w - 1)) * 0x10001u);  // 1024 + 2^(w-1), twice
  uint32_t o[4];
  if (w == 8) {
    const uint32_t hi = bytes_at(base, a + 4);
    o[0] = hsub2_bits(__byte_perm(lo, 0x64646464u, 0x5140), sub);
    o[1] = hsub2_bits(__byte_perm(lo, 0x64646464u, 0x5342), sub);
    o[2] = hsub2_bits(__byte_perm(hi, 0x64646464u, 0x5140), sub);
    o[3] = hsub2_bits(__byte_perm(hi, 0x64646464u, 0x5342), sub);
  } else if (w == 4) {
    const uint32_t L = lo & 0x0F0F0F0Fu, Hh = (lo >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t sel = (uint32_t)(q | (q << 4) | ((4 + q) << 8) | ((4 + q) << 12));
      o[q] = hsub2_bits((__byte_perm(L, Hh, sel) & 0x000F000Fu) | 0x64006400u, sub);
    }
  } else {
    const uint32_t mask = (1u << w) - 1u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t x = lo >> (2 * q * w);
      o[q] = hsub2_bits((x & mask) | ((x << (16 - w)) & (mask << 16)) | 0x64006400u, sub);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Eight codebook values (fp16 centroids) for codes of width w.
__device__ __forceinline__ uint4 decode_codebook(const unsigned char* base, int a, int w,
                                                 const uint16_t* cbh) {
  const uint32_t lo = bytes_at(base, a);
  const uint32_t hi = w > 4 ? bytes_at(base, a + 4) : 0u;
  const uint64_t bits = (uint64_t)lo | ((uint64_t)hi << 32);
  const uint32_t mask = (1u << w) - 1u;
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t c0 = (uint32_t)(bits >> (w * 2 * q)) & mask;
    const uint32_t c1 = (uint32_t)(bits >> (w * (2 * q + 1))) & mask;
    o[q] = (uint32_t)cbh[c0] | ((uint32_t)cbh[c1] << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int MODE, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 2)
    fetch_pipe_kernel(const Params p, const PipeArgs t, const __grid_constant__ CUtensorMap omap) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kStages], mma_bar[2];
  __shared__ int4 stage_info[kStages];  // per buffer: row bytes, basis, tokens of its tile
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int D = p.D, K = t.K, KC = K / 8, nbox = D / 64;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, row = quarter * 32 + lane;
  const int G = gridDim.x;
  const int first = (int)((int64_t)t.total_tiles * blockIdx.x / G);
  const int last = (int)((int64_t)t.total_tiles * (blockIdx.x + 1) / G);
  const int m = last - first;
  const int tps = t.tiles_per_slot;

  unsigned char* stage = smem;                              // 2 x nbox x 16 KB
  unsigned char* As = stage + 2 * nbox * 16384;             // 2 x [128 x K] fp16
  unsigned char* Bs = As + 2 * kTile * K * 2;               // [D x K] fp16
  uint16_t* cbh = reinterpret_cast<uint16_t*>(Bs + D * K * 2);  // [256] fp16 centroids
  uint32_t* chunk_s = reinterpret_cast<uint32_t*>(cbh + 256);    // [KC <= 32]
  float* norm_s = reinterpret_cast<float*>(chunk_s + 32);        // 2 x [128] codebook norms
  unsigned char* cbuf = reinterpret_cast<unsigned char*>(norm_s + 2 * kTile);  // kStages x cbuf
  const int side_off = t.cbuf - kTile * 2 - 16;
  const uint32_t sbo = (uint32_t)KC * 128;
  const uint32_t idesc = idesc_f16(kTile, D, 0);

  if (warp == 0) tmem_alloc(&tmem_base, t.cols);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    for (int i = 0; i < 2; ++i) mbar_init(&mma_bar[i], 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (MODE == KVC_MODE_CODEBOOK)
    for (int j = tid; j < p.cb_levels; j += kThreads)
      cbh[j] = __half_as_ushort(__float2half_rn(p.codebook[j]));

  // tile cursor: (slot, block) of tile `first`, advanced one tile per iteration
  int d_slot = first / tps, d_blk = first % tps;  // tile being decoded
  int e_slot = 0, e_blk = 0;                      // tile in the epilogue
  int f_slot = d_slot, f_blk = d_blk;             // next tile to prefetch
  // Slot tables for the next tile to prefetch, loaded one prefetch ahead so
  // their latency hides under an iteration (only thread 0 prefetches).
  struct SlotInfo { int P, beta; int64_t pay, side; };
  auto load_info = [&](int slot) {
    SlotInfo si{0, 0, 0, 0};
    if (slot < p.n_slots) {
      si.P = t.slotP[slot];
      si.beta = p.basis_of[slot];
      si.pay = p.pay_off[slot];
      si.side = p.side_off[slot];
    }
    return si;
  };
  SlotInfo f_info{0, 0, 0, 0};
  if (tid == 0) f_info = load_info(f_slot);
  auto prefetch = [&](int bi) {  // tile (f_slot, f_blk) into buffer bi; thread 0
    const int64_t t0 = (int64_t)f_blk * kTile;
    const int n = (int)min((int64_t)kTile, t.S - t0);
    const uint32_t cb = (uint32_t)((n * f_info.P + 15) & ~15);
    const uint32_t sbb = (uint32_t)((n * p.side_bytes + 15) & ~15);
    unsigned char* dst = cbuf + bi * t.cbuf;
    stage_info[bi] = make_int4(f_info.P, f_info.beta, n, 0);
    mbar_arrive_expect_tx(&full_bar[bi], cb + sbb);
    if (cb) bulk_load(dst, p.store + f_info.pay + t0 * f_info.P, cb, &full_bar[bi]);
    if (sbb) bulk_load(dst + side_off, p.store + f_info.side + t0 * p.side_bytes, sbb, &full_bar[bi]);
  };
  auto advance_f = [&]() {
    if (++f_blk == tps) {
      f_blk = 0;
      ++f_slot;
      if (tid == 0) f_info = load_info(f_slot);
    }
  };
  for (int j = 0; j < kStages - 1 && j < m; ++j) {
    if (tid == 0) prefetch(j);
    advance_f();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr0 = tmem_base;

  int cur_beta = -1;
  for (int it = 0; it <= m; ++it) {
    const int buf = it & 1, pb = buf ^ 1;
    // ---------------- phase A: decode of tile it, then the epilogue of tile it-1
    // (decoding first gives MMA(it-1), issued just before, time to finish)
    if (it < m) {
      const int stg_in = it % kStages;
      const int4 info = stage_info[stg_in];  // written with the prefetch (barriers since)
      const int P = info.x, beta = info.y, n = info.z;
      if (beta != cur_beta) {
        // MMA(it-1) is the last reader of B
        if (it >= 1 && !mbar_wait_bounded(&mma_bar[pb], ((it - 1) >> 1) & 1, kWaitNs))
          abort_flag = 1;
        const uint4* bsrc = reinterpret_cast<const uint4*>(t.B + (size_t)beta * D * K);
        for (int i = tid; i < D * K * 2 / 16; i += kThreads)
          reinterpret_cast<uint4*>(Bs)[i] = bsrc[i];
        if (tid < KC) chunk_s[tid] = t.chunks[(size_t)beta * KC + tid];
        cur_beta = beta;
        __syncthreads();  // chunk_s before decode (uniform branch: cur_beta is CTA-wide)
      }
      if (!mbar_wait_bounded(&full_bar[stg_in], (it / kStages) & 1, kWaitNs)) abort_flag = 1;
      const unsigned char* rows = cbuf + stg_in * t.cbuf;
      unsigned char* A = As + buf * kTile * K * 2;
      for (int item = tid; item < kTile * KC; item += kThreads) {
        const int tt = item & (kTile - 1), c = item >> 7;
        const uint32_t ent = chunk_s[c];
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tt < n) {
          if (ent >> 31) {
            const int a = tt * P + (int)(ent & 0xffffu), w = (int)((ent >> 16) & 0xfu);
            v = MODE == KVC_MODE_UNIFORM ? decode_uniform(rows, a, w)
                                         : decode_codebook(rows, a, w, cbh);
          } else if (ent >> 30) {
            v.x = 0x3C003C00u;  // (1, 1): the two bias columns of B
          }
        }
        *reinterpret_cast<uint4*>(A + (tt >> 3) * sbo + c * 128 + (tt & 7) * 16) = v;
        if (MODE == KVC_MODE_CODEBOOK && c == 0)  // kept until this tile's epilogue
          norm_s[buf * kTile + tt] =
              tt < n ? __half2float(__ushort_as_half(
                           reinterpret_cast<const uint16_t*>(rows + side_off)[tt]))
                     : 0.f;
      }
    }
    if (it >= 1) {
      if (!mbar_wait_bounded(&mma_bar[pb], ((it - 1) >> 1) & 1, kWaitNs)) abort_flag = 1;
      tc_fence_after();
      const float nrm = MODE == KVC_MODE_CODEBOOK ? norm_s[pb * kTile + row] : 1.f;
      const uint32_t lane_addr = taddr0 + pb * D + ((uint32_t)(quarter * 32) << 16);
      unsigned char* stg = stage + pb * nbox * 16384;
      for (int c32 = warp >> 2; c32 < D / 32; c32 += kThreads / 128) {
        uint32_t r[32];
        tmem_ld32(lane_addr + c32 * 32, r);
        tmem_wait_ld();
        unsigned char* dst = stg + (c32 >> 1) * 16384 + row * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float x[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            x[e] = MODE == KVC_MODE_CODEBOOK ? __uint_as_float(r[q * 8 + e]) * nrm
                                             : __uint_as_float(r[q * 8 + e]);
          const int c16 = (c32 & 1) * 4 + q;
          *reinterpret_cast<uint4*>(dst + ((c16 ^ (row & 7)) << 4)) =
              make_uint4(pack_out(x[0], x[1], OUT_BF16), pack_out(x[2], x[3], OUT_BF16),
                         pack_out(x[4], x[5], OUT_BF16), pack_out(x[6], x[7], OUT_BF16));
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    if (tid == 0) bulk_wait_read0();  // the store of tile it-2 has left staging buf
    __syncthreads();
    if (abort_flag) break;
    // ---------------- phase B: one thread issues the asynchronous work
    if (tid == 0) {
      tc_fence_after();
      if (it < m) {
        const uint32_t a0 = smem_u32(As + buf * kTile * K * 2), b0 = smem_u32(Bs);
        for (int ks = 0; ks < K / 16; ++ks)
          umma_f16(taddr0 + buf * D, desc_kmajor_noswizzle(a0 + ks * 256, 128, sbo),
                   desc_kmajor_noswizzle(b0 + ks * 256, 128, sbo), idesc, ks > 0 ? 1u : 0u);
        umma_commit(&mma_bar[buf]);
      }
      if (it >= 1) {  // one head per slot: the slot is the tensor map's (b, h) index
        unsigned char* stg = stage + pb * nbox * 16384;
        for (int bx = 0; bx < nbox; ++bx)
          tma_store_3d(&omap, stg + bx * 16384, bx * 64, e_blk * kTile, e_slot);
        bulk_commit();
      }
      if (it + kStages - 1 < m)  // its buffer held tile it-1, decoded last iteration
        prefetch((it + kStages - 1) % kStages);
    }
    if (it + kStages - 1 < m) advance_f();
    // advance the cursors
    e_slot = d_slot;
    e_blk = d_blk;
    if (++d_blk == tps) { d_blk = 0; ++d_slot; }
  }
  if (abort_flag && tid == 0) atomicCAS(p.err, 0, kErrTimeout);
  if (tid == 0) bulk_wait_read0();  // the stores may finish after the CTA: staging is read
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
  const PipeArgs t{plan.fetchB, plan.chunks, plan.slotP, plan.fetch_K, plan.pipe_cols, plan.pipe_cbuf,
                   f.S, tiles, total};
  k<<<(unsigned)grid, kThreads, plan.pipe_smem, s>>>(p, t, map);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
