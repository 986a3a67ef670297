// Warp-specialised persistent fetch for one head per slot (uniform and
// codebook modes): x_hat = A B^T (+ bias folded into B), A the decoded codes.
//
// One CTA per SM walks a contiguous run of 128-token tiles.  Four roles run
// concurrently and hand tiles on through mbarrier rings, with no CTA-wide
// barrier in the loop:
//   producer (one thread)  bulk-copies each tile's packed rows, side words and
//                          its basis' chunk table into a ring of row stages,
//                          and the basis B into one of (up to) two B buffers
//                          when the basis changes;
//   decoders (8 warps)     turn a row stage into the fp16 A operand, written
//                          straight into TMEM (a ring of A buffers there);
//   MMA (one thread)       issues tcgen05.mma of A (from TMEM) against B (from
//                          shared memory) into one of several TMEM accumulators;
//   epilogue (8 warps)     read an accumulator, convert to the output type,
//                          stage it swizzled in shared memory, and one thread
//                          TMA-stores the tile.  Up to four staging buffers keep
//                          three tiles of stores in flight per SM: HBM write
//                          bandwidth needs that many bytes outstanding.
// Every ring slot has a full and an empty barrier; each wait is bounded in
// time and a time-out sets the layer's error word and unwinds.
//
// Shared-memory bandwidth, not arithmetic, bounds this kernel: per tile the
// staging write and the TMA store's read move 2 x 32 KB (D = 128, fp16) and
// the MMA reads B.  Keeping A in TMEM takes its write and its read by the
// tensor core (2 x 16 KB at K = 64) off the shared-memory pipe.
//
// Decode works on 8-value chunks of K: every packed segment starts a chunk,
// so a chunk is w consecutive bytes of the row (w = the segment's width).
// A code c becomes fp16 through its bit pattern: 0x6400 | c is exactly
// 1024 + c, and one half2 subtraction of 1024 + 2^(w-1) gives c - 2^(w-1)
// exactly (uniform; the bias enters the contraction through a chunk of ones);
// codebook codes index an fp16 copy of the centroids, and the epilogue scales
// by the fp16 norm.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kvc_sm100.cuh"
#include "kvc_tc.h"

namespace kvc {

using namespace sm100;

namespace {

constexpr int kTile = 128;
constexpr int kEpiWarps = 8;   // warps 0..7: two per TMEM lane quarter
constexpr int kDecWarps = 8;   // warps 8..15
constexpr int kProdWarp = kEpiWarps + kDecWarps;
constexpr int kMmaWarp = kProdWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kMaxRS = 8, kMaxAS = 3, kMaxTS = 4, kMaxSS = 4;
constexpr int kNormRing = 8;   // >= A buffers + accumulators (see the decoders)
static_assert(kNormRing >= kMaxAS + kMaxTS, "norm ring shorter than the pipeline");
constexpr int kEpiBar = 1;     // named barriers 1, 2: the epilogue groups
constexpr uint64_t kWaitNs = 2000000000ull;

struct PipeArgs {
  const uint16_t* B;       // fp16 [nb][D_in][K] UMMA no-swizzle K-major (D_in = hpg D)
  const float* bias;       // fp32 [nb][D_in] (group mode: added in the epilogue)
  const uint32_t* chunks;  // [nb][32] chunk table, 128 bytes per basis
  const int32_t* slotP;    // [n_slots] packed row bytes
  int K, cols;             // K; TMEM columns allocated
  int n_acc, n_a, n_rs;    // accumulators, A buffers, row stages
  int a_col0, a_cols;      // TMEM column of the first A buffer; columns per A buffer
  int n_stg, n_b;          // staging buffers, B buffers (1 when every slot shares a basis)
  int rs_bytes;            // bytes of one row stage
  int cb_rep;              // codebook: 8-byte slots of the lane-replicated pair table (0: none)
  int uni_w, uni_chunks;   // uniform rows of one width from byte 0 (0: by the chunk table)
  int64_t S;
  int tiles_per_slot, total_tiles;
};

// Position in a ring of n buffers: the buffer of the current use and the
// parity of its barriers' phase; next() moves on one use.
struct Ring {
  int n, slot;
  uint32_t phase;
  __device__ explicit Ring(int n_) : n(n_), slot(0), phase(0u) {}
  __device__ void next() {
    if (++slot == n) { slot = 0; phase ^= 1u; }
  }
};

__device__ __forceinline__ uint32_t pack_out(float a, float b, bool bf) {
  if (bf) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b) {
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// The 64 bits of the packed stream starting at byte a of `base` (4-byte
// aligned buffer), as two words.
__device__ __forceinline__ uint2 bits_at(const unsigned char* base, int a) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(base) + (a >> 2);
  const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
  const uint32_t sh = 8 * (a & 3);
  return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// Eight centred codes of width w (uniform mode) as fp16 pairs.
__device__ __forceinline__ uint4 decode_uniform(uint2 b, int w) {
  const uint32_t lo = b.x;
  const uint32_t sub = 0x64006400u | ((1u << (w - 1)) * 0x10001u);  // 1024 + 2^(w-1), twice
  uint32_t o[4];
  if (w == 8) {
    o[0] = hsub2_bits(__byte_perm(lo, 0x64646464u, 0x5140), sub);
    o[1] = hsub2_bits(__byte_perm(lo, 0x64646464u, 0x5342), sub);
    o[2] = hsub2_bits(__byte_perm(b.y, 0x64646464u, 0x5140), sub);
    o[3] = hsub2_bits(__byte_perm(b.y, 0x64646464u, 0x5342), sub);
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
__device__ __forceinline__ uint4 decode_codebook(uint2 b, int w, const uint16_t* cbh) {
  const uint64_t bits = (uint64_t)b.x | ((uint64_t)b.y << 32);
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

// The same for widths w <= 4 through a table of code pairs: entry c0 | c1 << w
// holds the fp16 centroids of (c0, c1) as one half2 word.
__device__ __forceinline__ uint4 decode_codebook_pairs(uint2 b, int w, const uint32_t* cb2) {
  const uint64_t bits = (uint64_t)b.x | ((uint64_t)b.y << 32);
  const uint32_t mask2 = (1u << (2 * w)) - 1u;
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) o[q] = cb2[(uint32_t)(bits >> (2 * w * q)) & mask2];
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 2W bits at bit offset `off` of the words w (compile-time offsets).
template <int W>
__device__ __forceinline__ uint32_t pair_field(const uint32_t (&w)[W], int off) {
  const int i = off >> 5, sh = off & 31;
  const uint32_t x =
      sh + 2 * W <= 32 ? w[i] >> sh : __funnelshift_r(w[i], w[i + 1 < W ? i + 1 : W - 1], sh);
  return x & ((1u << (2 * W)) - 1u);
}

// Codebook rows of W-bit codes (W <= 3, one segment from byte 0): the codes
// [k0, k0 + 32 nblk) of one token's row in blocks of 32 (W aligned words),
// two codes per lookup in a table of pairs replicated once per lane (lane l
// reads column l: no bank conflicts), each chunk of 8 written to TMEM as 4
// columns.
template <int W>
__device__ __forceinline__ void decode_cb_rows(const unsigned char* row, bool live, int k0,
                                               int nblk, const uint32_t* cbr, uint32_t a_tm) {
  for (int b = 0; b < nblk; ++b) {
    const int kb = k0 + 32 * b;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(row + kb / 8 * W);
    uint32_t w[W];
#pragma unroll
    for (int i = 0; i < W; ++i) w[i] = live ? src[i] : 0u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (live) {
        const uint32_t* cl = cbr + (threadIdx.x & 31);
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = cl[pair_field<W>(w, W * (8 * c + 2 * i)) * 32];
        v = make_uint4(o[0], o[1], o[2], o[3]);
      }
      tmem_st4(a_tm + (kb / 8 + c) * 4, v);  // chunk kb / 8 + c: K positions 8 (kb / 8 + c) ..
    }
  }
}

template <int MODE, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fetch_pipe_kernel(const Params p, const PipeArgs t, const __grid_constant__ CUtensorMap omap) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t row_full[kMaxRS], row_empty[kMaxRS];
  __shared__ uint64_t a_full[kMaxAS], a_empty[kMaxAS];
  __shared__ uint64_t acc_full[kMaxTS], acc_empty[kMaxTS];
  __shared__ uint64_t b_full[2], b_empty[2], done_bar;
  __shared__ uint64_t norm_full[kNormRing];  // codebook norms of a tile decoded
  __shared__ int4 stage_hdr[kMaxRS];  // per row stage: row bytes, tokens, B buffer | first use << 1
  __shared__ int a_info[kMaxAS];      // per A buffer: B buffer | first use << 1
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;

  constexpr bool GRP = MODE == KVC_MODE_GROUP;  // a slot is a head group: A once, hpg heads of B
  const int D = p.D, K = t.K, KC = K / 8, nbox = D / 64;
  const int HPG = GRP ? p.hpg : 1;
  const int RS = t.n_rs, AS = t.n_a, TS = t.n_acc, SS = t.n_stg, NB = t.n_b;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int first = (int)((int64_t)t.total_tiles * blockIdx.x / G);
  const int m = (int)((int64_t)t.total_tiles * (blockIdx.x + 1) / G) - first;
  const int tps = t.tiles_per_slot;
  const size_t b_bytes = (size_t)D * K * 2;

  unsigned char* stage = smem;                                  // SS x nbox x 16 KB
  unsigned char* Bs = stage + SS * nbox * 16384;                // NB x [D x K] fp16
  unsigned char* rs = Bs + NB * b_bytes;                        // RS x row stage
  // after the row stages: codebook mode the fp16 centroids [256], the norm
  // ring [kNormRing][128] and the centroid pairs [256]; group mode the
  // epilogue groups' mean cache
  uint16_t* cbh = reinterpret_cast<uint16_t*>(rs + (size_t)RS * t.rs_bytes);
  float* norm_ring = reinterpret_cast<float*>(cbh + 256);
  uint32_t* cb2 = reinterpret_cast<uint32_t*>(norm_ring + kNormRing * kTile);  // [256] pairs
  uint32_t* cbr = cb2 + 256;  // [L^2][32]: each pair of centroids once per lane
  float* mean_c = reinterpret_cast<float*>(rs + (size_t)RS * t.rs_bytes);  // [hpg][D]
  // a row stage: [0, 128) chunk table, then the packed rows, then the side words
  const int side_off = t.rs_bytes - (int)(((size_t)kTile * p.side_bytes + 16 + 15) & ~size_t(15));

  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base, t.cols);
  }
  if (tid == 0) {
    for (int i = 0; i < RS; ++i) { mbar_init(&row_full[i], 1); mbar_init(&row_empty[i], kDecWarps); }
    for (int i = 0; i < AS; ++i) { mbar_init(&a_full[i], kDecWarps); mbar_init(&a_empty[i], 1); }
    for (int i = 0; i < TS; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], kEpiWarps); }
    for (int i = 0; i < 2; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
    mbar_init(&done_bar, 1);
    for (int i = 0; i < kNormRing; ++i) mbar_init(&norm_full[i], kDecWarps);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (MODE == KVC_MODE_CODEBOOK) {
    for (int j = tid; j < p.cb_levels; j += kThreads)
      cbh[j] = __half_as_ushort(__float2half_rn(p.codebook[j]));
    if (p.cb_bits <= 4)
      for (int j = tid; j < p.cb_levels * p.cb_levels; j += kThreads) {
        const int c0 = j & (p.cb_levels - 1), c1 = j >> p.cb_bits;
        cb2[j] = (uint32_t)__half_as_ushort(__float2half_rn(p.codebook[c0])) |
                 ((uint32_t)__half_as_ushort(__float2half_rn(p.codebook[c1])) << 16);
      }
    const int wb = p.cb_bits, lm = p.cb_levels - 1;
    for (int j = tid; j < 2 * t.cb_rep; j += kThreads) {  // word j: pair j / 32
      const int e = j >> 5;
      cbr[j] = (uint32_t)__half_as_ushort(__float2half_rn(p.codebook[e & lm])) |
               ((uint32_t)__half_as_ushort(__float2half_rn(p.codebook[(e >> wb) & lm])) << 16);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr0 = tmem_base;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int slot = first / tps, blk = first % tps;
      // the next slot's tables are read one slot ahead, off the critical path
      auto info_of = [&](int sl, int& P, int& beta, int64_t& pay, int64_t& side) {
        P = 0; beta = 0; pay = 0; side = 0;
        if (sl < p.n_slots) { P = t.slotP[sl]; beta = p.basis_of[sl]; pay = p.pay_off[sl]; side = p.side_off[sl]; }
      };
      int P, beta, nP, nbeta;
      int64_t pay, side, npay, nside;
      info_of(slot, P, beta, pay, side);
      info_of(slot + 1, nP, nbeta, npay, nside);
      int cur_beta = -1, bslot = NB - 1;
      uint32_t bload[2] = {0u, 0u};
      uint32_t gload = 0;  // group mode: head slices loaded
      int issued = 0;
      Ring rr(RS);
      for (int i = 0; i < m; ++i, rr.next()) {
        const int s = rr.slot;
        // the decode of tile i - RS released this stage
        if (i >= RS && !mbar_wait_bounded(&row_empty[s], rr.phase ^ 1u, kWaitNs)) { abort_flag = 1; break; }
        int first_use = 0;
        if (!GRP && beta != cur_beta) {
          bslot = NB == 2 ? bslot ^ 1 : 0;
          if (bload[bslot] > 0 &&
              !mbar_wait_bounded(&b_empty[bslot], (bload[bslot] - 1) & 1, kWaitNs)) { abort_flag = 1; break; }
          mbar_arrive_expect_tx(&b_full[bslot], (uint32_t)b_bytes);
          bulk_load(Bs + bslot * b_bytes, t.B + (size_t)beta * D * K, (uint32_t)b_bytes, &b_full[bslot]);
          ++bload[bslot];
          cur_beta = beta;
          first_use = 1;
        }
        const int64_t t0 = (int64_t)blk * kTile;
        const int n = (int)min((int64_t)kTile, t.S - t0);
        const uint32_t cb = (uint32_t)((n * P + 15) & ~15);
        const uint32_t sbb = (uint32_t)((n * p.side_bytes + 15) & ~15);
        unsigned char* dst = rs + (size_t)s * t.rs_bytes;
        stage_hdr[s] = make_int4(P, n, bslot | (first_use << 1), 0);
        mbar_arrive_expect_tx(&row_full[s], 128u + cb + sbb);
        bulk_load(dst, t.chunks + (size_t)beta * 32, 128u, &row_full[s]);
        if (cb) bulk_load(dst + 128, p.store + pay + t0 * P, cb, &row_full[s]);
        if (sbb) bulk_load(dst + side_off, p.store + side + t0 * p.side_bytes, sbb, &row_full[s]);
        ++issued;
        if (GRP) {  // the hpg heads' slices of B through a ring of two buffers
          for (int j = 0; j < HPG; ++j, ++gload) {
            const int bs = (int)(gload & 1u);
            if (gload >= 2 && !mbar_wait_bounded(&b_empty[bs], ((gload >> 1) - 1) & 1, kWaitNs)) {
              abort_flag = 1;
              break;
            }
            mbar_arrive_expect_tx(&b_full[bs], (uint32_t)b_bytes);
            bulk_load(Bs + bs * b_bytes, t.B + ((size_t)beta * HPG + j) * D * K, (uint32_t)b_bytes,
                      &b_full[bs]);
          }
          if (abort_flag) break;
        }
        if (++blk == tps) {
          blk = 0;
          ++slot;
          P = nP; beta = nbeta; pay = npay; side = nside;
          info_of(slot + 1, nP, nbeta, npay, nside);
        }
      }
      // copies still in flight (after a time-out) land before the CTA exits
      for (int j = max(0, issued - RS); j < issued; ++j)
        mbar_wait_bounded(&row_full[j % RS], (j / RS) & 1, kWaitNs);
      for (int b2 = 0; b2 < 2; ++b2)
        if (bload[b2]) mbar_wait_bounded(&b_full[b2], (bload[b2] - 1) & 1, kWaitNs);
      for (uint32_t u = gload >= 2 ? gload - 2 : 0; u < gload; ++u)
        mbar_wait_bounded(&b_full[u & 1], (u >> 1) & 1, kWaitNs);
    }
  } else if (warp == kMmaWarp && GRP) {
    // ------------------------------------------------------------ MMA issuer, group mode
    // per tile: A once, then one accumulator per head (units u = tile * hpg + j)
    if (lane == 0) {
      const uint32_t sbo = (uint32_t)KC * 128;
      const uint32_t idesc = idesc_f16(kTile, D, 0);
      Ring ra(AS), rt(TS);
      uint32_t u = 0;
      for (int i = 0; i < m && !abort_flag; ++i, ra.next()) {
        const int a = ra.slot;
        if (!mbar_wait_bounded(&a_full[a], ra.phase, kWaitNs)) { abort_flag = 1; break; }
        const uint32_t a0 = taddr0 + t.a_col0 + a * t.a_cols;
        for (int j = 0; j < HPG; ++j, ++u, rt.next()) {
          const int acc = rt.slot, bs = (int)(u & 1u);
          if (!mbar_wait_bounded(&b_full[bs], (u >> 1) & 1, kWaitNs)) { abort_flag = 1; break; }
          // the epilogue of unit u - TS released this accumulator
          if (u >= (uint32_t)TS && !mbar_wait_bounded(&acc_empty[acc], rt.phase ^ 1u, kWaitNs)) {
            abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t b0 = smem_u32(Bs + bs * b_bytes);
          for (int ks = 0; ks < K / 16; ++ks)
            umma_f16_tmem_a(taddr0 + acc * D, a0 + ks * 8,
                            desc_kmajor_noswizzle(b0 + ks * 256, 128, sbo), idesc, ks > 0 ? 1u : 0u);
          umma_commit(&acc_full[acc]);
          umma_commit(&b_empty[bs]);
        }
        umma_commit(&a_empty[a]);
      }
      umma_commit(&done_bar);
      mbar_wait_bounded(&done_bar, 0, kWaitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sbo = (uint32_t)KC * 128;
      const uint32_t idesc = idesc_f16(kTile, D, 0);
      uint32_t buse[2] = {0u, 0u};
      Ring ra(AS), rt(TS);
      for (int i = 0; i < m; ++i, ra.next(), rt.next()) {
        const int a = ra.slot, acc = rt.slot;
        if (!mbar_wait_bounded(&a_full[a], ra.phase, kWaitNs)) { abort_flag = 1; break; }
        const int info = a_info[a], bs = info & 1;
        if (info & 2) {  // first tile on a newly loaded B: the other buffer is free when
          if (i > 0) umma_commit(&b_empty[NB == 2 ? bs ^ 1 : 0]);  // the MMAs issued so far finish
          if (!mbar_wait_bounded(&b_full[bs], buse[bs] & 1, kWaitNs)) { abort_flag = 1; break; }
          ++buse[bs];
        }
        // the epilogue of tile i - TS released this accumulator
        if (i >= TS && !mbar_wait_bounded(&acc_empty[acc], rt.phase ^ 1u, kWaitNs)) { abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t a0 = taddr0 + t.a_col0 + a * t.a_cols, b0 = smem_u32(Bs + bs * b_bytes);
        for (int ks = 0; ks < K / 16; ++ks)  // 16 fp16 of K = 8 TMEM columns of A
          umma_f16_tmem_a(taddr0 + acc * D, a0 + ks * 8,
                          desc_kmajor_noswizzle(b0 + ks * 256, 128, sbo), idesc, ks > 0 ? 1u : 0u);
        umma_commit(&acc_full[acc]);
        umma_commit(&a_empty[a]);
      }
      umma_commit(&done_bar);  // TMEM is released only after every MMA has finished
      mbar_wait_bounded(&done_bar, 0, kWaitNs);
    }
  } else if (warp >= kEpiWarps) {
    // ------------------------------------------------------------ decoders
    // Warp 8 + j decodes tokens 32 (j % 4) .. of chunks j / 4, j / 4 + 2, ...:
    // its tokens are the TMEM lanes its warp may access.  tcgen05.st is
    // warp-collective, so a warp leaves the loop only as a whole.
    const int dtid = tid - kEpiThreads;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int tt = dtid & (kTile - 1), c0 = dtid >> 7;
    const int n_groups = p.n_groups;
    Ring rr(RS), ra(AS), rn(kNormRing);
    for (int i = 0; i < m; ++i, rr.next(), ra.next(), rn.next()) {
      const int s = rr.slot, a = ra.slot;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&row_full[s], rr.phase, kWaitNs))) {
        abort_flag = 1;
        break;
      }
      // A buffer a was last read by MMA(i - AS)
      if (i >= AS &&
          !__all_sync(0xffffffffu, mbar_wait_bounded(&a_empty[a], ra.phase ^ 1u, kWaitNs))) {
        abort_flag = 1;
        break;
      }
      const int4 hdr = stage_hdr[s];
      const int P = hdr.x, n = hdr.y;
      const unsigned char* st_base = rs + (size_t)s * t.rs_bytes;
      const uint32_t* chunk = reinterpret_cast<const uint32_t*>(st_base);
      const unsigned char* rows = st_base + 128;
      // thread: token tt, chunks c0, c0 + 2, ...; four chunks' loads are
      // issued before their arithmetic
      const bool live = tt < n;
      const int rowoff = tt * P;
      const uint32_t a_tm = taddr0 + lane_base + t.a_col0 + a * t.a_cols;
      if (MODE == KVC_MODE_CODEBOOK && t.cb_rep) {
        // thread c0 takes the codes [c0 K / 2, (c0 + 1) K / 2)
        const unsigned char* row = rows + rowoff;
        const int nq = K / 64;
        if (p.cb_bits == 3) decode_cb_rows<3>(row, live, c0 * (K / 2), nq, cbr, a_tm);
        else if (p.cb_bits == 2) decode_cb_rows<2>(row, live, c0 * (K / 2), nq, cbr, a_tm);
        else decode_cb_rows<1>(row, live, c0 * (K / 2), nq, cbr, a_tm);
      } else if (MODE == KVC_MODE_UNIFORM && t.uni_w) {
        // one width w: code chunk c is the w bytes at c w of the row; thread
        // c0 takes half of the code chunks, c0 = 1 also the bias chunk (ones)
        // and the zero chunks after it
        const int w = t.uni_w, kcc = t.uni_chunks, half = (kcc + 1) / 2;
        const unsigned char* row = rows + rowoff;
        const int cend = c0 ? KC : half;
        for (int c = c0 * half; c < cend; ++c) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (live && c < kcc) {
            uint2 b = make_uint2(0u, 0u);
            if (w == 8) b = *reinterpret_cast<const uint2*>(row + 8 * c);
            else if (w == 4) b.x = *reinterpret_cast<const uint32_t*>(row + 4 * c);
            else if (w == 2) b.x = *reinterpret_cast<const uint16_t*>(row + 2 * c);
            else b.x = row[c];
            v = decode_uniform(b, w);
          } else if (live && c == kcc) {
            v.x = 0x3C003C00u;  // (1, 1): the two bias columns of B
          }
          tmem_st4(a_tm + c * 4, v);
        }
      } else
      for (int cb = c0; cb < KC; cb += 8) {
        uint32_t ent[4];
        uint2 bits[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = cb + 2 * u;
          ent[u] = c < KC ? chunk[c] : 0u;
          bits[u] = (ent[u] >> 31) && live ? bits_at(rows, rowoff + (int)(ent[u] & 0xffffu))
                                           : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = cb + 2 * u;
          if (c < KC) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (live) {
              const int w = (int)((ent[u] >> 16) & 0xfu);
              if (ent[u] >> 31) {
                v = MODE == KVC_MODE_CODEBOOK
                        ? (w <= 4 ? decode_codebook_pairs(bits[u], w, cb2)
                                  : decode_codebook(bits[u], w, cbh))
                        : decode_uniform(bits[u], w);
                if (GRP) {  // (code - 2^(w-1)) * s, one fp16 rounding; s: the chunk's group scale
                  const uint32_t sg = (uint32_t)reinterpret_cast<const uint16_t*>(
                      st_base + side_off)[tt * n_groups + (int)((ent[u] >> 20) & 0xffu)];
                  const uint32_t s2 = sg | (sg << 16);
                  v = make_uint4(hmul2_bits(v.x, s2), hmul2_bits(v.y, s2), hmul2_bits(v.z, s2),
                                 hmul2_bits(v.w, s2));
                }
              } else if (ent[u] >> 30) {
                v.x = 0x3C003C00u;  // (1, 1): the two bias columns of B
              }
            }
            tmem_st4(a_tm + c * 4, v);  // chunk c: K positions 8c .. 8c+7
          }
        }
      }
      // Norm ring entry i % kNormRing is next written by the decode of tile
      // i + kNormRing, which waits for MMA(i + kNormRing - AS), which waited
      // for the epilogue of tile i + kNormRing - AS - TS >= i + 1 to release
      // its accumulator, after the epilogue of tile i had read its norms; so
      // the ring's barrier phases are never more than one apart.
      if (MODE == KVC_MODE_CODEBOOK && c0 == 0)
        norm_ring[rn.slot * kTile + tt] =
            live ? __half2float(__ushort_as_half(
                       reinterpret_cast<const uint16_t*>(st_base + side_off)[tt]))
                 : 0.f;
      if (dtid == 0) a_info[a] = hdr.z;
      tmem_wait_st();
      tc_fence_before();  // A is read by the MMA thread's tcgen05.mma
      __syncwarp();
      if (lane == 0) {
        if (MODE == KVC_MODE_CODEBOOK) mbar_arrive(&norm_full[rn.slot]);
        mbar_arrive(&a_full[a]);
        mbar_arrive(&row_empty[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32 (w % 4) .. (its tokens) and half w / 4 of the
    // columns.  When each half is a whole number of 64-column output boxes
    // (D = 128, 256) the two halves run as independent groups of four warps,
    // each with its own barrier, staging boxes and TMA store; otherwise the
    // eight warps form one group.
    const int quarter = warp & 3, half = warp >> 2, row = quarter * 32 + lane;
    const int nblk = D / 64;  // 32-column blocks per half
    const bool split = (nbox & 1) == 0;
    const int gthreads = split ? kEpiThreads / 2 : kEpiThreads;
    const int bar_id = kEpiBar + (split ? half : 0);
    const bool issuer = split ? (tid & (kEpiThreads / 2 - 1)) == 0 : tid == 0;
    const int box0 = split ? half * (nbox / 2) : 0, nbox_g = split ? nbox / 2 : nbox;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int slot = first / tps, blk = first % tps, head = 0;
    float* mean_g = mean_c + (split ? half : 0) * (HPG * (nbox / 2) * 64);  // [hpg][this group's columns]
    int mean_beta = -1;
    Ring rt(TS), rs_(SS), rn(kNormRing);
    for (int i = 0; i < m * HPG; ++i, rt.next(), rs_.next()) {  // units: tile x head
      const int acc = rt.slot;
      bool late = !mbar_wait_bounded(&acc_full[acc], rt.phase, kWaitNs);
      if (MODE == KVC_MODE_CODEBOOK)
        late = late || !mbar_wait_bounded(&norm_full[rn.slot], rn.phase, kWaitNs);
      if (issuer) bulk_wait_read_n(SS - 1);  // this group's store of tile i-SS has left staging
      if (named_bar_or(bar_id, gthreads, late || abort_flag)) { abort_flag = 1; break; }
      if (GRP) {  // this group's columns of the basis' mean rows, refreshed on a new basis
        const int beta = p.basis_of[slot];
        if (beta != mean_beta) {
          const int per = nbox_g * 64, gt = tid & (gthreads - 1);
          for (int e = gt; e < HPG * per; e += gthreads) {
            const int j = e / per, c = box0 * 64 + e % per;
            mean_g[j * per + (c - box0 * 64)] = t.bias[((size_t)beta * HPG + j) * D + c];
          }
          mean_beta = beta;
          named_bar_sync(bar_id, gthreads);
        }
      }
      tc_fence_after();
      const float nrm = MODE == KVC_MODE_CODEBOOK ? norm_ring[rn.slot * kTile + row] : 1.f;
      const float* brow = GRP ? mean_g + head * (nbox_g * 64) - box0 * 64 : nullptr;
      const uint32_t lane_addr = taddr0 + acc * D + lane_off;
      unsigned char* stg = stage + rs_.slot * nbox * 16384;
      for (int j = 0; j < nblk; j += 2) {  // two 32-column loads in flight
        const int c32a = half * nblk + j;
        const bool two = j + 1 < nblk;
        uint32_t r[2][32];
        tmem_ld32(lane_addr + c32a * 32, r[0]);
        if (two) tmem_ld32(lane_addr + (c32a + 1) * 32, r[1]);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (h == 1 && !two) break;
          const int c32 = c32a + h;
          unsigned char* dst = stg + (c32 >> 1) * 16384 + row * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              x[e] = MODE == KVC_MODE_CODEBOOK ? __uint_as_float(r[h][q * 8 + e]) * nrm
                                               : __uint_as_float(r[h][q * 8 + e]);
            if (GRP) {  // + mean, this head's slice
              const float4 b0 = *reinterpret_cast<const float4*>(brow + c32 * 32 + q * 8);
              const float4 b1 = *reinterpret_cast<const float4*>(brow + c32 * 32 + q * 8 + 4);
              x[0] += b0.x; x[1] += b0.y; x[2] += b0.z; x[3] += b0.w;
              x[4] += b1.x; x[5] += b1.y; x[6] += b1.z; x[7] += b1.w;
            }
            const int c16 = (c32 & 1) * 4 + q;
            *reinterpret_cast<uint4*>(dst + ((c16 ^ (row & 7)) << 4)) =
                make_uint4(pack_out(x[0], x[1], OUT_BF16), pack_out(x[2], x[3], OUT_BF16),
                           pack_out(x[4], x[5], OUT_BF16), pack_out(x[6], x[7], OUT_BF16));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      fence_proxy_async_smem();  // staging is read by the TMA store (async proxy)
      named_bar_sync(bar_id, gthreads);
      if (issuer) {  // the tensor map's (b, h) index: slot * hpg + head
        for (int bx = box0; bx < box0 + nbox_g; ++bx)
          tma_store_3d(&omap, stg + bx * 16384, bx * 64, blk * kTile, slot * HPG + head);
        bulk_commit();
      }
      if (++head == HPG) {
        head = 0;
        if (MODE == KVC_MODE_CODEBOOK) rn.next();
        if (++blk == tps) { blk = 0; ++slot; }
      }
    }
    if (issuer) bulk_wait_read0();  // staging is read before the CTA exits
  }
  __syncthreads();
  if (abort_flag && tid == 0) atomicCAS(p.err, 0, kErrTimeout);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(taddr0, t.cols);
  }
}

using PipeKernel = void (*)(const Params, const PipeArgs, const CUtensorMap);

PipeKernel pipe_kernel_for(int mode, int out_dtype) {
  const bool bf = out_dtype == KVC_BF16;
  if (mode == KVC_MODE_UNIFORM)
    return bf ? fetch_pipe_kernel<KVC_MODE_UNIFORM, true> : fetch_pipe_kernel<KVC_MODE_UNIFORM, false>;
  if (mode == KVC_MODE_GROUP)
    return bf ? fetch_pipe_kernel<KVC_MODE_GROUP, true> : fetch_pipe_kernel<KVC_MODE_GROUP, false>;
  return bf ? fetch_pipe_kernel<KVC_MODE_CODEBOOK, true> : fetch_pipe_kernel<KVC_MODE_CODEBOOK, false>;
}

}  // namespace

size_t fetch_pipe_smem(int mode, int D, int hpg, int K, int side_bytes, int pmax, int n_bases,
                       int min_rs, int cb_bits, FetchPipeShape* sh) {
  const size_t rows = ((size_t)kTile * pmax + 16 + 15) & ~size_t(15);
  const size_t side = ((size_t)kTile * side_bytes + 16 + 15) & ~size_t(15);
  FetchPipeShape z;
  z.rs_bytes = (int)(128 + rows + side);
  // TMEM (512 columns): accumulators of D columns, then A buffers of K/2
  // columns (two fp16 per column) rounded up to 32
  z.a_cols = (K / 2 + 31) / 32 * 32;
  z.n_a = 2;
  z.n_acc = std::min(kMaxTS, (512 - z.n_a * z.a_cols) / D);
  if (z.n_acc < 1) return 0;
  if (z.n_acc * D + (z.n_a + 1) * z.a_cols <= 512) z.n_a = kMaxAS;
  z.a_col0 = z.n_acc * D;
  z.n_b = n_bases > 1 ? 2 : 1;
  z.n_stg = 2;
  z.n_rs = min_rs;
  // codebook rows of at most 3-bit codes (one segment from byte 0, K = D a
  // multiple of 64) decode two codes per lookup from a pair table replicated
  // once per lane: 2^(2 bits) pairs x 32 copies, in 8-byte slots
  z.cb_rep = mode == KVC_MODE_CODEBOOK && cb_bits >= 1 && cb_bits <= 3 && K == D && K % 64 == 0
                 ? (1 << (2 * cb_bits)) * 16
                 : 0;
  const size_t tail = mode == KVC_MODE_CODEBOOK
                          ? 256 * 2 + (size_t)kNormRing * kTile * 4 + 256 * 4 + (size_t)z.cb_rep * 8
                      : mode == KVC_MODE_GROUP ? (size_t)hpg * D * 4
                                               : 0;
  auto total = [&](const FetchPipeShape& q) {
    return 1024 + (size_t)q.n_stg * (D / 64) * 16384 + (size_t)q.n_b * D * K * 2 +
           (size_t)q.n_rs * q.rs_bytes + tail;
  };
  const size_t limit = 226 * 1024;
  if (total(z) > limit) return 0;
  // grow, in order of benefit: staging (stores in flight), then row stages
  auto grow = [&](int FetchPipeShape::*f, int to) {
    while (z.*f < to) {
      FetchPipeShape q = z;
      ++(q.*f);
      if (total(q) > limit) break;
      z = q;
    }
  };
  grow(&FetchPipeShape::n_stg, kMaxSS);
  grow(&FetchPipeShape::n_rs, kMaxRS);
  *sh = z;
  return total(z);
}

cudaError_t launch_fetch_pipe(const TcPlan& plan, const Params& p, const FetchArgs& f,
                              const CUtensorMap& map, cudaStream_t s, int* nk) {
  PipeKernel k = pipe_kernel_for(p.mode, p.out_dtype);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)plan.pipe_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((f.S + kTile - 1) / kTile);
  const int total = tiles * p.n_slots;
  const int grid = std::min(total, sm_count());
  const FetchPipeShape& sh = plan.pipe;
  const PipeArgs t{plan.fetchB, plan.bias, plan.chunks32, plan.slotP, plan.fetch_K, plan.pipe_cols,
                   sh.n_acc, sh.n_a, sh.n_rs, sh.a_col0, sh.a_cols, sh.n_stg, sh.n_b, sh.rs_bytes,
                   sh.cb_rep, sh.uni_w, sh.uni_chunks, f.S, tiles, total};
  k<<<(unsigned)grid, kThreads, plan.pipe_smem, s>>>(p, t, map);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
