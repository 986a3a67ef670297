// Tensor-core projection of group mode (PALU-style head groups):
//   z = (x - mean) V,  x the group's hpg heads side by side (d_in = hpg D),
// written as fp32 rows for the CUDA-core group quantiser, which reads them in
// place of its own projection (append_generic_kernel with a ZIn).
//
// The operands are exact fp16 pieces:
//   x - mean is rounded once to fp32 (as the CUDA-core path does), scaled by
//   2^sx and split as xc = x_hi + x_lo (two fp16 roundings, residual
//   <= 2^-22 |xc| or 2^-25 near zero);
//   V is scaled by 2^se and split as V_hi + V_lo (residual <= 2^-22 |V|).
// Per head the MMA accumulates x_hi V_hi into one TMEM accumulator (a chain
// of D terms) and x_hi V_lo + x_lo V_hi into another; x_lo V_lo (<= 2^-22 of
// the product) is left out.  After each head the epilogue warps read both
// accumulators and add them into fp32 registers, so the tensor core's
// truncated accumulation never runs longer than one head:
//   |z32 - z| <= gamma ||x - mean|| ||V_k|| + ex ||V_k|| + en ||x - mean||,
// gamma, ex and en set on the host (kvc_tc.cu) from the same accumulation
// model as the uniform append's.
//
// One CTA per SM walks 128-token tiles of (batch, group) slots:
//   producer (warp 16)  x boxes (64 columns x 128 tokens, TMA, 128-byte
//                       swizzle) into four 32 KB stages, basis slices
//                       (rpad x 64 fp16, bulk copies) into a ring;
//   MMA (warp 17)       per box 12 MMAs of M = 128, N = rpad, K = 16;
//   warps 0-15          drain this head's accumulators (warp w reads TMEM
//                       lanes 32 (w % 4).. (its tokens) and the w / 4-th
//                       quarter of the columns), then split the boxes of the
//                       head two ahead in place (x_hi over the raw tile, x_lo
//                       beside it).
// A tile holding a value the split cannot represent (|xc 2^sx| >= 65504, or
// not finite) is flagged; the quantiser projects that tile itself.
#include <cuda_fp16.h>

#include <algorithm>

#include "kvc_sm100.cuh"
#include "kvc_tc.h"

namespace kvc {

using namespace sm100;

namespace {

constexpr int kTile = 128;
constexpr int kEW = 16;  // converter / epilogue warps
constexpr int kProdW = kEW, kMmaW = kEW + 1;
constexpr int kThr = (kEW + 2) * 32;
constexpr int kNA = 4;           // x stages
constexpr int kStage = 32768;    // x_hi (the raw tile lands here) + x_lo
constexpr int kMaxNB = 8;        // basis slice stages
constexpr int kBarConv = 1;      // named barrier of the 16 converter warps
constexpr uint64_t kWaitNs = 2000000000ull;

struct GpArgs {
  const uint16_t* B;  // [nb][hpg][D/64][2][rpad][64] fp16, core-matrix order
  float* z;           // [n_slots][Tc][r]
  int* ovf;           // [n_slots][tiles per slot]
  int64_t Tc;         // z rows per slot
  int rpad, nbx, n_b, tps, total;
  float xscale, zscale;
};

struct Ring {
  int n, slot;
  uint32_t phase;
  __device__ explicit Ring(int n_) : n(n_), slot(0), phase(0u) {}
  __device__ void next() {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

template <bool BF16IN>
__device__ __forceinline__ float in_to_float(uint32_t w, int half) {
  const uint16_t b = (uint16_t)(half ? (w >> 16) : (w & 0xffffu));
  if (BF16IN) return __uint_as_float((uint32_t)b << 16);
  return __half2float(__ushort_as_half(b));
}

template <int CPT, bool BF16IN>
// 18 warps: five share one SM sub-partition's 16K registers, so 96 per thread.
__global__ void __launch_bounds__(kThr, 1)
    group_proj_kernel(const Params p, const GpArgs g, const __grid_constant__ CUtensorMap xmap,
                      const AppendArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t x_full[kNA], a_full[kNA], a_empty[kNA], b_full[kMaxNB], b_empty[kMaxNB];
  __shared__ uint64_t acc_full, acc_empty, done_bar;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;

  const int hpg = p.hpg, D = p.D, r = p.r;
  const int rpad = g.rpad, nbx = g.nbx, NB = g.n_b, tps = g.tps;
  const int units = hpg * nbx;  // boxes per tile
  const uint32_t bblk = (uint32_t)rpad * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int first = (int)((int64_t)g.total * blockIdx.x / G);
  const int m = (int)((int64_t)g.total * (blockIdx.x + 1) / G) - first;
  const uint32_t ncols = (uint32_t)max(32, 2 * rpad);

  unsigned char* ast = smem;                 // kNA x kStage
  unsigned char* bst = smem + kNA * kStage;  // NB x bblk

  if (warp == kMmaW) tmem_alloc(&tmem_base, ncols);
  if (tid == 0) {
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&a_full[i], kEW);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < NB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEW);
    mbar_init(&done_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tacc = tmem_base;

  if (warp == kProdW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Ring ra(kNA), rb(NB);
      int na = 0, nl = 0;
      int slot = first / tps, blk = first % tps;
      for (int i = 0; i < m && !abort_flag; ++i) {
        const int beta = p.basis_of[slot];
        const int bb = slot / p.Hg, gg = slot - bb * p.Hg;
        for (int u = 0; u < units && !abort_flag; ++u) {
          const int h = u / nbx, bx = u - h * nbx;
          if (na >= kNA && !mbar_wait_bounded(&a_empty[ra.slot], ra.phase ^ 1u, kWaitNs)) {
            abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&x_full[ra.slot], 16384u);
          tma_load_4d(ast + (size_t)ra.slot * kStage, &xmap, &x_full[ra.slot], bx * 64, blk * kTile,
                      gg * hpg + h, bb);
          ra.next();
          ++na;
          for (int pc = 0; pc < 2; ++pc) {
            if (nl >= NB && !mbar_wait_bounded(&b_empty[rb.slot], rb.phase ^ 1u, kWaitNs)) {
              abort_flag = 1;
              break;
            }
            mbar_arrive_expect_tx(&b_full[rb.slot], bblk);
            const size_t blkno = (((size_t)beta * hpg + h) * nbx + bx) * 2 + pc;
            bulk_load(bst + (size_t)rb.slot * bblk, g.B + blkno * (bblk / 2), bblk, &b_full[rb.slot]);
            rb.next();
            ++nl;
          }
        }
        if (++blk == tps) {
          blk = 0;
          ++slot;
        }
      }
      // copies still in flight (after an abort) land before the CTA exits
      for (int j = max(0, na - kNA); j < na; ++j)
        mbar_wait_bounded(&x_full[j % kNA], (uint32_t)(j / kNA) & 1u, kWaitNs);
      for (int j = max(0, nl - NB); j < nl; ++j)
        mbar_wait_bounded(&b_full[j % NB], (uint32_t)(j / NB) & 1u, kWaitNs);
    }
  } else if (warp == kMmaW) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTile, rpad, 0);
      Ring ra(kNA), rb(NB);
      uint32_t heads = 0;
      bool ok = true;
      for (int i = 0; i < m && ok; ++i)
        for (int h = 0; h < hpg && ok; ++h, ++heads) {
          // the epilogue has read the previous head's accumulators
          if (heads > 0 && !mbar_wait_bounded(&acc_empty, (heads - 1) & 1u, kWaitNs)) ok = false;
          tc_fence_after();
          for (int bx = 0; bx < nbx && ok; ++bx) {
            if (!mbar_wait_bounded(&a_full[ra.slot], ra.phase, kWaitNs)) { ok = false; break; }
            if (!mbar_wait_bounded(&b_full[rb.slot], rb.phase, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const uint32_t xhi = smem_u32(ast + (size_t)ra.slot * kStage), xlo = xhi + 16384;
            uint32_t vb = smem_u32(bst + (size_t)rb.slot * bblk);
            // V_hi: x_hi V_hi -> hi accumulator, x_lo V_hi -> rest accumulator
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = desc_kmajor_noswizzle(vb + ks * 256, 128, 1024);
              const uint32_t acc = (bx | ks) ? 1u : 0u;
              umma_f16(tacc, desc_kmajor_sw128(xhi + ks * 32), bd, idesc, acc);
              umma_f16(tacc + rpad, desc_kmajor_sw128(xlo + ks * 32), bd, idesc, acc);
            }
            umma_commit(&b_empty[rb.slot]);
            rb.next();
            // V_lo: x_hi V_lo -> rest accumulator
            if (!mbar_wait_bounded(&b_full[rb.slot], rb.phase, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            vb = smem_u32(bst + (size_t)rb.slot * bblk);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              umma_f16(tacc + rpad, desc_kmajor_sw128(xhi + ks * 32),
                       desc_kmajor_noswizzle(vb + ks * 256, 128, 1024), idesc, 1u);
            umma_commit(&b_empty[rb.slot]);
            rb.next();
            umma_commit(&a_empty[ra.slot]);
            ra.next();
          }
          if (ok) umma_commit(&acc_full);
        }
      if (!ok) abort_flag = 1;
      // every MMA issued by this thread has completed before TMEM is freed
      umma_commit(&done_bar);
      mbar_wait_bounded(&done_bar, 0, kWaitNs);
    }
  } else {
    // ------------------------------------------------------------ split + epilogue
    const int quarter = warp & 3, cq = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t t_hi = tacc + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cq * CPT);
    const uint32_t t_rest = t_hi + (uint32_t)rpad;
    const float xscale = g.xscale;

    // split cursor: tile ci (slot cs, block cb), box cu
    Ring rc(kNA);
    int ci = 0, cs = first / tps, cb = first % tps, cu = 0;
    bool bad = false;
    // Splits the boxes of the next head in place.  Every converter warp runs
    // the same sequence (the tile-end barrier below needs all 16).
    auto split_head = [&]() {
      const int beta = p.basis_of[cs];
      for (int e = 0; e < nbx; ++e, ++cu) {
        const int h = cu / nbx, bx = cu - h * nbx;
        if (!abort_flag && !mbar_wait_bounded(&x_full[rc.slot], rc.phase, kWaitNs)) abort_flag = 1;
        unsigned char* st = ast + (size_t)rc.slot * kStage;
        const float* mrow = p.mean + (size_t)beta * p.d_in + h * D + bx * 64;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int L = cq * 2 + c;  // logical 16-byte chunk: columns 8L .. 8L+7
          const int off = row * 128 + ((L ^ (row & 7)) << 4);
          const uint4 raw = *reinterpret_cast<const uint4*>(st + off);
          const float4 m0 = __ldg(reinterpret_cast<const float4*>(mrow + L * 8));
          const float4 m1 = __ldg(reinterpret_cast<const float4*>(mrow + L * 8 + 4));
          const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t hp = 0, lp = 0;
#pragma unroll
            for (int s = 0; s < 2; ++s) {
              const float xc = (in_to_float<BF16IN>(rw[q], s) - mv[2 * q + s]) * xscale;
              bad |= !(fabsf(xc) < 65504.f);
              const __half hi = __float2half_rn(xc);
              const __half lo = __float2half_rn(xc - __half2float(hi));  // xc - hi is exact
              hp |= (uint32_t)__half_as_ushort(hi) << (16 * s);
              lp |= (uint32_t)__half_as_ushort(lo) << (16 * s);
            }
            hw[q] = hp;
            lw[q] = lp;
          }
          *reinterpret_cast<uint4*>(st + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(st + 16384 + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_smem();  // generic-proxy writes, read next by the MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[rc.slot]);
        rc.next();
      }
      if (cu == units) {  // the tile is split: publish whether the quantiser must project it
        const bool any = named_bar_or(kBarConv, kEW * 32, bad);
        if (tid == 0) g.ovf[(size_t)cs * tps + cb] = any ? 1 : 0;
        bad = false;
        cu = 0;
        ++ci;
        if (++cb == tps) {
          cb = 0;
          ++cs;
        }
      }
    };

    // Two heads are split ahead: the MMA of head j + 1 starts as soon as head
    // j is drained, and splitting head j + 2 overlaps it.
    if (m > 0) split_head();
    if (ci < m) split_head();
    int es = first / tps, eb = first % tps;
    uint32_t heads = 0;
    for (int i = 0; i < m; ++i) {
      float zacc[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) zacc[j] = 0.f;
      for (int h = 0; h < hpg; ++h, ++heads) {
        if (!abort_flag && !mbar_wait_bounded(&acc_full, heads & 1u, kWaitNs)) abort_flag = 1;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < CPT / 8; ++c) {
          uint32_t hi[8], lo[8];
          tmem_ld8(t_hi + c * 8, hi);
          tmem_ld8(t_rest + c * 8, lo);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            zacc[c * 8 + j] += __uint_as_float(hi[j]) + __uint_as_float(lo[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty);
        if (ci < m) split_head();
      }
      const int64_t t = (int64_t)eb * kTile + row;
      if (t < a.T) {
        float* zr = g.z + ((int64_t)es * g.Tc + t) * r;
        const int k0 = cq * CPT;
        if (k0 + CPT <= r && (r & 3) == 0) {
#pragma unroll
          for (int j = 0; j < CPT; j += 4)
            *reinterpret_cast<float4*>(zr + k0 + j) =
                make_float4(zacc[j] * g.zscale, zacc[j + 1] * g.zscale, zacc[j + 2] * g.zscale,
                            zacc[j + 3] * g.zscale);
        } else {
#pragma unroll
          for (int j = 0; j < CPT; ++j)
            if (k0 + j < r) zr[k0 + j] = zacc[j] * g.zscale;
        }
      }
      if (++eb == tps) {
        eb = 0;
        ++es;
      }
    }
  }
  __syncthreads();
  if (abort_flag && tid == 0) atomicCAS(p.err, 0, kErrTimeout);
  if (warp == kMmaW) {
    tc_fence_after();
    tmem_dealloc(tacc, ncols);
  }
}

using GpKernel = void (*)(const Params, const GpArgs, const CUtensorMap, const AppendArgs);

template <bool BF16IN>
GpKernel gp_kernel_for(int rpad) {
  switch (rpad) {
    case 32: return group_proj_kernel<8, BF16IN>;
    case 64: return group_proj_kernel<16, BF16IN>;
    case 128: return group_proj_kernel<32, BF16IN>;
    default: return group_proj_kernel<64, BF16IN>;
  }
}

}  // namespace

size_t group_proj_smem(int rpad, int* n_b) {
  const size_t bblk = (size_t)rpad * 128;
  const size_t budget = 227 * 1024 - 1024 - 1024;  // dynamic limit, alignment, static barriers
  const size_t fixed = (size_t)kNA * kStage;
  if (budget < fixed + 2 * bblk) return 0;
  const int nb = (int)std::min<size_t>(kMaxNB, (budget - fixed) / bblk);
  *n_b = nb;
  return 1024 + fixed + (size_t)nb * bblk;
}

cudaError_t launch_group_proj(const TcPlan& plan, const Params& p, const AppendArgs& a,
                              const CUtensorMap& xmap, cudaStream_t s, int* nk) {
  GpKernel kern = plan.gp_bf16 ? gp_kernel_for<true>(plan.gp_rpad) : gp_kernel_for<false>(plan.gp_rpad);
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.gp_smem);
  if (e != cudaSuccess) return e;
  GpArgs g;
  g.B = plan.gpB;
  g.z = plan.zbuf;
  g.ovf = plan.zovf;
  g.Tc = plan.gp_Tc;
  g.rpad = plan.gp_rpad;
  g.nbx = p.D / 64;
  g.n_b = plan.gp_nb;
  g.tps = (int)((a.T + kTile - 1) / kTile);
  g.total = g.tps * p.n_slots;
  g.xscale = plan.gp_xscale;
  g.zscale = plan.gp_zscale;
  const int grid = std::min(g.total, sm_count());
  kern<<<grid, kThr, plan.gp_smem, s>>>(p, g, xmap, a);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
