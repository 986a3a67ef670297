// Warp-specialised persistent append for one head per slot (uniform and
// codebook modes): z = x V (tensor cores), quantise, pack, write the rows.
//
// One CTA per SM walks a contiguous run of 128-token tiles.  Three roles hand
// tiles on through mbarrier rings:
//   producer (one thread)  TMA-loads each x tile (128-byte swizzle, the A
//                          operand as is) together with its basis' quantiser
//                          table into a ring of x stages, and the basis B into
//                          one of (up to) two B buffers when the basis changes;
//   MMA (one thread)       one chain of tcgen05.mma per tile with the basis'
//                          exact 16-bit pieces stacked along N, so x is read
//                          once: accumulator columns [piece][component];
//   quantiser (2 x 8 warps) two groups take alternate tiles; warp w of a group
//                          owns TMEM lanes 32 (w % 4) .. (its tokens) and half
//                          w / 4 of the components: ||x||, the
//                          fast-path codes z = hi + (mid + lo), the exact
//                          re-decision of codes near a boundary (one warp per
//                          queued code, V^T from shared memory), bit-packing
//                          and a coalesced copy of the packed rows to the store.
// Codes are staged at chunk-aligned positions: every packed segment starts on
// an 8-code chunk, and 8 codes of width w pack into exactly w bytes, so each
// (token, chunk) packs on its own from one 64-bit load.
// The x stage is released once the rows are packed (the re-decision reads x,
// the packing the stage's table), the accumulator right after the quantiser
// has read it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "kvc_append_exact.cuh"
#include "kvc_sm100.cuh"
#include "kvc_tc.h"

namespace kvc {

using namespace sm100;

namespace {

constexpr int kTile = 128;
// Two quantiser groups of 8 warps take alternate tiles, so one group's
// barrier and re-decision latency hides under the other's work.  Warp w of a
// group reads TMEM lanes 32 (w % 4) .. (its tokens) and column half w / 4.
constexpr int kQG = 2;
constexpr int kQWarps = 8;   // warps of one group
constexpr int kQThreads = kQWarps * 32;
constexpr int kNCB = kQWarps / 4;  // column blocks per group
constexpr int kThreadsWs = (kQG * kQWarps + 2) * 32;
constexpr int kMaxXS = 4, kMaxTS = 4;
constexpr int kQBar = 1;  // named barrier of the quantiser warps
constexpr uint64_t kWaitNs = 2000000000ull;

struct AppendWsArgs {
  const uint16_t* B;        // [nb][pieces * rpad][D] UMMA no-swizzle K-major
  const double* c64;        // [nb][r] mean . V_k
  const unsigned char* tab; // [nb][tab_bytes] quantiser table of each basis
  int rpad, npieces, acc_stride, cols;  // accumulator columns and stride; TMEM allocated
  int n_acc, n_x, n_b;      // accumulators, x stages, B buffers
  int x_stage, tab_bytes, pmax;
  int ks;                   // bytes per token row of the code staging (chunk-aligned)
  int nq;                   // queue entries per quantiser group
  int vt_smem;              // each group keeps its basis' V^T in shared memory
  float inv_scale, gamma;
  int tiles_per_slot, total_tiles;
  unsigned long long wait_ns;  // limit of the loop waits (the drains keep kWaitNs)
};

// Per-basis quantiser table (host layout in append_ws_table), per component:
//   q4    uniform fast path u = fma(z, A, Bc), bound tau = fma(T1, ||x||, T2)
//         (A = 2^-s / step, Bc = -(mean . V_k + lo) / step; see the plan);
//   cff   mean . V_k, iff 1/step (as double-float pairs), lo, vn = ||V_k||
//         (rounded up);
//   qp    qmax and the chunk-aligned position (not kept: the row's scratch byte);
// then the pack chunks.
struct Tab {
  const float4* q4;
  const float2 *cff, *iff;
  const float *lo, *vn;
  const int2* qp;
  const uint32_t* chunk;  // [32]: first byte | width << 16 | (codes - 1) << 20 | valid << 31
  __device__ Tab(const unsigned char* base, int rpad)
      : q4(reinterpret_cast<const float4*>(base)),
        cff(reinterpret_cast<const float2*>(q4 + rpad)),
        iff(cff + rpad),
        lo(reinterpret_cast<const float*>(iff + rpad)),
        vn(lo + rpad),
        qp(reinterpret_cast<const int2*>(vn + rpad)),
        chunk(reinterpret_cast<const uint32_t*>(qp + rpad)) {}
};

struct XHdr {  // per x stage, written by the producer
  int n, info, slot, P;     // tokens; B buffer | first use << 1; slot; packed row bytes
  int beta, pad;            // basis
  long long row0;           // store row of the tile's first token
  long long pay, side;      // the slot's payload and side-word offsets in the store
};

// Wait for phase `parity` of `bar`; false after `ns` of wall time, or as soon
// as another role has given up (*abort set), so that one time-out unwinds
// every role promptly.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint64_t ns,
                                              volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > ns) return false;
  }
}

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

// Shared-memory scratch of one quantiser group: code staging, packed rows,
// the re-decision queue and its aux values, partial norms, side words.
// nq: queue entries (near codes waiting for their exact decision)
__host__ __device__ constexpr size_t ws_group_bytes(int ks, int pmax, int nq) {
  return ((size_t)kTile * ks + (((size_t)kTile * pmax + 16 + 15) & ~size_t(15)) +
          (size_t)nq * 12 + kNCB * kTile * 4 + kTile * 2 + 15) & ~size_t(15);
}

// Decide code k of token tt exactly (k == kNormEntry: the fp16 norm of a
// codebook token) from x in shared memory, V^T row k and the basis table;
// lane 0 (or the lone thread) writes the result.  Double-float arithmetic
// (no fp64: its throughput is very low here): z from the compensated dot,
// u = (z - c - lo) (1/step), rounded half to even on the exact pair; the
// nearest centroid by comparing z with the exact midpoints times ||x||.
template <int MODE, bool BF16, bool WARP>
__device__ void refine_ws(const Params& p, const Tab& tb, const float* Vt, const float* cb_s,
                          const unsigned char* xs, unsigned char* codes_s, int ks, __half* side_s,
                          unsigned* nside, unsigned long long* cnt, int tt, int k, int lane,
                          float uf, float tau) {
  const int D = p.D;
  const int kp = k == (int)kNormEntry ? 0 : tb.qp[k].y;
  if (MODE == KVC_MODE_UNIFORM) {
    const ff2 z = dot2_ff<BF16, WARP>(xs, tt, D, Vt + (size_t)k * D, lane);
    if (lane == 0) {
      const float2 c = tb.cff[k], iv = tb.iff[k];
      const ff2 zl = ff_add(ff_add(z, ff2{-c.x, -c.y}), ff2{-tb.lo[k], 0.f});
      const ff2 u = ff_mul(zl, ff2{iv.x, iv.y});
      const float q = ff_rint(u);
      const int qmax = tb.qp[k].x;
      codes_s[tt * ks + kp] = (uint8_t)(int)fminf(fmaxf(q, 0.f), (float)qmax);
      if (tau > 0.f) atomicMax(&cnt[3], (unsigned long long)__float_as_uint(
                                                   fabsf(uf - u.hi) / tau));
    }
  } else {
    const ff2 nrm = ff_sqrt(dot2_ff<BF16, WARP>(xs, tt, D, nullptr, lane));
    if (k == (int)kNormEntry) {
      if (lane == 0) {
        const __half h = ff_to_half(nrm);
        side_s[tt] = h;
        atomicAdd(nside, 1u);
      }
    } else {
      const ff2 z = dot2_ff<BF16, WARP>(xs, tt, D, Vt + (size_t)k * D, lane);
      if (lane == 0) {
        // nearest centroid, ties to the lower one: the number of exact
        // midpoints m (double-float, from the fp32 centroids) with
        // m ||x|| < z; ||x|| = 0 means u = 0
        const bool zero = nrm.hi == 0.f;
        int lo_i = 0, hi_i = p.cb_levels - 1;
        while (lo_i < hi_i) {
          const int mid = (lo_i + hi_i) >> 1;
          float ms, me;
          two_sum(cb_s[mid], cb_s[mid + 1], ms, me);
          const ff2 m{0.5f * ms, 0.5f * me};
          const bool below = zero ? m.hi < 0.f : ff_less(ff_mul(m, nrm), z);
          if (below) lo_i = mid + 1; else hi_i = mid;
        }
        codes_s[tt * ks + kp] = (uint8_t)lo_i;
        if (tau > 0.f && !zero)
          atomicMax(&cnt[3], (unsigned long long)__float_as_uint(
                                        fabsf(uf - z.hi / nrm.hi) / tau));
      }
    }
  }
}

// The same decisions by a group of GL lanes, several groups of a warp each
// deciding its own queue entry (act: the group has one; every lane calls).
// A codebook code takes ||x||^2 and x . V_k from one pass over the row.
template <int MODE, bool BF16, int GL>
__device__ __forceinline__ void refine_group(const Params& p, const Tab& tb, const float* Vt,
                                             const float* cb_s, const unsigned char* xs,
                                             unsigned char* codes_s, int ks, __half* side_s,
                                             unsigned* nside, unsigned long long* cnt, int tt,
                                             int k, int sub, bool act, float uf, float tau) {
  const int D = p.D;
  const bool norm_entry = k == (int)kNormEntry;
  const int kk = norm_entry ? 0 : k;
  ff2 xx, z;
  dot2_ff_group<BF16, GL>(xs, tt, D, norm_entry ? nullptr : Vt + (size_t)kk * D, sub, xx, z);
  if (!act || sub != 0) return;
  const int kp = norm_entry ? 0 : tb.qp[k].y;
  if (MODE == KVC_MODE_UNIFORM) {
    const float2 c = tb.cff[k], iv = tb.iff[k];
    const ff2 zl = ff_add(ff_add(z, ff2{-c.x, -c.y}), ff2{-tb.lo[k], 0.f});
    const ff2 u = ff_mul(zl, ff2{iv.x, iv.y});
    const float q = ff_rint(u);
    const int qmax = tb.qp[k].x;
    codes_s[tt * ks + kp] = (uint8_t)(int)fminf(fmaxf(q, 0.f), (float)qmax);
    if (tau > 0.f)
      atomicMax(&cnt[3], (unsigned long long)__float_as_uint(fabsf(uf - u.hi) / tau));
    return;
  }
  const ff2 nrm = ff_sqrt(xx);
  if (norm_entry) {
    side_s[tt] = ff_to_half(nrm);
    atomicAdd(nside, 1u);
    return;
  }
  // nearest centroid, ties to the lower one: the number of exact midpoints m
  // (double-float, from the fp32 centroids) with m ||x|| < z; ||x|| = 0: u = 0
  const bool zero = nrm.hi == 0.f;
  int lo_i = 0, hi_i = p.cb_levels - 1;
  while (lo_i < hi_i) {
    const int mid = (lo_i + hi_i) >> 1;
    float ms, me;
    two_sum(cb_s[mid], cb_s[mid + 1], ms, me);
    const ff2 m{0.5f * ms, 0.5f * me};
    const bool below = zero ? m.hi < 0.f : ff_less(ff_mul(m, nrm), z);
    if (below) lo_i = mid + 1; else hi_i = mid;
  }
  codes_s[tt * ks + kp] = (uint8_t)lo_i;
  if (tau > 0.f && !zero)
    atomicMax(&cnt[3], (unsigned long long)__float_as_uint(fabsf(uf - z.hi / nrm.hi) / tau));
}

// Uniform fast path: u = (z - mean . V_k - lo) / step as one fma of the
// table's fused constants and the code; `near` flags a rounding boundary
// within the bound tau of u (host derivation in append_ws_table; tau holds for
// |u| <= qmax + 1, the range of the interior boundaries).  With `exact` the
// boundary is the nearest interior one (a first pass may flag outer ones too).
template <bool EXACT>
__device__ __forceinline__ int fast_uniform(const Tab& tb, int k, int qmax, float z, float nx,
                                            float& u, float& tau, bool& near) {
  const float4 q = tb.q4[k];
  u = fmaf(z, q.x, q.y);
  tau = fmaf(q.z, nx, q.w);
  // the interior boundary nearest u (0.5 .. qmax - 0.5); a first pass may
  // take the nearest half-integer, never farther than that one, so it flags a
  // superset (checked again with `exact`)
  const float hb0 = floorf(u) + 0.5f;
  const float hb = EXACT ? fminf(fmaxf(hb0, 0.5f), (float)qmax - 0.5f) : hb0;
  near = fabsf(u - hb) <= tau;
  return min(max(__float2int_rn(u), 0), qmax);
}

// The packed bytes of 32 consecutive W-bit codes (in: 32 code bytes as 8
// words, LSB-first) as W 32-bit words, LSB-first.
template <int W>
__device__ __forceinline__ void pack32(const uint32_t (&in)[8], uint32_t (&out)[W]) {
  uint64_t acc = 0;
  int nb = 0, o = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    acc |= (uint64_t)((in[j >> 2] >> (8 * (j & 3))) & 0xffu) << nb;
    nb += W;
    if (nb >= 32) {
      out[o++] = (uint32_t)acc;
      acc >>= 32;
      nb -= 32;
    }
  }
}

// Codebook rows (one segment of D codes, D a multiple of 32): one thread per
// (token, 32 codes), 8-byte loads of the codes, W 4-byte stores of the bits to
// out (rows P bytes apart, 4-byte aligned).
template <int W>
__device__ __forceinline__ void pack_codebook(int qt, int n, int D, const unsigned char* codes_s,
                                              int ks, unsigned char* out_s, int P) {
  const int ng = D / 32;
  for (int item = qt; item < n * ng; item += kQThreads) {
    const int tt = item / ng, g4 = item - tt * ng;
    const uint2* src = reinterpret_cast<const uint2*>(codes_s + tt * ks + 32 * g4);
    uint32_t in[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint2 v = src[q];
      in[2 * q] = v.x;
      in[2 * q + 1] = v.y;
    }
    uint32_t out[W];
    pack32<W>(in, out);
    uint32_t* dst = reinterpret_cast<uint32_t*>(out_s + tt * P + 4 * W * g4);
#pragma unroll
    for (int q = 0; q < W; ++q) dst[q] = out[q];
  }
}

// Codebook fast path: u = z / ||x||, the nearest centroid by the fp32
// midpoints, and whether a midpoint lies within the bound tau of u's error:
// tau = T1_k + |u| e, T1_k = gamma ||V_k|| (1 + 1e-3)(1 + 1e-6) + 2^-22 max|c|
// (table) and e = eps_n (1 + 1e-6) + 2^-22 (the norm's relative error and the
// roundings of u and of |u - m|).  Up to 8 levels the 7 midpoints sit in
// registers (+inf past the last) and a 3-step bisection finds the code and the
// two bracketing midpoints at once.
__device__ __forceinline__ int fast_codebook(const Params& p, float t1, const float* mids_s,
                                             const float* mpad, float m3, const float (&mr)[7],
                                             float z, float rnx, float e_u, bool tiny, float& u,
                                             float& tau, bool& near) {
  const int L = p.cb_levels;
  u = z * rnx;  // rnx = 2^-s fl(1 / ||x||) (0 for a tiny ||x||): two roundings, as z 2^-s / ||x||
  int c = 0;
  float dmin;
  if (L <= 8) {
    // a 3-step bisection over the midpoints held in registers (mr = m_0 ..
    // m_6, +inf past the last: no dependent shared-memory loads), then the
    // bracketing midpoints mpad[c] < u <= mpad[c + 1] (mpad = [-inf, m_0 ..
    // m_6, +inf])
    const bool b2 = u > m3;
    const float ma = b2 ? mr[5] : mr[1];
    const bool b1 = u > ma;
    const float mb = b2 ? (b1 ? mr[6] : mr[4]) : (b1 ? mr[2] : mr[0]);
    c = (b2 ? 4 : 0) + (b1 ? 2 : 0) + (u > mb ? 1 : 0);
    dmin = fminf(u - mpad[c], mpad[c + 1] - u);
  } else {
    int hi_i = L - 1;
    while (c < hi_i) {
      const int mid = (c + hi_i) >> 1;
      if (mids_s[mid] < u) c = mid + 1; else hi_i = mid;
    }
    dmin = 3.4e38f;
    if (c > 0) dmin = fminf(dmin, fabsf(u - mids_s[c - 1]));
    if (c < L - 1) dmin = fminf(dmin, fabsf(u - mids_s[c]));
  }
  tau = tiny ? 0.f : fmaf(fabsf(u), e_u, t1);
  near = tiny || dmin <= tau;
  return c;
}

template <int MODE, bool BF16, int CW>
__global__ void __launch_bounds__(kThreadsWs, 1)
    append_ws_kernel(const Params p, const AppendWsArgs t, const __grid_constant__ CUtensorMap xmap,
                     const AppendArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t x_full[kMaxXS], x_empty[kMaxXS];
  __shared__ uint64_t acc_full[kMaxTS], acc_empty[kMaxTS];
  __shared__ uint64_t b_full[2], b_empty[2], done_bar;
  __shared__ XHdr hdr[kMaxXS];
  __shared__ uint32_t tmem_base;
  __shared__ unsigned qcount_g[kQG], nside_g[kQG];
  __shared__ volatile int abort_flag;

  constexpr int rpad = kNCB * CW;         // CW: components per thread
  constexpr int SB = CW < 16 ? CW : 16;  // components per TMEM read
  constexpr int QG = kQG;
  constexpr int kProdWarp = QG * kQWarps, kMmaWarp = kProdWarp + 1;
  constexpr int kThreads = kThreadsWs;
  const int D = p.D, r = p.r, nbox = D / 64;
  const int XS = t.n_x, TS = t.n_acc, NB = t.n_b;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int first = (int)((int64_t)t.total_tiles * blockIdx.x / G);
  const int m = (int)((int64_t)t.total_tiles * (blockIdx.x + 1) / G) - first;
  const int tps = t.tiles_per_slot;
  const size_t b_bytes = (size_t)t.npieces * rpad * D * 2;

  const size_t vt_bytes = t.vt_smem ? (size_t)r * D * 4 : 0;  // per group
  unsigned char* xst = smem;                                        // XS x (x tile, table)
  unsigned char* Bs = xst + (size_t)XS * t.x_stage;                 // NB x (B, V^T)
  unsigned char* grp0 = Bs + NB * b_bytes;                          // QG x group scratch
  float* vt0 = reinterpret_cast<float*>(grp0 + QG * ws_group_bytes(t.ks, t.pmax, t.nq));  // QG x V^T
  float* mids_s = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(vt0) + QG * vt_bytes);
  float* cb_s = mids_s + 256;                                       // [256]
  __shared__ float mpad[9];  // codebooks of <= 8 levels: -inf, the midpoints, +inf
  __shared__ unsigned long long cnt_s[4];  // this CTA's counters, added to p.counters at exit
  const int tab_off = nbox * 16384;                                 // table after the x boxes

  if (warp == kMmaWarp) tmem_alloc(&tmem_base, t.cols);
  if (tid == 0) {
    for (int i = 0; i < XS; ++i) { mbar_init(&x_full[i], 1); mbar_init(&x_empty[i], kQWarps); }
    for (int i = 0; i < TS; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], kQWarps); }
    for (int i = 0; i < 2; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
    mbar_init(&done_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
    for (int i = 0; i < kQG; ++i) qcount_g[i] = nside_g[i] = 0;
    for (int i = 0; i < 4; ++i) cnt_s[i] = 0ull;
  }
  if (MODE == KVC_MODE_CODEBOOK) {
    for (int j = tid; j < p.cb_levels - 1; j += kThreads) mids_s[j] = p.mids[j];
    if (tid < 9)
      mpad[tid] = tid == 0 ? -INFINITY : (tid < p.cb_levels ? p.mids[tid - 1] : INFINITY);
    for (int j = tid; j < p.cb_levels; j += kThreads) cb_s[j] = p.codebook[j];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr0 = tmem_base;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int slot = first / tps, blk = first % tps;
      // a slot's tables are read one slot ahead, off the critical path
      struct SlotInfo { int beta, P; long long pay, side; };
      auto info_of = [&](int sl) {
        SlotInfo si{0, 0, 0, 0};
        if (sl < p.n_slots) {
          si.beta = p.basis_of[sl];
          si.P = p.P[si.beta];
          si.pay = p.pay_off[sl];
          si.side = p.side_off[sl];
        }
        return si;
      };
      SlotInfo cur = info_of(slot), nxt = info_of(slot + 1);
      int beta = cur.beta;
      int cur_beta = -1, bslot = NB - 1, issued = 0;
      uint32_t bload[2] = {0u, 0u};
      Ring rx(XS);
      for (int i = 0; i < m; ++i, rx.next()) {
        const int s = rx.slot;
        // the quantiser of tile i - XS released this stage
        if (i >= XS && !wait_or_abort(&x_empty[s], rx.phase ^ 1u, t.wait_ns, &abort_flag)) { abort_flag = 1; break; }
        int first_use = 0;
        if (beta != cur_beta) {
          bslot = NB == 2 ? bslot ^ 1 : 0;
          if (bload[bslot] > 0 &&
              !wait_or_abort(&b_empty[bslot], (bload[bslot] - 1) & 1, t.wait_ns, &abort_flag)) { abort_flag = 1; break; }
          mbar_arrive_expect_tx(&b_full[bslot], (uint32_t)b_bytes);
          bulk_load(Bs + bslot * b_bytes, t.B + (size_t)beta * (b_bytes / 2), (uint32_t)b_bytes,
                    &b_full[bslot]);
          ++bload[bslot];
          cur_beta = beta;
          first_use = 1;
        }
        const int64_t t0 = (int64_t)blk * kTile;
        unsigned char* dst = xst + (size_t)s * t.x_stage;
        hdr[s] = XHdr{(int)min((int64_t)kTile, a.T - t0), bslot | (first_use << 1), slot, cur.P,
                      beta, 0, (long long)(a.t_base + t0), cur.pay, cur.side};
        mbar_arrive_expect_tx(&x_full[s], (uint32_t)(nbox * 16384 + t.tab_bytes));
        const int bb = slot / p.H, hh = slot - bb * p.H;
        for (int bx = 0; bx < nbox; ++bx)
          tma_load_4d(dst + bx * 16384, &xmap, &x_full[s], bx * 64, (int)t0, hh, bb);
        bulk_load(dst + tab_off, t.tab + (size_t)beta * t.tab_bytes, (uint32_t)t.tab_bytes, &x_full[s]);
        ++issued;
        if (++blk == tps) {
          blk = 0;
          ++slot;
          cur = nxt;
          nxt = info_of(slot + 1);
          beta = cur.beta;
        }
      }
      // copies still in flight (after a time-out) land before the CTA exits
      for (int j = max(0, issued - XS); j < issued; ++j)
        mbar_wait_bounded(&x_full[j % XS], (j / XS) & 1, kWaitNs);
      for (int b2 = 0; b2 < 2; ++b2)
        if (bload[b2]) mbar_wait_bounded(&b_full[b2], (bload[b2] - 1) & 1, kWaitNs);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const int ncols = t.npieces * rpad;
      const bool stacked = ncols <= 256;  // one chain with the pieces along N
      const uint32_t idesc = idesc_f16(kTile, stacked ? ncols : rpad, BF16 ? 1 : 0);
      const uint32_t sbo = (uint32_t)(D / 8) * 128;
      uint32_t buse[2] = {0u, 0u};
      Ring rx(XS), rt(TS);
      for (int i = 0; i < m; ++i, rx.next(), rt.next()) {
        const int s = rx.slot, acc = rt.slot;
        if (!wait_or_abort(&x_full[s], rx.phase, t.wait_ns, &abort_flag)) { abort_flag = 1; break; }
        const int info = hdr[s].info, bs = info & 1;
        if (info & 2) {  // first tile on a newly loaded B: the other buffer is free when
          if (i > 0) umma_commit(&b_empty[NB == 2 ? bs ^ 1 : 0]);  // the MMAs issued so far finish
          if (!wait_or_abort(&b_full[bs], buse[bs] & 1, t.wait_ns, &abort_flag)) { abort_flag = 1; break; }
          ++buse[bs];
        }
        // the quantiser of tile i - TS released this accumulator
        if (i >= TS && !wait_or_abort(&acc_empty[acc], rt.phase ^ 1u, t.wait_ns, &abort_flag)) { abort_flag = 1; break; }
        tc_fence_after();
        const uint32_t xa = smem_u32(xst + (size_t)s * t.x_stage);
        const uint32_t b0 = smem_u32(Bs + bs * b_bytes);
        const uint32_t d0 = taddr0 + acc * t.acc_stride;
        for (int pc = 0; pc < (stacked ? 1 : t.npieces); ++pc)
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t ad = desc_kmajor_sw128(xa + (ks >> 2) * 16384 + (ks & 3) * 32);
            const uint64_t bd = desc_kmajor_noswizzle(b0 + pc * (rpad / 8) * sbo + ks * 256, 128, sbo);
            umma_f16(d0 + pc * rpad, ad, bd, idesc, ks > 0 ? 1u : 0u);
          }
        umma_commit(&acc_full[acc]);
      }
      umma_commit(&done_bar);  // TMEM is released only after every MMA has finished
      mbar_wait_bounded(&done_bar, 0, kWaitNs);
    }
  } else {
    // ------------------------------------------------------------ quantiser
    const int g = warp / kQWarps, wq = warp - g * kQWarps, qt = tid - g * kQThreads;
    const int quarter = wq & 3, cblk = wq >> 2, row = quarter * 32 + lane;
    const int qbar = kQBar + g;
    unsigned char* gbase = grp0 + (size_t)g * ws_group_bytes(t.ks, t.pmax, t.nq);
    unsigned char* codes_s = gbase;                                   // [128][ks] chunk-aligned
    unsigned char* out_s = codes_s + (size_t)kTile * t.ks;            // [128][P] packed rows
    uint32_t* queue = reinterpret_cast<uint32_t*>(out_s + ((kTile * t.pmax + 16 + 15) & ~15));
    float2* aux = reinterpret_cast<float2*>(queue + t.nq);
    float* nsq_s = reinterpret_cast<float*>(aux + t.nq);              // [2][128]
    __half* side_s = reinterpret_cast<__half*>(nsq_s + kNCB * kTile); // [128]
    unsigned& qcount = qcount_g[g];
    unsigned& nside = nside_g[g];
    float* vt_s = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(vt0) + g * vt_bytes);
    int vt_beta = -1;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int ks = t.ks;
    const float kU = 5.9604644775390625e-08f;
    const float eps_n = 0.5f * ((D + 2) * kU) / (1.f - (D + 2) * kU) + 2.f * kU;
    const float e_u = (eps_n * (1.f + 1e-6f) + 4.f * kU) * (1.f + 1e-6f);  // |u| term of tau
    const float m3 = MODE == KVC_MODE_CODEBOOK ? mpad[4] : 0.f;  // the first bisection step
    float mr[7];  // the midpoints m_0 .. m_6 (+inf past the last) in registers
#pragma unroll
    for (int q = 0; q < 7; ++q) mr[q] = MODE == KVC_MODE_CODEBOOK ? mpad[q + 1] : 0.f;
    Ring rx(XS), rt(TS);
    for (int j = 0; j < g; ++j) { rx.next(); rt.next(); }
    for (int i = g; i < m; i += QG) {
      if (i > g)
        for (int j = 0; j < QG; ++j) { rx.next(); rt.next(); }
      const int s = rx.slot, acc = rt.slot;
      bool late = !wait_or_abort(&x_full[s], rx.phase, t.wait_ns, &abort_flag);
      late = late || !wait_or_abort(&acc_full[acc], rt.phase, t.wait_ns, &abort_flag);
      const unsigned char* xs = xst + (size_t)s * t.x_stage;
      const Tab tb(xs + tab_off, rpad);
      const float t1 = MODE == KVC_MODE_CODEBOOK ? tb.q4[0].z : 0.f;  // the codebook bound's base
      const XHdr hd = hdr[s];
      const int n = hd.n;
      // V^T for the re-decision: the group's copy (refreshed when the basis
      // changes; B1 below publishes it) or global memory
      const float* Vt = p.Vt + (size_t)hd.beta * r * D;
      if (t.vt_smem) {
        if (hd.beta != vt_beta) {
          const float4* src = reinterpret_cast<const float4*>(Vt);
          float4* dst = reinterpret_cast<float4*>(vt_s);
          for (int e = qt; e < r * D / 4; e += kQThreads) dst[e] = src[e];
          vt_beta = hd.beta;
        }
        Vt = vt_s;
      }
      // partial ||x||^2 over this warp's share of the row
      {
        float sq = 0.f;
        const int c0 = cblk * (D / kNCB);
        for (int c = c0; c < c0 + D / kNCB; c += 8) {
          const uint4 v = *reinterpret_cast<const uint4*>(
              xs + (c >> 6) * 16384 + row * 128 + ((((c & 63) >> 3) ^ (row & 7)) << 4));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float e0, e1;
            if (BF16) {
              e0 = __uint_as_float(w4[q] << 16);
              e1 = __uint_as_float(w4[q] & 0xffff0000u);
            } else {
              e0 = __half2float(__ushort_as_half((uint16_t)(w4[q] & 0xffff)));
              e1 = __half2float(__ushort_as_half((uint16_t)(w4[q] >> 16)));
            }
            sq = fmaf(e0, e0, sq);
            sq = fmaf(e1, e1, sq);
          }
        }
        nsq_s[cblk * kTile + row] = sq;
      }
      // B1: norms complete; the previous tile's queue and staging are done with
      if (named_bar_or(qbar, kQThreads, late || abort_flag)) { abort_flag = 1; break; }
      // the first tile on a new B buffer: the other buffer's last reader was the
      // previous tile, finished now
      float nsq = nsq_s[row];
#pragma unroll
      for (int cb = 1; cb < kNCB; ++cb) nsq += nsq_s[cb * kTile + row];
      const float nx = sqrtf(nsq);
      const bool tiny = MODE == KVC_MODE_CODEBOOK && nx < 1e-18f;
      const float rnx = MODE == KVC_MODE_CODEBOOK && !tiny ? t.inv_scale * (1.f / nx) : 0.f;
      const bool live = row < n;
      unsigned char* crow = codes_s + row * ks;
      // components in sub-blocks of SB: z = hi + (mid + lo) from TMEM, the
      // fast-path codes, a mask of the ones near a boundary
      tc_fence_after();
      const uint32_t la0 = taddr0 + acc * t.acc_stride + lane_off + cblk * CW;
#pragma unroll(CW <= 16 ? CW / SB : 1)  // wide ranks: one sub-block of code, not CW / SB
      for (int sb = 0; sb < CW / SB; ++sb) {
        float z[SB];
        {
          const uint32_t la = la0 + sb * SB;
          uint32_t rr[SB];
#pragma unroll
          for (int j = 0; j < SB; ++j) z[j] = 0.f;
          if (t.npieces == 2) {  // both pieces loaded before one wait
            uint32_t r1[SB];
            tmem_ld_n<SB>(la + rpad, r1);
            tmem_ld_n<SB>(la, rr);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < SB; ++j) z[j] = __uint_as_float(rr[j]) + __uint_as_float(r1[j]);
          } else {
          for (int pc = t.npieces - 1; pc >= 1; --pc) {
            tmem_ld_n<SB>(la + pc * rpad, rr);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < SB; ++j) z[j] += __uint_as_float(rr[j]);
          }
          tmem_ld_n<SB>(la, rr);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < SB; ++j) z[j] = __uint_as_float(rr[j]) + z[j];
          }
        }
        if (!live) continue;
        uint32_t nmask = 0;
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          const int k = cblk * CW + sb * SB + j;  // < rpad; components past r are not kept
          // position (not kept: the row's scratch byte) and qmax; a codebook's
          // one segment keeps the components in order from position 0, and its
          // staging row holds rpad codes (k >= r lands past the packed ones)
          int pos = MODE == KVC_MODE_CODEBOOK ? k : (k < r ? k : ks - 1), qmax = 0;
          if (MODE == KVC_MODE_UNIFORM) {
            const int2 qp = tb.qp[k];
            qmax = qp.x;
            pos = qp.y;
          }
          float uf, tf;
          bool near;
          const int code = MODE == KVC_MODE_UNIFORM
                               ? fast_uniform<false>(tb, k, qmax, z[j], nx, uf, tf, near)
                               : fast_codebook(p, t1, mids_s, mpad, m3, mr, z[j], rnx, e_u, tiny, uf,
                                               tf, near);
          crow[pos] = (uint8_t)code;
          nmask |= (uint32_t)near << j;
        }
        // queue the near ones (rare); past the queue's end they are decided
        // below, one at a time, by their own thread
        uint32_t ovf = 0;
        if (nmask) {
#pragma unroll
          for (int j = 0; j < SB; ++j) {
            if (!((nmask >> j) & 1u)) continue;
            const int k = cblk * CW + sb * SB + j;
            float uf, tf;
            bool near;
            if (MODE == KVC_MODE_UNIFORM) {
              fast_uniform<true>(tb, k, tb.qp[k].x, z[j], nx, uf, tf, near);
              if (!near) continue;  // an outer boundary: the clamped code is certain
            } else {
              fast_codebook(p, t1, mids_s, mpad, m3, mr, z[j], rnx, e_u, tiny, uf, tf, near);
            }
            const unsigned q = atomicAdd(&qcount, 1u);
            if (q < (unsigned)t.nq) {
              queue[q] = ((uint32_t)row << 16) | (uint32_t)k;
              aux[q] = make_float2(uf, tf);
            } else {
              ovf |= 1u << j;
            }
          }
        }
        for (; ovf; ovf &= ovf - 1) {
          const int k = cblk * CW + sb * SB + (__ffs(ovf) - 1);
          refine_ws<MODE, BF16, false>(p, tb, Vt, cb_s, xs, codes_s, ks, side_s, &nside, cnt_s, row, k, 0,
                                       0.f, 0.f);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (live) {
        if (MODE == KVC_MODE_CODEBOOK && cblk == 0) {
          if (tiny || !same_half(nx * (1.f - eps_n), nx * (1.f + eps_n))) {
            const unsigned q = atomicAdd(&qcount, 1u);
            if (q < (unsigned)t.nq) {
              queue[q] = ((uint32_t)row << 16) | kNormEntry;
              aux[q] = make_float2(0.f, 0.f);
            } else {
              refine_ws<MODE, BF16, false>(p, tb, Vt, cb_s, xs, codes_s, ks, side_s, &nside, cnt_s, row,
                                           (int)kNormEntry, 0, 0.f, 0.f);
            }
          } else {
            side_s[row] = __float2half_rn(nx);
          }
        }
      }
      named_bar_sync(qbar, kQThreads);  // B2: fast-path codes and the queue complete
      const unsigned nq = qcount;
      {  // entries per warp at a time: codebook tiles queue few (two of sixteen
         // lanes each: shorter chains), uniform tiles about twenty (four of eight
         // lanes each: one round)
        constexpr int GL = MODE == KVC_MODE_UNIFORM ? 8 : 16, PER = 32 / GL;
        const unsigned nqe = min(nq, (unsigned)t.nq);
        for (unsigned e0 = wq * PER; e0 < nqe; e0 += kQWarps * PER) {
          const unsigned e = e0 + lane / GL;
          const bool act = e < nqe;
          const uint32_t ent = queue[act ? e : e0];
          const float2 ax = aux[act ? e : e0];
          refine_group<MODE, BF16, GL>(p, tb, Vt, cb_s, xs, codes_s, ks, side_s, &nside, cnt_s,
                                       (int)(ent >> 16), (int)(ent & 0xffffu), lane & (GL - 1),
                                       act, ax.x, ax.y);
        }
      }
      named_bar_sync(qbar, kQThreads);  // B3: every code decided
      if (qt == 0) {
        if (nq > nside) atomicAdd(&cnt_s[0], (unsigned long long)(nq - nside));
        if (nside) atomicAdd(&cnt_s[1], (unsigned long long)nside);
        if (hd.slot == 0) atomicAdd(&cnt_s[2], (unsigned long long)n);
      }
      const int P = hd.P;
      if (MODE == KVC_MODE_CODEBOOK && D % 32 == 0) {
        // a codebook's single segment, 32 codes at a time, written straight to
        // the store: every re-decision is done (B3), so the x stage is free and
        // no staging or second barrier is needed
        __syncwarp();
        if (lane == 0) mbar_arrive(&x_empty[s]);
        unsigned char* dst = p.store + hd.pay + hd.row0 * P;
        switch (p.cb_bits) {
          case 1: pack_codebook<1>(qt, n, D, codes_s, ks, dst, P); break;
          case 2: pack_codebook<2>(qt, n, D, codes_s, ks, dst, P); break;
          case 3: pack_codebook<3>(qt, n, D, codes_s, ks, dst, P); break;
          case 4: pack_codebook<4>(qt, n, D, codes_s, ks, dst, P); break;
          default: pack_codebook<8>(qt, n, D, codes_s, ks, dst, P); break;
        }
      } else {
      // pack: one thread per (token, 8-code chunk) -> w bytes, LSB-first
      for (int item = qt; item < kTile * 32; item += kQThreads) {
        const int tt = item & (kTile - 1), c = item >> 7;
        const uint32_t ent = tb.chunk[c];
        if (!(ent >> 31)) break;  // chunks are contiguous from 0: c is past the last one
        if (tt >= n) continue;
        const int wd = (int)((ent >> 16) & 0xfu), nc = (int)((ent >> 20) & 7u) + 1;
        uint64_t v = *reinterpret_cast<const uint64_t*>(codes_s + tt * ks + c * 8);
        if (nc < 8) v &= (1ull << (8 * nc)) - 1ull;
        uint64_t packed = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) packed |= ((v >> (8 * j)) & 0xffull) << (wd * j);
        unsigned char* o = out_s + tt * P + (int)(ent & 0xffffu);
        const int nbytes = (nc * wd + 7) >> 3;
        for (int j = 0; j < nbytes; ++j) o[j] = (unsigned char)(packed >> (8 * j));
      }
      named_bar_sync(qbar, kQThreads);  // B4: packed rows staged; the stage (x, table) is free
      __syncwarp();
      if (lane == 0) mbar_arrive(&x_empty[s]);
      unsigned char* dst = p.store + hd.pay + hd.row0 * P;
      if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {  // 16-byte copies, then the tail
        const int nv = (n * P) >> 4;
        for (int v = qt; v < nv; v += kQThreads)
          reinterpret_cast<uint4*>(dst)[v] = reinterpret_cast<const uint4*>(out_s)[v];
        for (int idx = 16 * nv + qt; idx < n * P; idx += kQThreads) dst[idx] = out_s[idx];
      } else {
        for (int idx = qt; idx < n * P; idx += kQThreads) dst[idx] = out_s[idx];
      }
      }
      if (MODE == KVC_MODE_CODEBOOK && qt < n)
        reinterpret_cast<__half*>(p.store + hd.side)[hd.row0 + qt] = side_s[qt];
      if (qt == 0) {  // the next tile starts with an empty queue (read above, before B3)
        qcount = 0;
        nside = 0;
      }
    }
  }
  __syncthreads();
  if (abort_flag && tid == 0) atomicCAS(p.err, 0, kErrTimeout);
  if (tid < 3 && cnt_s[tid]) atomicAdd(&p.counters[tid], cnt_s[tid]);  // once per CTA
  if (tid == 3 && cnt_s[3]) atomicMax(&p.counters[3], cnt_s[3]);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(taddr0, t.cols);
  }
}

using WsKernel = void (*)(const Params, const AppendWsArgs, const CUtensorMap, const AppendArgs);

template <int MODE, bool BF16>
WsKernel ws_for(int rpad) {  // CW = rpad / kNCB components per thread
  switch (rpad) {
    case 16: return append_ws_kernel<MODE, BF16, 16 / kNCB>;
    case 32: return append_ws_kernel<MODE, BF16, 32 / kNCB>;
    case 64: return append_ws_kernel<MODE, BF16, 64 / kNCB>;
    default: return append_ws_kernel<MODE, BF16, 128 / kNCB>;
  }
}

WsKernel ws_kernel_for(int mode, int bf16, int rpad) {
  if (mode == KVC_MODE_UNIFORM)
    return bf16 ? ws_for<KVC_MODE_UNIFORM, true>(rpad) : ws_for<KVC_MODE_UNIFORM, false>(rpad);
  return bf16 ? ws_for<KVC_MODE_CODEBOOK, true>(rpad) : ws_for<KVC_MODE_CODEBOOK, false>(rpad);
}

}  // namespace

size_t append_ws_tab_bytes(int rpad) { return ((size_t)rpad * 48 + 128 + 15) & ~size_t(15); }

int append_ws_chunks(const Geo& g, int b) {
  int nch = 0;
  for (int sg = 0; sg < kMaxSeg; ++sg) {
    const int32_t* e = &g.seg[((size_t)b * kMaxSeg + sg) * 4];
    if (!e[3]) break;
    nch += (e[3] + 7) / 8;
  }
  return nch;
}

namespace {
float round_up_f(double v) {  // the smallest float >= v
  float f = (float)v;
  if ((double)f < v) f = std::nextafter(f, INFINITY);
  return f;
}
}  // namespace

int append_ws_table(const Geo& g, const kvc_layer_desc& d, int rpad, const double* c64,
                    double inv_scale, double gamma, int ks, int b, unsigned char* out) {
  const int r = g.r, D = d.D;
  float4* q4 = reinterpret_cast<float4*>(out);
  float2* cff = reinterpret_cast<float2*>(q4 + rpad);
  float2* iff = cff + rpad;
  float* lo = reinterpret_cast<float*>(iff + rpad);
  float* vn = lo + rpad;
  int2* qp = reinterpret_cast<int2*>(vn + rpad);
  uint32_t* chunk = reinterpret_cast<uint32_t*>(qp + rpad);
  double vmax = 0.0;  // the largest ||V_k||, rounded up as below
  for (int k = 0; k < r; ++k) {
    double ss = 0.0;
    for (int i = 0; i < D; ++i) {
      const double v = d.V[((size_t)b * D + i) * r + k];
      ss += v * v;
    }
    vmax = std::max(vmax, (double)std::nextafter((float)std::sqrt(ss), INFINITY));
  }
  for (int k = 0; k < rpad; ++k) {
    const bool in = k < r;
    const size_t bk = (size_t)b * r + k;
    const bool q = in && d.mode == KVC_MODE_UNIFORM && g.bits[bk] > 0;
    double ss = 0.0;  // ||V_k|| rounded up, as the parameter block's
    for (int i = 0; in && i < D; ++i) {
      const double v = d.V[((size_t)b * D + i) * r + k];
      ss += v * v;
    }
    vn[k] = in ? std::nextafter((float)std::sqrt(ss), INFINITY) : 0.f;
    const auto pair = [](double v) {  // v as hi + lo, two floats
      const float hi = (float)v;
      return make_float2(hi, (float)(v - (double)hi));
    };
    cff[k] = pair(in ? c64[bk] : 0.0);
    lo[k] = q ? d.qmin[bk] : 0.f;
    iff[k] = pair(q ? 1.0 / (double)d.qstep[bk] : 0.0);
    q4[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q) {
      // u = fma(z_tc, A, Bc) with A, Bc rounded once from double.  |u - u_exact|
      // <= [gamma ||x|| ||V_k|| (tensor-core accumulation) + 2^-24 |z| (A) ]
      //    / step + 2^-24 |c + lo| / step (Bc) + 2^-24 |u| (fma), |z| <= ||x|| ||V_k||;
      // T1, T2 carry twice that, ||x|| a 1e-3 margin, the kernel 2^-22 (|u| + 1).
      const double st = (double)d.qstep[bk];
      q4[k].x = (float)(inv_scale / st);
      q4[k].y = (float)(-(c64[bk] + (double)d.qmin[bk]) / st);
      q4[k].z = round_up_f((double)vn[k] / st * (gamma + std::ldexp(1.0, -23)) *
                           (1.0 + std::ldexp(1.0, -20)) * (1.0 + 1e-3));
      // + 2^-22 (|u| + 1) for |u| <= qmax + 1 (interior boundaries only)
      const int qm = (1 << g.bits[bk]) - 1;
      q4[k].w = round_up_f((std::fabs(c64[bk]) + std::fabs((double)d.qmin[bk])) / st *
                               std::ldexp(1.0, -23) +
                           std::ldexp(1.0, -22) * (qm + 2));
    }
    if (in && d.mode == KVC_MODE_CODEBOOK) {
      // one bound for every component (the quantiser reads it once per tile):
      // the basis' largest ||V_k||
      double cmax = 0.0;
      for (int j = 0; j < g.cb_levels; ++j) cmax = std::max(cmax, std::fabs((double)d.codebook[j]));
      q4[k].z = round_up_f(gamma * vmax * (1.0 + 1e-3) * (1.0 + 1e-6) + std::ldexp(1.0, -22) * cmax);
    }
    const int width = in ? g.bits[bk] : 0;
    qp[k] = make_int2(d.mode == KVC_MODE_UNIFORM && width ? (1 << width) - 1 : 0, ks - 1);
  }
  // chunk-aligned positions: segment s (packed order) starts on a chunk
  int nch = 0;
  for (int sg = 0; sg < kMaxSeg; ++sg) {
    const int32_t* e = &g.seg[((size_t)b * kMaxSeg + sg) * 4];
    if (!e[3]) break;
    for (int mm = 0; mm < e[3]; ++mm) {
      const int k = g.order[(size_t)b * r + e[2] + mm];
      qp[k].y = nch * 8 + mm;
    }
    for (int ci = 0; ci * 8 < e[3]; ++ci) {
      if (nch == 32) return -1;
      const int nc = std::min(8, e[3] - ci * 8);
      chunk[nch++] = (uint32_t)(e[0] + e[1] * ci) | ((uint32_t)e[1] << 16) |
                     ((uint32_t)(nc - 1) << 20) | (1u << 31);
    }
  }
  for (int j = nch; j < 32; ++j) chunk[j] = 0u;
  return nch;
}

size_t append_ws_plan(int D, int r, int rpad, int npieces, int pmax, int max_chunks, int n_bases,
                      bool direct, AppendWsShape* sh) {
  AppendWsShape z;
  // codebook rows are packed straight to the store (no staging of packed
  // rows), and their tiles queue few near codes: a short queue (past its end
  // a code is decided by its own thread) leaves room for a third x stage
  z.pmax = direct ? 0 : pmax;
  z.nq = direct ? 128 : kQueue;
  const int ncols = npieces * rpad;
  z.acc_stride = (ncols + 31) / 32 * 32;
  z.n_acc = std::min(kMaxTS, 512 / z.acc_stride);
  if (z.n_acc < 1 || max_chunks < 1 || max_chunks > 32) return 0;
  int cols = 32;
  while (cols < z.n_acc * z.acc_stride) cols *= 2;
  z.cols = cols;
  z.tab_bytes = (int)append_ws_tab_bytes(rpad);
  z.x_stage = ((D / 64) * 16384 + z.tab_bytes + 1023) / 1024 * 1024;
  z.n_b = n_bases > 1 ? 2 : 1;
  // the extra 8 bytes spread the rows over the banks; a codebook row holds
  // rpad codes (the components past r land beyond the packed ones)
  z.ks = std::max(max_chunks * 8, direct ? rpad : 0) + 8;
  const size_t limit = 226 * 1024;
  for (int vt = 1; vt >= 0; --vt) {  // the groups' V^T copies where they fit
    const size_t fixed = 1024 + (size_t)z.n_b * ncols * D * 2 +
                         (size_t)kQG * (ws_group_bytes(z.ks, z.pmax, z.nq) + (vt ? (size_t)r * D * 4 : 0)) +
                         2 * 256 * 4;
    for (int xs = kMaxXS; xs >= (vt ? 3 : 2); --xs)
      if (fixed + (size_t)xs * z.x_stage <= limit) {
        z.n_x = xs;
        z.vt_smem = vt;
        *sh = z;
        return fixed + (size_t)xs * z.x_stage;
      }
  }
  return 0;
}

cudaError_t launch_append_ws(const TcPlan& plan, const Params& p, const AppendArgs& a,
                             const CUtensorMap& xmap, uint64_t wait_ns, cudaStream_t s, int* nk) {
  WsKernel k = ws_kernel_for(p.mode, plan.app_bf16, plan.app_rpad);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)plan.ws_smem);
  if (e != cudaSuccess) return e;
  const int tiles = (int)((a.T + kTile - 1) / kTile);
  const int total = tiles * p.n_slots;
  const int grid = std::min(total, sm_count());
  const AppendWsShape& sh = plan.ws;
  const AppendWsArgs t{plan.appB,    plan.c64,     plan.wsTab,   plan.app_rpad,      plan.app_pieces,
                       sh.acc_stride, sh.cols,      sh.n_acc,     sh.n_x,             sh.n_b,
                       sh.x_stage,    sh.tab_bytes, sh.pmax,      sh.ks,   sh.nq,     sh.vt_smem,
                       plan.app_inv_scale, plan.app_gamma, tiles, total, wait_ns};
  k<<<(unsigned)grid, kThreadsWs, plan.ws_smem, s>>>(p, t, xmap, a);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
