// On-device prefill fit of the uniform (KVTC-style) mode: for every (batch,
// head) slot, the local PCA of its first S_fit rows, the dynamic-programming
// bit allocation and the frozen per-component minimum and step (kvtc_cache
// page: module docstring "Design", prefill step 1, and
// KVTCKVCache.update_and_fetch, which fits the PCA basis of all B*H rows in
// one batched call; the module docstring's DP allocation over the analytic
// distortion proxy; _TensorKVTC._requantize, where quantize_component gives
// each kept component a minimum and a scale).  The arithmetic is float64
// until the fitted parameters are rounded to fp32.
//
// Four launches, one CTA per slot each:
//   fit_cov_kernel     mean and covariance C = (X - mean)^T (X - mean) / S
//   fit_jacobi_kernel  C = U diag(lambda) U^T by cyclic Jacobi rotations in
//                      round-robin order (D / 2 disjoint rotations a step,
//                      D - 1 steps a sweep), C in shared memory
//   fit_select_kernel  eigenpairs ordered largest first (ties by index),
//                      each vector's sign fixed so that its first
//                      largest-magnitude entry is positive; V and mean in fp32
//   fit_alloc_kernel   the DP allocation (products and sums rounded once
//                      each, ties to the smaller width), then
//                      lo = min z, step = max((max z - lo) / (2^b - 1), 1e-8)
//                      over z = (x - mean32) V32 of the fit rows
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "kvc_internal.h"

namespace kvc {

namespace {

constexpr int kFitThreads = 256;
constexpr int kMaxSweeps = 40;

__device__ __forceinline__ double load_x(const void* x, int dt, int64_t off) {
  if (dt == KVC_F32) return (double)static_cast<const float*>(x)[off];
  const uint16_t h = static_cast<const uint16_t*>(x)[off];
  if (dt == KVC_F16) return (double)__half2float(__ushort_as_half(h));
  return (double)__bfloat162float(__ushort_as_bfloat16(h));
}

__device__ __forceinline__ int64_t row_off(const FitArgs& f, int slot, int64_t t) {
  const int b = slot / f.H, h = slot - b * f.H;
  return (int64_t)b * f.sb + (int64_t)h * f.sh + t * f.st;
}

// mean and covariance [D][D] of the slot's fit rows.  Thread (bi, bj), bi <= bj,
// owns the 8 x 8 block of C at rows 8 bi, columns 8 bj, sums it over the rows
// in order and writes it and its mirror image (C is exactly symmetric).
__global__ void __launch_bounds__(kFitThreads) fit_cov_kernel(const FitArgs f) {
  extern __shared__ double xs[];  // [32][D] centred rows of one pass
  __shared__ double mu[kFitMaxD];
  const int slot = blockIdx.x, tid = threadIdx.x, D = f.D;
  double* C = f.cov + (size_t)slot * D * D;
  for (int c = tid; c < D; c += kFitThreads) {
    double s = 0.0;
    for (int64_t t = 0; t < f.S; ++t) s += load_x(f.x, f.dtype, row_off(f, slot, t) + c);
    mu[c] = s / (double)f.S;
    f.mean64[(size_t)slot * D + c] = mu[c];
  }
  __syncthreads();
  const int nb = D / 8;
  const int bi = tid / 16, bj = tid % 16;
  const bool owns = bi <= bj && bj < nb;
  double acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0;
  for (int64_t t0 = 0; t0 < f.S; t0 += 32) {
    const int n = (int)min((int64_t)32, f.S - t0);
    __syncthreads();
    for (int e = tid; e < n * D; e += kFitThreads) {
      const int rr = e / D, c = e - rr * D;
      xs[rr * D + c] = load_x(f.x, f.dtype, row_off(f, slot, t0 + rr) + c) - mu[c];
    }
    __syncthreads();
    if (owns)
      for (int rr = 0; rr < n; ++rr) {
        double a[8], b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          a[i] = xs[rr * D + 8 * bi + i];
          b[i] = xs[rr * D + 8 * bj + i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = __dadd_rn(acc[i][j], __dmul_rn(a[i], b[j]));
      }
  }
  if (owns)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const double v = acc[i][j] / (double)f.S;
        C[(size_t)(8 * bi + i) * D + 8 * bj + j] = v;
        C[(size_t)(8 * bj + j) * D + 8 * bi + i] = v;
      }
}

// Cyclic Jacobi on A = C in shared memory, U = product of the rotations in
// global memory.  Pair i of step s couples positions i and D - 1 - i of a
// round-robin ordering in which index 0 stays and the others move by one
// place each step, so a sweep meets every pair once.  A rotation is skipped
// where |a_pq| is below 2^-53 sqrt(|a_pp a_qq|) or 2^-60 ||C||_F; the
// iteration stops after a sweep without a rotation (or after kMaxSweeps).
__global__ void __launch_bounds__(kFitThreads) fit_jacobi_kernel(const FitArgs f) {
  extern __shared__ double A[];  // [D][D]
  __shared__ double cs[kFitMaxD / 2][2];
  __shared__ int pq[kFitMaxD / 2][2];
  __shared__ double red[kFitThreads / 32];
  __shared__ double fro;
  __shared__ int rotations;
  const int slot = blockIdx.x, tid = threadIdx.x, n = f.D, np = n / 2;
  double* U = f.vec + (size_t)slot * n * n;
  const double* C = f.cov + (size_t)slot * n * n;
  double ss = 0.0;
  for (int e = tid; e < n * n; e += kFitThreads) {
    A[e] = C[e];
    ss += C[e] * C[e];
    U[e] = (e / n == e % n) ? 1.0 : 0.0;
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  if (tid == 0) {
    double s = 0.0;
    for (int w = 0; w < kFitThreads / 32; ++w) s += red[w];
    fro = sqrt(s);
  }
  __syncthreads();
  const double abs_floor = ldexp(fro, -60);
  for (int sweep = 0; sweep < kMaxSweeps; ++sweep) {
    if (tid == 0) rotations = 0;
    __syncthreads();
    for (int step = 0; step < n - 1; ++step) {
      if (tid < np) {
        const int k0 = tid, k1 = n - 1 - tid;
        int p = k0 == 0 ? 0 : 1 + (k0 - 1 + step) % (n - 1);
        int q = 1 + (k1 - 1 + step) % (n - 1);
        if (p > q) {
          const int t = p;
          p = q;
          q = t;
        }
        const double apq = A[p * n + q], app = A[p * n + p], aqq = A[q * n + q];
        double c = 1.0, s = 0.0;
        if (fabs(apq) > fmax(ldexp(sqrt(fabs(app * aqq)), -53), abs_floor)) {
          const double tau = (aqq - app) / (2.0 * apq);
          const double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
          c = 1.0 / sqrt(1.0 + t * t);
          s = t * c;
          atomicAdd(&rotations, 1);
        }
        cs[tid][0] = c;
        cs[tid][1] = s;
        pq[tid][0] = p;
        pq[tid][1] = q;
      }
      __syncthreads();
      // rows: A <- J^T A (lanes along a row)
      for (int e = tid; e < np * n; e += kFitThreads) {
        const int i = e / n, k = e - i * n;
        if (cs[i][1] == 0.0) continue;
        const int p = pq[i][0], q = pq[i][1];
        const double c = cs[i][0], s = cs[i][1];
        const double ap = A[p * n + k], aq = A[q * n + k];
        A[p * n + k] = c * ap - s * aq;
        A[q * n + k] = s * ap + c * aq;
      }
      __syncthreads();
      // columns: A <- A J (lanes across the pairs of one row); the entry the
      // rotation annihilates is set to zero rather than left at rounding level
      for (int e = tid; e < np * n; e += kFitThreads) {
        const int k = e / np, i = e - k * np;
        if (cs[i][1] == 0.0) continue;
        const int p = pq[i][0], q = pq[i][1];
        const double c = cs[i][0], s = cs[i][1];
        const double ap = A[k * n + p], aq = A[k * n + q];
        A[k * n + p] = k == q ? 0.0 : c * ap - s * aq;
        A[k * n + q] = k == p ? 0.0 : s * ap + c * aq;
      }
      // U <- U J, four elements' loads issued before their stores (the
      // elements of one step are distinct, so the batch cannot alias)
      for (int e0 = tid; e0 < np * n; e0 += 4 * kFitThreads) {
        double up[4], uq[4];
        int at_p[4], at_q[4], pi[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = e0 + j * kFitThreads;
          pi[j] = -1;
          if (e < np * n) {
            const int k = e / np, i = e - k * np;
            if (cs[i][1] != 0.0) {
              pi[j] = i;
              at_p[j] = k * n + pq[i][0];
              at_q[j] = k * n + pq[i][1];
              up[j] = U[at_p[j]];
              uq[j] = U[at_q[j]];
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (pi[j] >= 0) {
            const double c = cs[pi[j]][0], s = cs[pi[j]][1];
            U[at_p[j]] = c * up[j] - s * uq[j];
            U[at_q[j]] = s * up[j] + c * uq[j];
          }
      }
      __syncthreads();
    }
    if (rotations == 0) break;
    __syncthreads();  // every thread has read the count before it is reset
  }
  for (int i = tid; i < n; i += kFitThreads) f.lam[(size_t)slot * n + i] = A[i * n + i];
}

// Eigenpairs ordered largest eigenvalue first (ties by index); each kept
// vector's sign fixed so that its first largest-magnitude entry is positive.
__global__ void __launch_bounds__(kFitThreads) fit_select_kernel(const FitArgs f) {
  __shared__ int order[kFitMaxD];
  __shared__ double sgn[kFitMaxD];
  const int slot = blockIdx.x, tid = threadIdx.x, n = f.D;
  const double* lam = f.lam + (size_t)slot * n;
  const double* U = f.vec + (size_t)slot * n * n;
  for (int i = tid; i < n; i += kFitThreads) {
    int rank = 0;  // eigenvalues ahead of i: larger, or equal at a smaller index
    for (int j = 0; j < n; ++j) rank += lam[j] > lam[i] || (lam[j] == lam[i] && j < i);
    order[rank] = i;
  }
  __syncthreads();
  for (int k = tid; k < n; k += kFitThreads) {
    const int col = order[k];
    int piv = 0;
    double best = -1.0;
    for (int i = 0; i < n; ++i) {
      const double a = fabs(U[(size_t)i * n + col]);
      if (a > best) {
        best = a;
        piv = i;
      }
    }
    sgn[k] = U[(size_t)piv * n + col] < 0.0 ? -1.0 : 1.0;
    f.lam_sorted[(size_t)slot * n + k] = lam[col];
  }
  __syncthreads();
  for (int e = tid; e < n * f.r; e += kFitThreads) {
    const int i = e / f.r, k = e - i * f.r;
    f.V[(size_t)slot * n * f.r + e] = (float)(U[(size_t)i * n + order[k]] * sgn[k]);
  }
  for (int i = tid; i < n; i += kFitThreads)
    f.mean[(size_t)slot * n + i] = (float)f.mean64[(size_t)slot * n + i];
}

// DP allocation: minimise sum_k lam_k 2^(-2 b_k) over b_k in the choices with
// sum_k b_k <= budget.  cost[k][c] is the least distortion of components
// k .. r-1 with c bits free; a row is filled by all threads, one entry each,
// the allocation read forward by one thread (the smallest width wins a tie).
// Then the frozen minimum and step of every kept component.
__global__ void __launch_bounds__(kFitThreads) fit_alloc_kernel(const FitArgs f) {
  extern __shared__ double dyn_smem[];
  __shared__ int bits_s[kFitMaxD];
  const int slot = blockIdx.x, tid = threadIdx.x, r = f.r, D = f.D, W = f.budget + 1;
  const double* lam = f.lam_sorted + (size_t)slot * D;
  double* cost = f.dp + (size_t)slot * (r + 1) * W;
  for (int c = tid; c < W; c += kFitThreads) cost[(size_t)r * W + c] = 0.0;
  __syncthreads();
  for (int k = r - 1; k >= 0; --k) {
    double* ck = cost + (size_t)k * W;
    const double* cn = cost + (size_t)(k + 1) * W;
    for (int c = tid; c < W; c += kFitThreads) {
      double v = INFINITY;
      for (int ci = 0; ci < f.n_choices; ++ci) {
        const int b = f.choices[ci];
        if (b > c) break;
        v = fmin(v, __dadd_rn(__dmul_rn(lam[k], ldexp(1.0, -2 * b)), cn[c - b]));
      }
      ck[c] = v;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int free_bits = f.budget;
    for (int k = 0; k < r; ++k) {
      int best_b = f.choices[0];
      double best_v = INFINITY;
      for (int ci = 0; ci < f.n_choices; ++ci) {
        const int b = f.choices[ci];
        if (b > free_bits) break;
        const double v = __dadd_rn(__dmul_rn(lam[k], ldexp(1.0, -2 * b)),
                                   cost[(size_t)(k + 1) * W + free_bits - b]);
        if (v < best_v) {
          best_v = v;
          best_b = b;
        }
      }
      bits_s[k] = best_b;
      f.bits[(size_t)slot * r + k] = (uint8_t)best_b;
      free_bits -= best_b;
    }
  }
  __syncthreads();
  // z = (x - mean32) V32 of the fit rows, staged 32 rows at a time; thread
  // (g, k) takes component k of rows g, g + G, ... and keeps their min and max
  double* xs = dyn_smem;  // [32][D]
  __shared__ double lo_s[kFitThreads], hi_s[kFitThreads];
  const float* V = f.V + (size_t)slot * D * r;
  const float* m = f.mean + (size_t)slot * D;
  const int G = kFitThreads / r, k = tid % r, g = tid / r;
  const bool act = g < G && bits_s[k] > 0;
  double lo = INFINITY, hi = -INFINITY;
  for (int64_t t0 = 0; t0 < f.S; t0 += 32) {
    const int n = (int)min((int64_t)32, f.S - t0);
    __syncthreads();
    for (int e = tid; e < n * D; e += kFitThreads) {
      const int rr = e / D, c = e - rr * D;
      xs[rr * D + c] = __dadd_rn(load_x(f.x, f.dtype, row_off(f, slot, t0 + rr) + c), -(double)m[c]);
    }
    __syncthreads();
    if (act)
      for (int rr = g; rr < n; rr += G) {
        double z = 0.0;
        for (int i = 0; i < D; ++i) z = __dadd_rn(z, __dmul_rn(xs[rr * D + i], (double)V[(size_t)i * r + k]));
        lo = fmin(lo, z);
        hi = fmax(hi, z);
      }
  }
  lo_s[tid] = lo;
  hi_s[tid] = hi;
  __syncthreads();
  for (int kk = tid; kk < r; kk += kFitThreads) {
    const int b = bits_s[kk];
    float lo32 = 0.f, st32 = 0.f;
    if (b > 0) {
      double l = INFINITY, h = -INFINITY;
      for (int gg = 0; gg < G; ++gg) {
        l = fmin(l, lo_s[gg * r + kk]);
        h = fmax(h, hi_s[gg * r + kk]);
      }
      lo32 = (float)l;
      st32 = (float)fmax((h - l) / (ldexp(1.0, b) - 1.0), 1e-8);
    }
    f.qmin[(size_t)slot * r + kk] = lo32;
    f.qstep[(size_t)slot * r + kk] = st32;
  }
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

size_t fit_workspace_bytes(int n_slots, int D, int r, int budget) {
  return align256((size_t)n_slots * D * 8) * 3 +                 // mean64, lam, sorted lam
         align256((size_t)n_slots * D * D * 8) * 2 +             // covariance, vectors
         align256((size_t)n_slots * (r + 1) * (budget + 1) * 8);  // DP tables
}

cudaError_t launch_fit_uniform(FitArgs f, void* workspace, cudaStream_t s, int* nk) {
  const int ns = f.B * f.H, D = f.D;
  unsigned char* w = static_cast<unsigned char*>(workspace);
  auto take = [&](size_t bytes) {
    double* p = reinterpret_cast<double*>(w);
    w += align256(bytes);
    return p;
  };
  f.mean64 = take((size_t)ns * D * 8);
  f.lam = take((size_t)ns * D * 8);
  f.lam_sorted = take((size_t)ns * D * 8);
  f.cov = take((size_t)ns * D * D * 8);
  f.vec = take((size_t)ns * D * D * 8);
  f.dp = take((size_t)ns * (f.r + 1) * (f.budget + 1) * 8);
  if (f.lam_out) f.lam_sorted = f.lam_out;
  cudaError_t e;
  const size_t cov_smem = (size_t)32 * D * 8;
  const size_t jac_smem = (size_t)D * D * 8;
  if ((e = cudaFuncSetAttribute(fit_jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)jac_smem)) != cudaSuccess)
    return e;
  fit_cov_kernel<<<ns, kFitThreads, cov_smem, s>>>(f);
  ++*nk;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fit_jacobi_kernel<<<ns, kFitThreads, jac_smem, s>>>(f);
  ++*nk;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fit_select_kernel<<<ns, kFitThreads, 0, s>>>(f);
  ++*nk;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fit_alloc_kernel<<<ns, kFitThreads, cov_smem, s>>>(f);
  ++*nk;
  return cudaGetLastError();
}

}  // namespace kvc
