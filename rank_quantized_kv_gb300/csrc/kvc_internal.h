// Internal declarations shared by the host library and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int kMaxSeg = 5;        // widths 8, 4, 3, 2, 1
constexpr int kMaxRank = 1024;
constexpr int kMaxGroupSize = 32;

// Device error codes written to Params::err (first writer wins).
enum : int { kErrNone = 0, kErrTimeout = 1, kErrRange = 2 };

// Frozen per-layer parameters in kernel layouts.  Every pointer is device
// memory inside the layer's parameter block.  Passed by value to kernels.
struct Params {
  int mode, B, H, D, hpg, Hg, d_in, r, n_bases, n_slots;
  int in_dtype, out_dtype;
  int group_size, n_groups, cb_levels, cb_bits;
  int side_bytes;  // per token

  const float* V;         // [nb][d_in][r]
  const float* Vt;        // [nb][r][d_in]
  const float* mean;      // [nb][d_in] (zeros when absent)
  const float* lo;        // [nb][r]   UNIFORM
  const float* step;      // [nb][r]   UNIFORM
  const float* inv_step;  // [nb][r]   UNIFORM (fp32 1/step)
  const float* vnorm;     // [nb][r]   ||V_k||_2, rounded up (error-bound scale)
  const uint8_t* bits;    // [nb][r]
  const int16_t* order;   // [nb][r]   kept components in packed order
  const int32_t* seg;     // [nb][kMaxSeg][4]: start byte, width, first order slot, count
  const int32_t* P;       // [nb]      packed row bytes
  const int32_t* n_kept;  // [nb]
  const int32_t* groups;  // [n_groups][3]: first component, count, width (GROUP)
  const float* codebook;  // [cb_levels] ascending (CODEBOOK)
  const float* mids;      // [cb_levels-1] fp32 midpoints (CODEBOOK fast path)
  const int32_t* basis_of;  // [n_slots]

  uint8_t* store;
  const int64_t* pay_off;   // [n_slots]
  const int64_t* side_off;  // [n_slots]

  int* err;                        // device error word
  unsigned long long* counters;    // [4]
};

struct AppendArgs {
  const void* x;
  int64_t sb, sh, st;  // element strides of batch, head, token
  int64_t T;           // tokens in this call
  int64_t t_base;      // length before the call (first store row written)
};

struct FetchArgs {
  void* out;
  int64_t ld_s;  // rows per (b, h) in out
  int64_t S;     // tokens to reconstruct
};

// Kernel launchers (kvc_generic.cu).  Return the launch's cudaError_t and add
// the number of kernels launched to *nk.
cudaError_t launch_append_generic(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk);
cudaError_t launch_fetch_generic(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk);
cudaError_t launch_append_int8(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk);
cudaError_t launch_fetch_int8(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk);

}  // namespace kvc
