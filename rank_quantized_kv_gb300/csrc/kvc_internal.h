// Internal declarations shared by the host library and the kernels.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

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

  // Residual sketch and outlier stream of a codebook key layer (kvc_prod.cu);
  // prod == 0 elsewhere.  Row: [codes | sign bits | outlier int8]; side words
  // [norm, residual norm (m > 0), outlier scale (n_out > 0)] in fp16.
  int prod = 0, m = 0, n_out = 0, code_bytes = 0, sign_bytes = 0;
  int64_t split_from = 0;
  const float* W1 = nullptr;       // [D][256]: R | S^T | 0
  const float* SRt = nullptr;      // [D][128]: (S R)^T, zero columns beyond m
  const float* W3 = nullptr;       // [D + m][D]: R^T over S
  const float* s_norm = nullptr;   // [m] ||S_j||_2, rounded up
  const float* sr_norm = nullptr;  // [m] ||(S R)_j||_2, rounded up
  const int32_t* channels = nullptr;  // [n_slots][n_out] ascending
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

// Latents projected elsewhere (group mode: the tensor-core projection), read
// by the CUDA-core append in place of its own projection, with the error bound
// that projection guarantees:
//   |z32 - z| <= gamma ||x - mean|| ||V_k|| + ex ||V_k|| + en ||x - mean||.
struct ZIn {
  const float* z = nullptr;  // [n_slots][Tc][r] fp32 latents of the call's tokens
  const int* ovf = nullptr;  // [n_slots][tps]: nonzero where a 128-token tile is not in z
  int64_t Tc = 0;            // rows per slot in z
  int tps = 0;               // 128-token tiles per slot
  float gamma = 0.f, ex = 0.f, en = 0.f;
};

// Decode attention over a key layer and a value layer (kvc_attend.cu).
struct AttendArgs {
  const float* q = nullptr;  // [B][Hq][D] fp32
  void* out = nullptr;       // [B][Hq][D] fp16 or bf16
  int Hq = 0, rep = 0;       // query heads; query heads per key/value head
  float scale_log2 = 0.f;    // score scale times log2(e)
  int out_bf16 = 0;
  int64_t S = 0;             // stored tokens
  int splits = 0;            // token splits per slot
  int64_t span = 0;          // tokens per split (a multiple of 128)
  int NCk = 0;               // packed positions of the key codes (chunk-aligned)
  int Dv = 0;                // accumulator width: D (int8 values) or the value positions
  int Pk_max = 0, Pv_max = 0;  // largest packed key / value row
  float* w = nullptr;        // workspace: [B Hq][NCk] key weights
  float* c1 = nullptr;       // workspace: [B Hq] score offsets
  float* part = nullptr;     // workspace: [n_slots][splits][rep][2 + Dv] partials
  // keys with a residual sketch and/or an outlier stream
  int prod = 0, m = 0, n_out = 0;
  int kcode = 0;             // code bytes of a key row (the sign bytes follow)
  int knw = 1;               // fp16 side words per key
  float* wx = nullptr;       // workspace: [B Hq][m + n_out] sketch and outlier weights
};
// Workspace bytes (and the split) of an attention call; the launcher.
// extra: sketch rows plus outlier channels of the keys (0 without them).
size_t attend_plan(int B, int Hq, int n_slots, int rep, int64_t S, int NCk, int Dv, int sms,
                   int extra, int* splits, int64_t* span);
cudaError_t launch_attend(const Params& kp, const Params& vp, AttendArgs a, void* workspace,
                          cudaStream_t s, int* nk);

// On-device prefill fit of the uniform mode (kvc_fit.cu).  Every pointer is
// device memory; the float64 scratch lives in the caller's workspace.
constexpr int kFitMaxD = 128;
constexpr int kFitMaxChoices = 8;
struct FitArgs {
  const void* x = nullptr;
  int dtype = 0;
  int B = 0, H = 0, D = 0, r = 0;
  int64_t S = 0;                // fit rows per slot
  int64_t sb = 0, sh = 0, st = 0;  // element strides of batch, head, token
  int n_choices = 0;
  int choices[kFitMaxChoices] = {};  // ascending, distinct
  int budget = 0;               // bits per token, at most max(choices) * r
  float* V = nullptr;           // [n_slots][D][r]
  float* mean = nullptr;        // [n_slots][D]
  uint8_t* bits = nullptr;      // [n_slots][r]
  float* qmin = nullptr;        // [n_slots][r]
  float* qstep = nullptr;       // [n_slots][r]
  double* lam_out = nullptr;    // [n_slots][D] sorted eigenvalues (may be null)
  // workspace
  double *mean64 = nullptr, *lam = nullptr, *lam_sorted = nullptr, *cov = nullptr,
         *vec = nullptr, *dp = nullptr;
};
size_t fit_workspace_bytes(int n_slots, int D, int r, int budget);
cudaError_t launch_fit_uniform(FitArgs f, void* workspace, cudaStream_t s, int* nk);

// Residual-sketch / outlier-stream codebook keys (kvc_prod.cu).
constexpr int kProdMaxD = 128;
constexpr int kProdMaxM = 128;
constexpr int kProdMaxOut = 32;
cudaError_t launch_append_prod(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk);
cudaError_t launch_fetch_prod(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk);
cudaError_t launch_fit_outliers(const void* x, int dt, int B, int H, int D, int64_t n, int64_t sb,
                                int64_t sh, int64_t st, int n_out, int32_t* channels,
                                cudaStream_t s);

// Code histogram of the store (kvc_entropy.cu): counts [n_slots][NC][256]
// (NC chunk-aligned positions); Huffman code lengths of n symbol counts.
size_t histogram_bytes(int n_slots, int NC);
cudaError_t launch_code_histogram(const Params& p, uint32_t* counts, int NC, int64_t S,
                                  cudaStream_t s, int* nk);
std::vector<int> huffman_code_lengths(const uint32_t* counts, int n);

// Everything derived from a descriptor, on the host (kvc_api.cu).
struct Geo {
  int d_in = 0, Hg = 0, n_slots = 0, nb = 0, r = 0;
  int cb_levels = 0, n_groups = 0, side_bytes = 0;
  std::vector<uint8_t> bits;     // [nb][r]
  std::vector<int32_t> P, n_kept, seg, groups, basis;
  std::vector<int16_t> order;
  std::vector<int64_t> pay_off, side_off;
  int64_t store_total = 0;
  int64_t fixed = 0;
  // residual sketch / outlier stream (kvc_init_layer_prod)
  int prod = 0, m = 0, n_out = 0, code_bytes = 0, sign_bytes = 0;
  int64_t split_from = 0;
  std::vector<float> S;             // [m][D]
  std::vector<int32_t> channels;    // [n_slots][n_out]
};

// Host image of a layer's parameter block: arrays appended at 256-byte
// alignment, with each array's offset.
struct ParamImage {
  std::vector<uint8_t> bytes;
  size_t oV = 0, oVt = 0, oMean = 0, oLo = 0, oStep = 0, oInv = 0, oVn = 0, oBits = 0,
         oOrder = 0, oSeg = 0, oP = 0, oKept = 0, oGroups = 0, oCb = 0, oMids = 0, oBasis = 0,
         oPay = 0, oSide = 0, oErr = 0, oCnt = 0, oW1 = 0, oSRt = 0, oW3 = 0, oSn = 0, oSRn = 0,
         oCh = 0;
  template <class T>
  size_t put(const T* src, size_t n) {
    const size_t off = (bytes.size() + 255) / 256 * 256;
    bytes.resize(off + sizeof(T) * std::max<size_t>(n, 1), 0);
    if (n) std::memcpy(bytes.data() + off, src, sizeof(T) * n);
    return off;
  }
  size_t zeros(size_t nbytes) {
    const size_t off = (bytes.size() + 255) / 256 * 256;
    bytes.resize(off + std::max<size_t>(nbytes, 1), 0);
    return off;
  }
};

// Validate a descriptor and derive its layout; on failure the message is
// available from kvc_last_error().
kvc_status build_geo(const kvc_layer_desc* d, Geo& g);
kvc_status build_geo_prod(const kvc_layer_desc* d, const kvc_prod_desc* pd, Geo& g);
void build_param_image(const kvc_layer_desc* d, const Geo& g, ParamImage& im);
void bind_params(Params& p, const kvc_layer_desc* d, const Geo& g, const ParamImage& im,
                 uint8_t* base);
kvc_status set_error(kvc_status s, const char* msg);
bool device_ptr_on(const void* ptr, int dev);

// Kernel launchers (kvc_generic.cu).  Return the launch's cudaError_t and add
// the number of kernels launched to *nk.
cudaError_t launch_append_generic(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk,
                                  const ZIn* zin = nullptr);
cudaError_t launch_fetch_generic(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk);
cudaError_t launch_append_int8(const Params& p, const AppendArgs& a, cudaStream_t s, int* nk);
cudaError_t launch_fetch_int8(const Params& p, const FetchArgs& f, cudaStream_t s, int* nk);

}  // namespace kvc
