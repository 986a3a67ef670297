// Tensor-core (tcgen05 / TMEM / TMA) kernels of the hot path: host-side plan.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda.h>

#include "kvc_internal.h"

namespace kvc {

// Ring sizes of the warp-specialised fetch (kvc_fetch_pipe.cu).
struct FetchPipeShape {
  int n_acc = 0;     // TMEM accumulators of D columns
  int n_a = 0;       // A operand buffers (in TMEM after the accumulators)
  int a_col0 = 0;    // TMEM column of the first A buffer
  int a_cols = 0;    // TMEM columns of one A buffer
  int n_rs = 0;      // row stages (packed rows, side words, chunk table)
  int n_stg = 0;     // output staging buffers
  int n_b = 0;       // B buffers
  int rs_bytes = 0;  // bytes of one row stage
  int cb_rep = 0;    // codebook: 8-byte slots of the lane-replicated pair table (0: none)
  int uni_w = 0;     // uniform rows of one width (1, 2, 4 or 8) from byte 0: the width
  int uni_chunks = 0;  // ... and their 8-code chunks (the bias chunk follows)
};

// Ring sizes of the warp-specialised append (kvc_append_ws.cu).
struct AppendWsShape {
  int acc_stride = 0;  // TMEM columns per accumulator (pieces x rpad, rounded up to 32)
  int n_acc = 0;       // accumulators
  int cols = 0;        // TMEM columns allocated
  int tab_bytes = 0;   // bytes of one basis' quantiser table
  int x_stage = 0;     // bytes of one x stage (x tile + table)
  int n_x = 0;         // x stages
  int n_b = 0;         // B buffers
  int ks = 0;          // bytes per token row of the chunk-aligned code staging
  int pmax = 0;        // bytes per token row of the packed-row staging (0: none)
  int nq = 0;          // queue entries per quantiser group
  int vt_smem = 0;     // V^T kept in shared memory beside B
};

// Tables the tensor-core kernels need, appended to the layer's parameter
// block by tc_prepare (as offsets) and turned into device pointers by tc_bind.
struct TcPlan {
  // fetch: x_hat = A B^T + bias, A = decoded codes [tokens x K], B [D_in x K]
  bool fetch_ready = false;
  int fetch_K = 0;             // K: segments padded to 8, total rounded up to 16
  int fetch_cols = 0;          // TMEM columns (D, a power of two)
  size_t fetch_smem = 0;       // dynamic shared memory per CTA
  size_t oFetchB = 0, oBias = 0, oChunks = 0, oSlotP = 0;
  const uint16_t* fetchB = nullptr;  // fp16 [nb][D_in][K] in UMMA no-swizzle K-major order
  const float* bias = nullptr;       // fp32 [nb][D_in]
  const uint32_t* chunks = nullptr;  // [nb][K/8]: first byte | width << 16 | valid << 31;
                                     // 1 << 30 marks the chunk of ones (bias columns);
                                     // group mode: the chunk's group << 20
  bool bias_folded = false;          // B carries the bias (uniform mode)
  const int32_t* slotP = nullptr;    // [n_slots] packed row bytes of each slot
  size_t oChunks32 = 0;
  const uint32_t* chunks32 = nullptr;  // [nb][32]: the chunk table padded to 128 bytes
  // warp-specialised persistent fetch (one head per slot), one CTA per SM
  bool pipe_ready = false;
  int pipe_cols = 0;           // TMEM columns: pipe_acc accumulators of D columns
  FetchPipeShape pipe;
  size_t pipe_smem = 0;

  // append: z = x (V_hi + V_rest) * 2^-scale_exp - mean V, the fp32 basis split
  // into exact 16-bit pieces, the hi piece and the rest in two TMEM accumulators
  bool append_ready = false;
  int app_rpad = 0;            // r rounded up to 16 (N of each piece)
  int app_cols = 0;            // TMEM columns
  size_t app_smem = 0;
  int app_bf16 = 0;            // operands bf16 (else fp16)
  int app_pieces = 3;          // 16-bit pieces of the basis (3 bf16 or 2 fp16)
  float app_inv_scale = 1.f;   // 2^-scale_exp
  float app_gamma = 0.f;       // accumulation error bound per unit of ||x|| ||V_k||
  size_t oAppB = 0, oC64 = 0;
  const uint16_t* appB = nullptr;  // [nb][pieces][rpad][D] UMMA no-swizzle K-major order
  const double* c64 = nullptr;     // [nb][r] mean . V_k in double
  // warp-specialised persistent append (one head per slot), one CTA per SM
  bool ws_ready = false;
  AppendWsShape ws;
  size_t ws_smem = 0;
  size_t oWsTab = 0;
  const unsigned char* wsTab = nullptr;  // [nb][tab_bytes] quantiser tables

  // group mode: z = (x - mean) V on the tensor cores (kvc_group_proj.cu) into a
  // scratch the CUDA-core quantiser reads, in chunks of gp_Tc tokens
  bool gp_ready = false;
  int gp_bf16 = 0;             // x is bf16 (else fp16)
  int gp_rpad = 0;             // N of the MMA: r rounded up to a power of two >= 32
  int gp_nb = 0;               // basis slice stages
  size_t gp_smem = 0;
  float gp_xscale = 1.f;       // 2^sx applied to x - mean before the fp16 split
  float gp_zscale = 1.f;       // 2^-(sx + se)
  float gp_gamma = 0.f, gp_ex = 0.f, gp_en = 0.f;  // the latents' error bound (ZIn)
  int64_t gp_Tc = 0;           // tokens per chunk
  size_t oGpB = 0;
  const uint16_t* gpB = nullptr;  // [nb][hpg][D/64][2][rpad][64] fp16 slices, core-matrix order
  float* zbuf = nullptr;          // [n_slots][gp_Tc][r], owned (tc_alloc / tc_release)
  int* zovf = nullptr;            // [n_slots][gp_Tc / 128]
};

kvc_status tc_prepare(const kvc_layer_desc& d, const Geo& g, std::vector<uint8_t>& image,
                      TcPlan& plan);
void tc_bind(TcPlan& plan, uint8_t* block_base);
kvc_status tc_alloc(TcPlan& plan, int n_slots, int r);  // device scratch the plan needs
void tc_release(TcPlan& plan);

bool tc_append_ok(const TcPlan& plan, const Params& p, const AppendArgs& a);
bool tc_fetch_ok(const TcPlan& plan, const Params& p, const FetchArgs& f);
cudaError_t launch_append_tc(const TcPlan& plan, const Params& p, const AppendArgs& a,
                             uint64_t wait_ns, cudaStream_t s, int* nk);
cudaError_t launch_fetch_tc(const TcPlan& plan, const Params& p, const FetchArgs& f,
                            cudaStream_t s, int* nk);
bool tc_group_ok(const TcPlan& plan, const Params& p, const AppendArgs& a);
cudaError_t launch_append_group_tc(const TcPlan& plan, const Params& p, const AppendArgs& a,
                                   cudaStream_t s, int* nk);

// Warp-specialised persistent fetch (kvc_fetch_pipe.cu); `map` is the output
// tensor map.  fetch_pipe_smem sizes its rings for D, K, the side bytes, the
// largest packed row and the number of bases; 0 when they do not fit.
size_t fetch_pipe_smem(int mode, int D, int hpg, int K, int side_bytes, int pmax, int n_bases,
                       int min_rs, int cb_bits, FetchPipeShape* sh);
cudaError_t launch_fetch_pipe(const TcPlan& plan, const Params& p, const FetchArgs& f,
                              const CUtensorMap& map, cudaStream_t s, int* nk);
// Warp-specialised append (kvc_append_ws.cu): table bytes per basis, one
// basis' table, the ring plan (0 when it does not fit), the launcher.
size_t append_ws_tab_bytes(int rpad);
int append_ws_chunks(const Geo& g, int b);  // pack chunks of basis b
int append_ws_table(const Geo& g, const kvc_layer_desc& d, int rpad, const double* c64,
                    double inv_scale, double gamma, int ks, int b,
                    unsigned char* out);  // returns the basis' pack chunks, -1 if over 32
size_t append_ws_plan(int D, int r, int rpad, int npieces, int pmax, int max_chunks, int n_bases,
                      bool direct,
                      AppendWsShape* sh);
cudaError_t launch_append_ws(const TcPlan& plan, const Params& p, const AppendArgs& a,
                             const CUtensorMap& xmap, uint64_t wait_ns, cudaStream_t s, int* nk);
// Group-mode projection (kvc_group_proj.cu): shared memory for N = rpad and
// the basis slice stages it leaves room for (0 when two do not fit); the
// launcher for one chunk of tokens (`map` covers exactly that chunk).
size_t group_proj_smem(int rpad, int* n_b);
cudaError_t launch_group_proj(const TcPlan& plan, const Params& p, const AppendArgs& a,
                              const CUtensorMap& map, cudaStream_t s, int* nk);
int sm_count();

}  // namespace kvc
