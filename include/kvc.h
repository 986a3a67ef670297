/*
 * kvc.h -- C ABI of the projected-and-quantized KV cache hot path (GB300, sm_103a).
 *
 * A layer holds one tensor (keys or values) of one attention layer.  Its
 * parameters are frozen at init: a basis V (rank r) with a mean, a per
 * component bit width b_k in {0,1,2,3,4,8} (0 drops the component) and the
 * quantiser's parameters.  The hot path is two calls:
 *
 *   kvc_append  z = (x - mean) V ; quantise each kept component ; bit-pack
 *               the codes into a growing store (one row of P bytes per token);
 *   kvc_fetch   unpack ; dequantise ; x_hat = z_hat V^T + mean, written as
 *               fp16 (or bf16) [B, H, S, D] for attention.
 *
 * Sources (VeloxQuant-MLX documentation pages): the kvtc_cache page (module
 * docstring "Design" and "NOT PATH-DEPENDENT"; _TensorKVTC._requantize;
 * KVTCKVCache.trim and its byte accounting), the turboquant_cache page
 * (TurboQuantKVCache: bit-packed indices, append_key, append_value,
 * _unpack_indices_block, memory_bytes, reset) and the palu_cache page
 * (PALUKVCache "Design" and "Byte accounting", trim).
 *
 * Memory: every pointer named "device" is CUDA device memory on the layer's
 * device; every pointer named "host" is ordinary host memory read during the
 * call only.  The caller owns the store, the inputs and the outputs.  The
 * library owns one small block of device memory per layer (its frozen
 * parameters in kernel layouts, plus an error word and counters) and, in
 * group mode with 16-bit inputs and D a multiple of 64, a scratch of at most
 * 32 MiB for the tensor-core projection's fp32 latents; both are allocated in
 * kvc_init_layer and freed in kvc_destroy; no other call allocates.
 *
 * Errors: every call returns a kvc_status.  Arguments are checked on the host
 * before any launch; on error nothing is launched and the layer is unchanged.
 * kvc_last_error() returns a message for the last failure on this thread.
 * Work is asynchronous on the given stream (a cudaStream_t passed as void*;
 * NULL is the legacy default stream); device-side conditions surface through
 * kvc_sync_status.  Calls on one layer write its store (and scratch) and must
 * be ordered: issue them on one stream, or order the streams with events.
 * Different layers are independent.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 1

typedef struct kvc_layer kvc_layer; /* opaque, host-owned */

typedef enum {
  KVC_OK = 0,
  KVC_EINVAL = -1,    /* bad argument or descriptor field */
  KVC_ESTATE = -2,    /* call not valid for this layer (NULL or destroyed layer) */
  KVC_ECAPACITY = -3, /* the append would exceed the capacity; nothing was written */
  KVC_ECUDA = -4,     /* a CUDA runtime call failed (no device, bad stream, launch error) */
  KVC_ETIMEOUT = -5,  /* a bounded device-side wait gave up (read by kvc_sync_status) */
  KVC_EDEVICE = -6    /* reserved for data a kernel cannot encode exactly (read by
                         kvc_sync_status); no current kernel reports it */
} kvc_status;

enum {
  KVC_MODE_UNIFORM = 0,  /* KVTC-style: code = clip(rint((z - lo)/step), 0, 2^b - 1) */
  KVC_MODE_GROUP = 1,    /* PALU-style: symmetric per-token scale per group of components */
  KVC_MODE_CODEBOOK = 2, /* TurboQuant-MSE-style: rotation + scalar codebook + fp16 norm */
  KVC_MODE_INT8 = 3      /* per-token int8 with an fp16 scale (values) */
};

enum { KVC_F32 = 0, KVC_F16 = 1, KVC_BF16 = 2 };

/* Kernel path selection (kvc_set_path). */
enum {
  KVC_PATH_AUTO = 0,    /* tensor-core kernels where the shape allows, else CUDA cores */
  KVC_PATH_GENERIC = 1  /* CUDA-core kernels only (any shape) */
};

/*
 * Layer descriptor.  Slots: the layer has B * (H / heads_per_group) slots;
 * slot (b, g) holds head group g of batch entry b and uses basis
 * basis_of[b * (H / heads_per_group) + g].  Its token row is the
 * concatenation of the group's heads: D_in = heads_per_group * D values.
 *
 *  mode             KVC_MODE_*.
 *  B, H, D          batch, KV heads, head dimension (> 0).
 *  heads_per_group  heads sharing one projection (palu_cache page: contiguous
 *                   head groups); must be 1 unless mode == GROUP.  Divides H.
 *  r                rank (columns of V).  CODEBOOK: r == D.  INT8: ignored.
 *  n_bases          number of distinct bases (>= 1; ignored for INT8).
 *  basis_of         host int32 [n_slots]; NULL means every slot uses basis 0.
 *  V                host fp32 [n_bases][D_in][r], row-major (column k = basis
 *                   vector k).  CODEBOOK: the D x D rotation.
 *  mean             host fp32 [n_bases][D_in] or NULL (zero).  CODEBOOK: must be NULL.
 *  bits             host uint8 [n_bases][r], each in {0,1,2,3,4,8}.  GROUP: widths
 *                   in {0,2,3,4,8}, non-increasing in k and equal for every basis.
 *                   CODEBOOK: ignored (every component has cb_bits).
 *  qmin, qstep      host fp32 [n_bases][r] (UNIFORM only): frozen minimum and step
 *                   (step > 0 for kept components).
 *  group_size       GROUP only: components per scale group, 1..32 (palu_group_size).
 *  codebook         host fp32 [1 << cb_bits], strictly ascending (CODEBOOK only).
 *  cb_bits          CODEBOOK only: 1, 2, 3, 4 or 8.
 *  in_dtype         dtype of appended rows: KVC_F32, KVC_F16 or KVC_BF16.
 *  out_dtype        dtype of fetched rows: KVC_F16 or KVC_BF16.
 *  capacity         tokens each slot can hold (>= 1).
 *  store            device, caller-owned, at least kvc_store_bytes() bytes,
 *                   256-byte aligned; borrowed for the layer's lifetime.
 *  store_bytes      size of store in bytes.
 */
typedef struct {
  int32_t mode;
  int32_t B, H, D;
  int32_t heads_per_group;
  int32_t r;
  int32_t n_bases;
  const int32_t *basis_of;
  const float *V;
  const float *mean;
  const uint8_t *bits;
  const float *qmin;
  const float *qstep;
  int32_t group_size;
  const float *codebook;
  int32_t cb_bits;
  int32_t in_dtype;
  int32_t out_dtype;
  int64_t capacity;
  void *store;
  size_t store_bytes;
} kvc_layer_desc;

/* Byte accounting (kvtc_cache page "Byte accounting"; turboquant_cache page
 * memory_bytes; palu_cache page "Byte accounting").
 *  payload     packed code bytes: sum over slots of length * P(slot),
 *              P = sum over widths b of ceil(r_b * b / 8) (INT8: D).
 *  side        per-token fp16 side words: GROUP 2 * n_groups, CODEBOOK 2 (norm),
 *              INT8 2 (scale), UNIFORM 0 -- times length, summed over slots.
 *  fixed       frozen parameters counted beside the codes, as the pages count
 *              them: UNIFORM n_bases * (4 D_in r + 4 D_in + r) + 8 * (kept
 *              components over all bases) -- basis and mean in fp32, a width
 *              byte per component, an fp32 minimum and step per kept
 *              component (kvtc_cache page, "Byte accounting" and
 *              _TensorKVTC._requantize); GROUP n_bases * (4 D_in r + 4 D_in),
 *              V_g and mu_g in fp32 (palu_cache page, projection_bytes);
 *              CODEBOOK and INT8 0 (turboquant_cache page, memory_bytes counts
 *              per-token bytes only: the rotation follows from the seed).
 *  fp16_equiv  B * H * length * D * 2, the uncompressed fp16 size. */
typedef struct {
  int64_t payload;
  int64_t side;
  int64_t fixed;
  int64_t fp16_equiv;
} kvc_bytes;

/* Where slot s lives inside the store: token t's packed row is the row_bytes
 * bytes at store + payload_offset + t * row_bytes; its side words are the
 * side_bytes bytes at store + side_offset + t * side_bytes (GROUP: fp16
 * scales in group order; CODEBOOK: fp16 norm; INT8: fp16 scale). */
typedef struct {
  int64_t payload_offset;
  int64_t row_bytes;
  int64_t side_offset;
  int64_t side_bytes;
} kvc_slot_layout;

/* ABI version of the loaded library (KVC_ABI_VERSION). */
int32_t kvc_abi_version(void);

/* Message for the last failing call on this thread ("" if none). */
const char *kvc_last_error(void);

/* Bytes of device store the descriptor needs (host-only; desc->store unused).
 * KVC_EINVAL on a bad descriptor. */
kvc_status kvc_store_bytes(const kvc_layer_desc *desc, size_t *out);

/* Validate the descriptor, copy the frozen parameters to the device in the
 * kernels' layouts and return a layer of length 0 (kvtc_cache page "Design":
 * basis and allocation fit once at prefill, then reused unchanged).  Runs on
 * the current CUDA device and synchronises with it.  Host arrays are only read
 * during the call.  KVC_EINVAL on a bad descriptor, KVC_ECUDA on a CUDA error. */
kvc_status kvc_init_layer(const kvc_layer_desc *desc, kvc_layer **out);

/* Append T tokens: x is device memory, [B, H, T, D] contiguous in in_dtype.
 * Equivalent to kvc_append_strided with strides (H*T*D, T*D, D). */
kvc_status kvc_append(kvc_layer *layer, const void *x, int64_t T, void *stream);

/* Append T tokens from x (device) with element strides: token t of head h of
 * batch b starts at x + b*stride_b + h*stride_h + t*stride_t (elements of
 * in_dtype); the D values of a token are contiguous.  Each token is
 * projected, quantised and packed independently (kvtc_cache page, "Design",
 * decode step 1; turboquant_cache page, append_key / append_value), so T
 * tokens in one call store exactly what T calls of one token store.
 * KVC_ECAPACITY if length + T > capacity (nothing written); T == 0 is a no-op. */
kvc_status kvc_append_strided(kvc_layer *layer, const void *x, int64_t T, int64_t stride_b,
                              int64_t stride_h, int64_t stride_t, void *stream);

/* Reconstruct every stored token: out is device memory [B, H, ld_s, D] in
 * out_dtype; rows 0..length-1 of each (b, h) are written, rows length..ld_s-1
 * are left untouched.  *S_out (may be NULL) receives length.  (kvtc_cache page,
 * "Design": every call returns reconstructed [B, H, S_total, D] for SDPA;
 * palu_cache page: latent -> dequant -> reconstruct.)  KVC_EINVAL if
 * ld_s < length or out is not device memory. */
kvc_status kvc_fetch(kvc_layer *layer, void *out, int64_t ld_s, int64_t *S_out, void *stream);

/* Drop the n most recent tokens (kvtc_cache page KVTCKVCache.trim; palu_cache
 * page trim): n is clamped to the length, n <= 0 drops nothing; *dropped (may
 * be NULL) receives the count.  Host-only, O(1).  The frozen parameters stay,
 * also at length 0 (as turboquant_cache page reset keeps its quantiser). */
kvc_status kvc_trim(kvc_layer *layer, int64_t n, int64_t *dropped);

/* Current length (tokens per slot). */
kvc_status kvc_length(const kvc_layer *layer, int64_t *out);

/* Byte accounting, see kvc_bytes.  Host-only. */
kvc_status kvc_nbytes(const kvc_layer *layer, kvc_bytes *out);

/* Store layout of one slot (0 <= slot < n_slots).  Host-only. */
kvc_status kvc_get_slot_layout(const kvc_layer *layer, int32_t slot, kvc_slot_layout *out);

/* Choose the kernels used by later calls (KVC_PATH_*).  Host-only. */
kvc_status kvc_set_path(kvc_layer *layer, int32_t path);

/* Decode attention on the stored codes (turboquant_cache page,
 * TurboQuantKVCache.attend: the query's score against every stored key,
 * softmax of the scaled scores, weighted sum of the decoded values;
 * palu_cache page, module docstring: the latents are reconstructed only at
 * attend time).  For every batch entry b and query head hq, over all
 * `length` stored tokens t of key/value head h = hq / (Hq / H):
 *   out[b, hq] = sum_t softmax_t(scale * q[b, hq] . k_hat[b, h, t]) v_hat[b, h, t],
 * with k_hat and v_hat the rows kvc_fetch would reconstruct, but computed
 * from the codes without reconstructing them: uniform keys through the
 * per-query weights (V^T q)_k step_k, codebook keys through (R^T q)_k times
 * the centroids and the norm; int8 values as q8 * scale, uniform values as
 * the weighted mean latent projected once.
 *
 *  keys       a KVC_MODE_UNIFORM or KVC_MODE_CODEBOOK layer, heads_per_group 1.
 *  values     a KVC_MODE_INT8 or KVC_MODE_UNIFORM layer with the keys' B, H, D,
 *             device and length; D is 64, 128 or 256.
 *  q          device fp32 [B, Hq, D]; Hq / H is 1, 2, 4 or 8.
 *  scale      the score scale; 0 means 1 / sqrt(D), the pages' scale.
 *  out        device [B, Hq, D] in the value layer's out_dtype.
 *  workspace  device, 256-byte aligned, at least kvc_attend_workspace_bytes()
 *             bytes; caller-owned scratch, overwritten by the call.
 * With length 0 the output is zero.  Asynchronous on `stream`.  Returns
 * KVC_EINVAL for unsupported modes or shapes, mismatched layers, host
 * pointers or a short workspace; nothing is launched then. */
kvc_status kvc_attend(const kvc_layer *keys, const kvc_layer *values, const float *q, int32_t Hq,
                      float scale, void *out, void *workspace, size_t workspace_bytes,
                      void *stream);

/* Workspace bytes kvc_attend needs for these layers at their current length
 * and Hq query heads (host-only). */
kvc_status kvc_attend_workspace_bytes(const kvc_layer *keys, const kvc_layer *values, int32_t Hq,
                                      size_t *out);

/* Order-0 Huffman accounting of the stored codes (kvtc_cache page, module
 * docstring "Byte accounting" and KVTCKVCache.entropy_coding_gain).  Not on
 * the hot path: the store stays fixed width; these calls report what an
 * entropy-coded store would take.  Each kept component of a slot gets its
 * own Huffman code over the values it takes across the slot's tokens; its
 * table costs one byte per symbol of its 2^b alphabet; a slot stores
 * min(ceil(payload bits / 8) + tables, fixed-width bytes).
 *  pre_entropy     fixed-width payload bytes (sum over slots of length * P)
 *  stored_payload  payload after entropy coding and the fixed-width fallback
 *  params          the layer's frozen parameter bytes (kvc_bytes.fixed)
 *  gain            pre_entropy / (stored_payload + params); below 1 when the
 *                  parameters dominate, as the page notes. */
typedef struct {
  int64_t pre_entropy;
  int64_t stored_payload;
  int64_t params;
  double gain;
} kvc_entropy;

/* Bytes of the code histogram of a coded layer: n_slots * NC * 256 uint32
 * counts, NC the basis' largest number of chunk-aligned packed positions
 * (every width segment starts on a multiple of 8).  Host-only.  KVC_EINVAL
 * for an int8 layer. */
kvc_status kvc_code_histogram_bytes(const kvc_layer *layer, size_t *out);

/* Count the stored codes: counts (device, caller-owned, 4-byte aligned, at
 * least kvc_code_histogram_bytes) receives, for slot s and packed position j
 * (segments in descending width, components ascending, each segment starting
 * on a multiple of 8), how many of the slot's tokens hold code v at
 * [(s * NC + j) * 256 + v].  Asynchronous on `stream` (the counts are zeroed
 * first on the same stream). */
kvc_status kvc_code_histogram(kvc_layer *layer, uint32_t *counts, size_t counts_bytes,
                              void *stream);

/* The Huffman byte accounting from a histogram copied to host memory
 * (counts: host, as kvc_code_histogram wrote it for the current length). */
kvc_status kvc_entropy_bytes(const kvc_layer *layer, const uint32_t *counts, kvc_entropy *out);

/* Residual sketch and outlier two-stream store of a KVC_MODE_CODEBOOK key
 * layer (turboquant_cache page: the class docstring -- indices at b_mse bits
 * and QJL sign bits at one bit each; __init__ -- ceil(m / 8) sign bytes, an
 * fp16 residual norm, the outlier detector's n_outliers channels after
 * n_calib keys with an int8 row and fp16 scale per key; append_key;
 * _unpack_signs_block; attend; memory_bytes).  For key t of slot (b, h):
 *   if n_outliers > 0 and t >= split_from: o = x[channels] is stored as int8
 *     codes rint(o / s) with s = max(max|o| / 127, 1e-8) and fp16(s), and
 *     those channels of x are set to 0 (earlier keys: codes 0, scale 0);
 *   the codebook mode's indices and fp16 norm n16 of (the rest of) x, with
 *     desc->cb_bits = b_mse (b - 1 bits for a b-bit prod quantiser);
 *   if m > 0: r = x - n16 R c[idx]; sign bit j = [(S r)_j > 0]; fp16 ||r||.
 * kvc_fetch returns n16 R c[idx] + sqrt(pi/2)/m ||r||16 S^T (2 bits - 1) plus
 * the outlier channels' int8 decode; kvc_attend scores with the same sum.
 * A stored row is [indices | ceil(m/8) sign bytes | n_outliers int8 codes];
 * its side words are fp16 [n16, ||r|| (m > 0), s (n_outliers > 0)].
 *
 *  m            sketch rows (the pages' jl_dim): 0, or a multiple of 16 up to 128.
 *  S            host fp32 [m][D]: the sketch (seeded N(0, 1) entries, the
 *               caller's draw).  NULL when m == 0.
 *  n_outliers   outlier channels per slot: 0 .. min(32, D - 1).
 *  channels     host int32 [B*H][n_outliers], ascending and distinct in [0, D).
 *  split_from   first key index that is split (n_calib - 1: the key that
 *               completes the calibration is split), >= 0.
 * The key layer must have heads_per_group 1, n_bases 1 and D in {32, 64, 128}. */
typedef struct {
  int32_t m;
  const float *S;
  int32_t n_outliers;
  const int32_t *channels;
  int64_t split_from;
} kvc_prod_desc;

/* kvc_store_bytes / kvc_init_layer for a codebook key layer with a residual
 * sketch and/or an outlier stream (prod may not be NULL). */
kvc_status kvc_store_bytes_prod(const kvc_layer_desc *desc, const kvc_prod_desc *prod,
                                size_t *out);
kvc_status kvc_init_layer_prod(const kvc_layer_desc *desc, const kvc_prod_desc *prod,
                               kvc_layer **out);

/* The outlier channels of every slot from its first n_calib keys (device
 * work): the n_outliers channels of largest mean |x| (the lower channel first
 * among equals), ascending, into channels (device int32 [B*H][n_outliers]).
 * x, in_dtype and strides as for kvc_append_strided; n_calib >= 1;
 * 1 <= n_outliers <= min(32, D - 1); D <= 256.  Asynchronous on `stream`. */
kvc_status kvc_fit_outliers(const void *x, int32_t in_dtype, int32_t B, int32_t H, int32_t D,
                            int64_t n_calib, int64_t stride_b, int64_t stride_h,
                            int64_t stride_t, int32_t n_outliers, int32_t *channels,
                            void *stream);

/* On-device prefill fit of the KVC_MODE_UNIFORM parameters (kvtc_cache page:
 * module docstring "Design", prefill step 1, a local PCA per (b, h) fitted
 * in one batched call by KVTCKVCache.update_and_fetch; the module
 * docstring's DP-optimal discrete allocation under a bit budget, 0 bits
 * dropping a component; _TensorKVTC._requantize, a minimum and a step per
 * kept component, frozen here at fit time).  For every slot (b, h), over its
 * first S_fit rows X (float64 throughout, rounded to fp32 at the end):
 *   mean = the column means of X;  C = (X - mean)^T (X - mean) / S_fit;
 *   C = U diag(lam) U^T (cyclic Jacobi), eigenpairs ordered largest first,
 *   ties by index, each vector's sign such that its first largest-magnitude
 *   entry is positive;  V = the first r columns of U in fp32;
 *   bits = argmin sum_k lam_k 2^(-2 b_k) over b_k in bit_choices with
 *   sum_k b_k <= bit_budget (dynamic programme; the smaller width wins a tie);
 *   qmin_k = min_t z_tk, qstep_k = max((max_t z_tk - qmin_k) / (2^b_k - 1), 1e-8)
 *   over z = (x - fp32 mean) V in float64, rounded to fp32 (0 for dropped
 *   components).
 * The outputs are what kvc_layer_desc takes for a UNIFORM layer with one
 * basis per slot (n_bases = B * H, basis_of = identity), in device memory.
 *
 *  x            device [.., D] rows in in_dtype; row t of head h of batch b
 *               starts at x + b*stride_b + h*stride_h + t*stride_t (elements).
 *  S_fit        fit rows per slot (>= 2; the pages fit on the prefill).
 *  D            8 .. 128, a multiple of 8.  r: 1 .. D.
 *  bit_choices  host int32 [n_choices], 1 .. 8 distinct widths from
 *               {0,1,2,3,4,8}; some allocation must fit the budget
 *               (min(bit_choices) * r <= bit_budget).
 *  outputs      device, written for every slot: V fp32 [B*H][D][r], mean fp32
 *               [B*H][D], bits uint8 [B*H][r], qmin and qstep fp32 [B*H][r];
 *               lam float64 [B*H][D] (the sorted eigenvalues) may be NULL. */
typedef struct {
  const void *x;
  int32_t in_dtype;
  int32_t B, H, D;
  int64_t S_fit;
  int64_t stride_b, stride_h, stride_t;
  int32_t r;
  const int32_t *bit_choices;
  int32_t n_choices;
  int32_t bit_budget;
  float *V;
  float *mean;
  uint8_t *bits;
  float *qmin;
  float *qstep;
  double *lam;
} kvc_fit_desc;

/* Workspace bytes kvc_fit_uniform needs for this descriptor (host-only;
 * float64 covariance, eigenvectors and DP tables of every slot). */
kvc_status kvc_fit_uniform_workspace_bytes(const kvc_fit_desc *desc, size_t *out);

/* Run the fit on the current device, asynchronously on `stream` (four kernel
 * launches).  workspace: device, 256-byte aligned, at least
 * kvc_fit_uniform_workspace_bytes() bytes, overwritten.  KVC_EINVAL for a bad
 * field, host pointers or a short workspace; nothing is launched then. */
kvc_status kvc_fit_uniform(const kvc_fit_desc *desc, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Limit, in nanoseconds, of the waits inside the warp-specialised tensor-core
 * append kernel (one role waiting for another: a tile loaded, an accumulator
 * written or released).  A kernel whose wait runs out stops its work, waits
 * for its copies and tensor-core work already in flight (up to 2 s), frees its
 * tensor memory and returns; kvc_sync_status then reports KVC_ETIMEOUT and the
 * rows of that call are undefined.  ns == 0 restores the default of 2 s; a
 * limit shorter than a kernel's normal waits makes every call time out.
 * Host-only.  KVC_EINVAL if ns < 0. */
kvc_status kvc_set_wait_limit(kvc_layer *layer, int64_t ns);

/* Synchronise `stream`, then read and clear the layer's device error word:
 * KVC_OK, KVC_ETIMEOUT (a bounded wait gave up) or KVC_EDEVICE (data the kernel
 * cannot encode exactly).  KVC_ECUDA if the synchronisation itself failed. */
kvc_status kvc_sync_status(kvc_layer *layer, void *stream);

/* Synchronise `stream` and copy the layer's counters to host out[6]:
 * [0] components whose code was re-decided exactly (near a rounding boundary),
 * [1] per-token fp16 side words re-decided, [2] appended tokens, [3] kernels
 * this layer has launched (counted on the host), [4] the largest
 * |fast-path value - exact value| / (error bound) seen among re-decided codes
 * of the tensor-core append, times 1e6 (below 1e6 means the bound held with
 * margin), [5] reserved (0).  With reset != 0 the counters are then zeroed. */
kvc_status kvc_counters(kvc_layer *layer, int64_t out[6], int32_t reset, void *stream);

/* Free the layer's device memory (synchronises the device first).  NULL is a no-op. */
void kvc_destroy(kvc_layer *layer);

/* Append without allocating any device memory.  The pages have no
 * counterpart of this call: it exists for callers that are handed their
 * device buffers and may not allocate, such as a plugin or custom operator
 * run inside another inference engine's execution step, or a server whose
 * device memory is all reserved by its own pool.
 *
 * Stores exactly what kvc_init_layer(desc) followed by kvc_append_strided(x,
 * T, ...) on a layer of length `length` stores: rows length .. length+T-1 of
 * every slot in desc->store (and their side words), computed by the CUDA-core
 * kernels.  The caller keeps track of the length.  x, strides and dtypes as
 * for kvc_append_strided; desc and its host arrays as for kvc_init_layer.
 *
 * Memory: the kernel's parameter tables, error word and counters live in one
 * static device array of 8 MiB that every GPU loading this library holds
 * until exit.  Each call uploads its tables there (cudaMemcpyAsync on
 * `stream`, from host memory, which synchronises the stream first) and
 * zeroes the error word and counters.  All calls share that array, so calls
 * whose work overlaps on the GPU (other streams, other threads) race and
 * corrupt each other's tables: order them on one stream.  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current.  The call cannot be captured into a CUDA graph (the
 * upload reads a host buffer that is freed on return): while `stream` is
 * capturing it returns KVC_EINVAL and enqueues nothing.  The
 * address is that of the CUDA runtime's primary context of the device: call
 * this entry point from the runtime's context, not from a context created
 * with the driver API.
 *
 * Errors: KVC_EINVAL for a bad descriptor or pointers, under stream capture,
 * or when the tables exceed 8 MiB (e.g. many bases of a large D_in x r); KVC_ECAPACITY if
 * length + T > capacity; KVC_ECUDA on a CUDA error.  Nothing is written on
 * error.  Calls no cudaMalloc or cudaFree. */
kvc_status kvc_append_noalloc(const kvc_layer_desc *desc, int64_t length, const void *x,
                              int64_t T, int64_t stride_b, int64_t stride_h, int64_t stride_t,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
