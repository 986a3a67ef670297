// Append for callers that cannot allocate device memory.
//
// Some callers are handed their device buffers and must not allocate any of
// their own: a plugin or custom operator run from inside another inference
// engine's execution step receives its inputs and outputs from that engine
// and may not call cudaMalloc there, and a server whose device memory is all
// reserved up front by its own pool has no memory left for one.  Such a
// caller cannot use kvc_init_layer, which allocates the layer's parameter
// block.  kvc_append_noalloc does the same append with no allocation at all:
// the parameter tables the kernel reads (basis, transposed basis, quantiser
// tables, store offsets) and its error word and counters are written into
// one file-scope device array, g_noalloc_scratch, which every GPU that loads
// this library holds until the process exits.
#include <mutex>

#include "kvc_internal.h"

namespace {

// Largest parameter image the entry point accepts.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on device `dev` (the current device).
// Looked up once per device, in the CUDA runtime's primary context of that
// device (the context every runtime call uses); the name itself is only a
// host-side stand-in.  Callers that bind a context of their own with the
// driver API are not supported.
kvc_status scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return kvc::set_error(KVC_ECUDA, "device index out of range");
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      return kvc::set_error(KVC_ECUDA, "cudaGetSymbolAddress(g_noalloc_scratch) failed");
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_append_noalloc(const kvc_layer_desc* desc, int64_t length,
                                         const void* x, int64_t T, int64_t stride_b,
                                         int64_t stride_h, int64_t stride_t, void* stream) {
  kvc::Geo g;
  kvc_status st = kvc::build_geo(desc, g);
  if (st) return st;
  if (length < 0 || T < 0) return kvc::set_error(KVC_EINVAL, "length and T must be >= 0");
  if (T > desc->capacity - length)
    return kvc::set_error(KVC_ECAPACITY, "length + T exceeds the capacity; nothing written");
  if (!desc->store || (uintptr_t)desc->store % 256)
    return kvc::set_error(KVC_EINVAL, "store must be a 256-byte aligned device pointer");
  if (desc->store_bytes < (size_t)g.store_total)
    return kvc::set_error(KVC_EINVAL, "store_bytes is below kvc_store_bytes()");
  if (stride_b < 0 || stride_h < 0 || stride_t < 0)
    return kvc::set_error(KVC_EINVAL, "strides must be >= 0");

  kvc::ParamImage im;
  kvc::build_param_image(desc, g, im);
  if (im.bytes.size() > kNoAllocScratchBytes)
    return kvc::set_error(KVC_EINVAL,
                          "the layer's parameter tables exceed the 8 MiB the no-allocation "
                          "append holds; use kvc_init_layer + kvc_append");
  if (T == 0) return KVC_OK;
  if (!x) return kvc::set_error(KVC_EINVAL, "x is NULL");

  // The tables are uploaded from a host vector that is freed on return, so
  // the call cannot be recorded into a CUDA graph: a replay would upload
  // whatever then occupies that memory.
  auto s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return kvc::set_error(KVC_ECUDA, "cudaStreamIsCapturing failed");
  if (cap != cudaStreamCaptureStatusNone)
    return kvc::set_error(KVC_EINVAL,
                          "kvc_append_noalloc cannot run under stream capture; call it "
                          "outside the captured region");

  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvc::set_error(KVC_ECUDA, "cudaGetDevice failed");
  if (!kvc::device_ptr_on(desc->store, dev) || !kvc::device_ptr_on(x, dev))
    return kvc::set_error(KVC_EINVAL, "store and x must be device memory of the current device");
  void* scratch = nullptr;
  st = scratch_address(dev, &scratch);
  if (st) return st;

  // The image carries a zeroed error word and zeroed counters, so every call
  // starts them from zero; the tables overwrite the previous call's.
  e = cudaMemcpyAsync(scratch, im.bytes.data(), im.bytes.size(), cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return kvc::set_error(KVC_ECUDA, "upload of the parameter tables failed");

  kvc::Params p{};
  kvc::bind_params(p, desc, g, im, static_cast<uint8_t*>(scratch));
  const kvc::AppendArgs a{x, stride_b, stride_h, stride_t, T, length};
  int nk = 0;
  // The error word and counters in the array cannot be read back through this
  // entry point, so only kernels that report nothing through them may run
  // here: the CUDA-core append kernels have no bounded waits and no device
  // error paths.  A kernel that reports a time-out or a range error must not
  // be launched from this call.
  e = desc->mode == KVC_MODE_INT8 ? kvc::launch_append_int8(p, a, s, &nk)
                                  : kvc::launch_append_generic(p, a, s, &nk);
  if (e != cudaSuccess) return kvc::set_error(KVC_ECUDA, "append launch failed");
  return kvc::set_error(KVC_OK, "");
}
