// Allocation-free variant of the weight fold + quantization entry point.
//
// sq_fold_quantize_weight needs a small device scratch buffer (one 32-bit
// running maximum per output channel) that its caller provides.  Some
// callers have no way to provide one: code that runs inside another
// engine's execution callback and is handed only a stream and its tensors,
// or a host that has reserved its whole device-memory budget up front, may
// not call cudaMalloc (it can fail for lack of memory, or stall every
// stream on the device while it runs).  sq_fold_quantize_weight_noalloc
// serves them: its scratch is a fixed array in this library's own device
// memory, so the call allocates nothing.
#include <mutex>

#include "sq_common.cuh"

namespace sq {
sq_status fold_quantize_weight(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*,
                               void*, sq_codes, float*, int32_t*, void*, cudaStream_t);

namespace {

// One running maximum per output channel; every device that loads the
// library holds this array (256 KiB) until the process exits.
static __device__ __align__(256) uint32_t g_fold_scratch[SQ_NOALLOC_MAX_COUT];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fold_scratch on the current device.  In host code the
// array's name only stands in for the device symbol, so the address must
// come from cudaGetSymbolAddress.  Outside stream capture it is looked up
// on every call (cheap once the module is loaded), so a device reset, which
// reloads the module and may move the array, never leaves a stale address;
// a call made while `stream` is capturing reuses the last address seen on
// this device, since capture forbids the module loading a first lookup may
// need.
sq_status scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SQ_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    return SQ_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fold_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // reset the runtime's last-error state for later calls
      return SQ_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SQ_OK;
}

}  // namespace
}  // namespace sq

extern "C" sq_status sq_fold_quantize_weight_noalloc(const void* w, sq_dtype dt, int64_t cin,
                                                     int64_t cout, int64_t ldw, const float* s,
                                                     void* wq, sq_codes fmt, float* w_scale,
                                                     int32_t* dev_flags, cudaStream_t stream) {
  if (!w || !s || !wq || !w_scale || cin < 1 || cout < 1 || ldw < cout || cin % 16 != 0 ||
      (dt != SQ_F32 && dt != SQ_BF16) || (fmt != SQ_CODES_I8 && fmt != SQ_CODES_BF16))
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) % sq::elem_bytes(dt)) != 0 || !sq::aligned16(wq) ||
      (reinterpret_cast<uintptr_t>(s) & 3) || (reinterpret_cast<uintptr_t>(w_scale) & 3))
    return SQ_ERR_INVALID_ARG;
  if (cout > SQ_NOALLOC_MAX_COUT) return SQ_ERR_WORKSPACE;  // beyond the fixed scratch
  void* scratch = nullptr;
  const sq_status st = sq::scratch_address(stream, &scratch);
  if (st != SQ_OK) return st;
  // the fold zeroes the cout maxima it uses before accumulating into them
  return sq::fold_quantize_weight(w, dt, cin, cout, ldw, s, wq, fmt, w_scale, dev_flags, scratch,
                                  stream);
}
