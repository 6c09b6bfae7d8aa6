// tsel_importance_noalloc: importance scores without any device allocation.
//
// Who needs this: callers that may not allocate device memory at all once
// they are running — an inference-engine plugin whose host framework has
// already handed all of HBM to its own pool (KV cache, activations), or an
// embedded / automotive stack whose rules forbid allocation after start-up —
// and that have no workspace buffer of their own to lend. For them the
// scratch space lives in one file-scope device array of this library,
// reserved when the library's code is loaded on a GPU and held by every GPU
// that loads the library until the process exits.
//
// The first call on each device does the set-up (looks up the array's device
// address with that device current), so make that first call before any
// stream capture.
//
// The scratch array is shared by every call on a device and keeps whatever
// the last call left there; the device status word in it is cleared at the
// start of each call. Two calls that overlap on the GPU (other streams,
// other threads) race on the array and give undefined results: serialise
// them.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace tsel {
void record_error(const char* msg);  // tsel_api.cu
}

namespace {

// 16 MiB: enough for the schedule, the per-head-group partial sums and the
// padded row-LSE buffer of, e.g., 16 heads over 131072 query and key tokens
// in 128 segments (about 14.1 MB; 30 images of 61,385 tokens need about 6 MB).
constexpr size_t kNoallocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device. In host code
// the array's name is only a host-side stand-in, so the real address comes
// from cudaGetSymbolAddress, once per device, with that device current.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" TSEL_API tsel_status tsel_importance_noalloc(
    const void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seg, int total_q,
    int total_k, int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
    int head_dim, float softmax_scale, float* lse, float* scores, uint32_t* device_status,
    void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (num_seg < 0 || total_q < 0 || total_k < 0 || num_heads < 1)
    return tsel_importance(q, q_row_stride, k, k_row_stride, cu_seqlens_q, cu_seqlens_k, num_seg,
                           total_q, total_k, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads,
                           head_dim, softmax_scale, 0u, lse, scores, nullptr, 0, stream_);
  const int64_t need = tsel::imp_ws_layout(num_seg, total_q, total_k, num_heads).total;
  if (need > int64_t(kNoallocScratchBytes)) {
    char msg[160];
    snprintf(msg, sizeof(msg),
             "tsel_importance_noalloc: this problem needs %lld bytes of scratch, the static "
             "scratch array holds %zu",
             (long long)need, kNoallocScratchBytes);
    tsel::record_error(msg);
    return TSEL_ERR_WORKSPACE;
  }
  if (stream != nullptr) {
    // The scratch array used is the current device's; a stream of another
    // device would run the kernels there against this device's address.
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
      tsel::record_error("tsel_importance_noalloc: cannot query the current or the stream's device");
      return TSEL_ERR_CUDA;
    }
    if (sdev != cur) {
      char msg[160];
      snprintf(msg, sizeof(msg),
               "tsel_importance_noalloc: the stream belongs to device %d, the current device is %d",
               sdev, cur);
      tsel::record_error(msg);
      return TSEL_ERR_INVALID_VALUE;
    }
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) {
    tsel::record_error("tsel_importance_noalloc: cudaGetSymbolAddress of the scratch array failed");
    return TSEL_ERR_CUDA;
  }
  e = cudaMemsetAsync(scratch, 0, sizeof(uint32_t), stream);  // status word starts clear
  if (e != cudaSuccess) {
    tsel::record_error("tsel_importance_noalloc: clearing the status word failed");
    return TSEL_ERR_CUDA;
  }
  tsel_status s = tsel_importance(q, q_row_stride, k, k_row_stride, cu_seqlens_q, cu_seqlens_k,
                                  num_seg, total_q, total_k, max_seqlen_q, max_seqlen_k,
                                  num_heads, num_kv_heads, head_dim, softmax_scale, 0u, lse,
                                  scores, scratch, kNoallocScratchBytes, stream_);
  if (s != TSEL_OK) return s;
  if (device_status != nullptr) {
    e = cudaMemcpyAsync(device_status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                        stream);
    if (e != cudaSuccess) {
      tsel::record_error("tsel_importance_noalloc: copying the status word failed");
      return TSEL_ERR_CUDA;
    }
  }
  return TSEL_OK;
}
