// kda_chunk_prefill_fwd_noalloc: the tcgen05 prefill for callers that cannot
// allocate device memory, so cannot hand the library a workspace -- for
// instance a plugin running inside a host framework that owns every byte of
// device memory, or a latency-critical loop where a cudaMalloc (which may
// synchronise the device) is not allowed.
//
// The only scratch the prefill needs is the device status word (plus two
// words of error detail).  Here it lives in a file-scope device array that
// every GPU loading this library holds until the process exits.  Host code
// cannot pass the array's name to a kernel (in host code that name is a
// host-side stand-in, not a device address), so the device address is looked
// up with cudaGetSymbolAddress, once per device, by the first call made on
// that device while it is current.  That first call should therefore come
// before any stream capture.  The looked-up address is kept for the life of
// the process: after a cudaDeviceReset (which unloads the library's device
// module) this entry point must not be called again on that device.
//
// The warp-specialised kernel runs (KDA_KERNEL_PIPE, P = 1): the regular entry
// point's AUTO choice whenever the workspace holds no per-chunk records.
//
// Every call shares the array.  Each call clears the status word on its
// stream before the kernel runs; calls that overlap on the GPU (different
// streams, no ordering between them) race on it.  Errors the kernel finds
// on the device are recorded there and are not reported back through this
// entry point; callers that need them use kda_chunk_prefill_fwd with a
// workspace of their own and kda_last_device_status().
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kNoAllocScratchBytes = 256;   // the stated maximum
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchBytes / 4];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (nullptr on error).
void* scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int kda_chunk_prefill_fwd_noalloc(
    const void* q, const void* k, const void* v, const void* g, const void* beta,
    const float* A_log, const float* dt_bias, float lower_bound, float scale,
    const void* initial_state, const int32_t* cu_seqlens, void* out, void* final_state,
    int state_dtype, kda_stream_t stream, int64_t total_tokens, int32_t num_seqs,
    int32_t heads) {
  // The warp-specialised kernel needs only the status words; the split path (whose
  // per-chunk records need a real workspace) is never taken here.
  static_assert(kda::kWorkspaceBytes <= kNoAllocScratchBytes, "scratch too small");
  if (total_tokens < 0 || num_seqs < 0 || heads <= 0) return KDA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  int rc = kda_device_check(dev);
  if (rc != KDA_OK) return rc;
  void* scratch = scratch_address(dev);
  if (!scratch) return KDA_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 16, s) != cudaSuccess) {
    cudaGetLastError();
    return KDA_ERR_CUDA;
  }
  return kda_chunk_prefill_fwd_ex(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                                  initial_state, cu_seqlens, out, final_state, state_dtype,
                                  scratch, stream, total_tokens, num_seqs, heads,
                                  (size_t)kNoAllocScratchBytes, 1, KDA_KERNEL_PIPE);
}
