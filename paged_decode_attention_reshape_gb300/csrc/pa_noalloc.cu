// pa_noalloc.cu -- pa_decode_noalloc: paged decode that never allocates device memory.
//
// Some callers cannot allocate at the point where they run decode attention:
// a plugin hosted by an inference runtime that is handed only its input and
// output buffers has no allocator to call, and a serving loop that has given all
// free device memory to its KV-cache pool must not allocate on the hot path (the
// allocation can fail there, and cudaMalloc/cudaFree may synchronise the device
// and stall the other streams).  pa_decode needs split-KV scratch it allocates
// itself, and pa_decode_ex needs the caller to provide it; this entry point uses a
// fixed scratch buffer that is part of the loaded library instead.
//
// The scratch is a file-scope __device__ array of PA_NOALLOC_SCRATCH_BYTES.  Every
// GPU that loads the library holds it until the process exits, and all calls on a
// device share it.  Host code cannot use the array's name as a device address
// (the host-side symbol is only a stand-in), so the first call on each device
// looks the address up with cudaGetSymbolAddress while that device is current,
// checks the result and keeps it for later calls.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

PA_API int pa_decode_noalloc(pa_tensor *out, const pa_tensor *q, const pa_tensor *k_cache,
                             const pa_tensor *v_cache, const pa_tensor *block_table, const pa_tensor *seq_lens,
                             float scale, int num_kv_heads, const float *k_scale, const float *v_scale,
                             int partition_size, int *device_error, pa_stream_t stream) {
  // Every argument is checked first, exactly as pa_decode_ex checks it, and the scratch the
  // call's own plan needs is computed; nothing is launched before that.
  size_t need = 0, counter_bytes = 0;
  int rc = pa::decode_ex_requirements(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, k_scale,
                                      v_scale, partition_size, device_error, &need, &counter_bytes);
  if (rc != PA_OK) return rc;
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // bigger than the fixed buffer

  void *scratch = nullptr;
  if ((rc = scratch_address(&scratch)) != PA_OK) return rc;
  if (counter_bytes > 0) {
    // The split-KV arrival counters sit at the start of the scratch and must be zero when
    // the decode starts.  The previous call may have left partial results there (a
    // different shape puts them at different offsets), so the counter region is cleared
    // on the call's stream first.
    if (cudaMemsetAsync(scratch, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  // The whole buffer is always passed, so pa_decode_ex never takes an allocating path.
  return pa_decode_ex(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, k_scale, v_scale,
                      partition_size, scratch, PA_NOALLOC_SCRATCH_BYTES, device_error, stream);
}
