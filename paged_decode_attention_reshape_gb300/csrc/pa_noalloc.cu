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

#include "../../include/pa.h"

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
  if (!q || !k_cache || !block_table || q->ndim != 3 || k_cache->ndim != 4 || block_table->ndim != 2)
    return PA_ERR_INVALID_ARG;
  const int S = static_cast<int>(q->shape[0]), Hq = static_cast<int>(q->shape[1]);
  const int D = static_cast<int>(q->shape[2]), max_blocks = static_cast<int>(block_table->shape[1]);
  if (num_kv_heads <= 0 || Hq <= 0 || Hq % num_kv_heads) return PA_ERR_INVALID_ARG;

  // How much scratch this call needs: none when the plan does not split.
  int P = 0, nparts = 1;
  int rc = pa_decode_plan(S, Hq, num_kv_heads, D, max_blocks, k_cache->dtype, 0, partition_size, &P, &nparts);
  if (rc != PA_OK) return rc;
  const size_t need = (P > 0 || P == PA_PARTITION_BALANCED)
                          ? pa_decode_workspace_size(S, Hq, num_kv_heads, D, max_blocks, P)
                          : 0;
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // bigger than the fixed buffer

  void *scratch = nullptr;
  if (need > 0) {
    if ((rc = scratch_address(&scratch)) != PA_OK) return rc;
    // The split-KV arrival counters sit at the start of the scratch and must be
    // zero when the decode starts.  The previous call may have left partial
    // results there (a different shape puts them at different offsets), so the
    // counter region is cleared on the call's stream first.
    const int G = Hq / num_kv_heads;
    const size_t counter_bytes = static_cast<size_t>(S) * num_kv_heads * ((G + 7) / 8) * sizeof(int);
    if (cudaMemsetAsync(scratch, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return pa_decode_ex(out, q, k_cache, v_cache, block_table, seq_lens, scale, num_kv_heads, k_scale, v_scale,
                      partition_size, scratch, need > 0 ? PA_NOALLOC_SCRATCH_BYTES : 0, device_error, stream);
}
