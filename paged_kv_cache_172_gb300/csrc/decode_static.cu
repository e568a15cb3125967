// decode_static.cu -- pa_decode_static: decode attention without any
// caller-supplied or library-allocated workspace.
//
// Some callers cannot allocate device memory for a call: a host runtime that
// has already handed the whole device heap to its own pool allocator, a
// plugin embedded in another engine that forbids allocations outside that
// engine's allocator, or a latency-critical loop that cannot afford the
// implicit device synchronisation of cudaMalloc/cudaFree.  For them this
// entry point keeps the split-KV partition scratch in a fixed device array
// that lives in the library image itself.
//
// The array below is a file-scope __device__ variable: every GPU on which
// the library is loaded holds these PA_DECODE_STATIC_SCRATCH_BYTES until
// the process exits.  In host code its name is only a host-side stand-in,
// so the device address is fetched once per device with
// cudaGetSymbolAddress (with that device current) and cached; that happens
// inside the first pa_decode_static call on each device.
#include <mutex>

#include "pk_internal.h"

namespace {

constexpr size_t kScratchFloats = PA_DECODE_STATIC_SCRATCH_BYTES / sizeof(float);

static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set up on first
// use per device).  Returns nullptr and records the CUDA error on failure.
void* scratch_address(cudaError_t* err) {
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" pa_status pa_decode_static(const pa_half* q, const pa_half* k_cache,
                                      const pa_half* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, int B, int H, int D,
                                      int block_size, int num_blocks, int max_blocks_per_seq,
                                      int max_context_len, int partition_tokens, float scale,
                                      pa_half* out, int32_t* status, pa_stream_t stream) {
  const size_t need = pa_decode_workspace_size(B, H, D, block_size,
                                               max_context_len > 0 ? max_context_len : 1,
                                               partition_tokens);
  if (need > PA_DECODE_STATIC_SCRATCH_BYTES) {
    // The plan does not fit the array.  pa_decode without a workspace checks
    // every argument first (an unsupported head_dim or block size, a bad
    // partition size, a null pointer ...) and returns that code; for a call
    // whose arguments are all valid it returns PA_ERR_WORKSPACE.  Either way
    // it returns before any launch.
    return pa_decode(q, k_cache, v_cache, block_tables, context_lens, B, H, D, block_size,
                     num_blocks, max_blocks_per_seq, max_context_len, partition_tokens, scale,
                     out, nullptr, 0, status, stream);
  }
  void* ws = nullptr;
  if (need > 0) {
    cudaError_t e = cudaSuccess;
    ws = scratch_address(&e);
    if (ws == nullptr) {
      cudaGetLastError();  // reset the runtime's last-error slot of this thread
      pk::record_cuda_error(e);
      return PA_ERR_CUDA;
    }
  }
  return pa_decode(q, k_cache, v_cache, block_tables, context_lens, B, H, D, block_size,
                   num_blocks, max_blocks_per_seq, max_context_len, partition_tokens, scale, out,
                   ws, need > 0 ? (size_t)PA_DECODE_STATIC_SCRATCH_BYTES : 0, status, stream);
}
