// pa_v2_forward_noalloc: V2 decode attention for callers that cannot
// allocate device memory.
//
// Some callers cannot hand libpa a workspace.  Examples: a plug-in inside a
// host framework that owns every byte of device memory and forbids
// cudaMalloc while a request is being served, or a latency-critical serving
// loop that must never hit cudaMalloc's implicit synchronisation.  This entry
// point needs nothing from them but the inputs and outputs.  V2's scratch
// (status word + Phase 1 partials) lives in a fixed array in device memory
// that belongs to the library.
//
// The array is allocated when this module is loaded on a device.  Every GPU
// that loads the library keeps it, kNoAllocScratchBytes of it, until the
// process exits.  Requests whose V2 workspace would not fit are refused with
// PA_ERR_WORKSPACE_TOO_SMALL.  All calls on a device share the one array, so
// calls whose kernels overlap on the GPU (two streams, two host threads) race
// and give wrong results.  Callers must serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;  // 32 MiB per device

// In host code this name is only a stand-in for the device array, not its
// address.  The device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of this device's scratch array, looked up once per device
// (with that device current).
pa_status_t scratch_for_current_device(void **ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_v2_forward_noalloc(
    void *out, const void *query, const void *key_cache, const void *value_cache,
    const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_heads,
    int num_kv_heads, int head_size, int num_blocks, int block_size, int max_blocks_per_seq,
    int max_seq_len, float scale, int partition_size, int dtype, void *stream) {
  const size_t need =
      pa_workspace_bytes(num_seqs, num_heads, head_size, max_seq_len, partition_size);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return PA_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = nullptr;
  pa_status_t st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  // The array keeps whatever the previous call left in it.  The status block
  // and the combine counters must start at zero; the partials are written
  // before they are read.
  size_t off[5];
  if (pa_workspace_layout(num_seqs, num_heads, head_size, max_seq_len, partition_size, off) !=
      PA_OK)
    return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_seqs > 0 &&
      (cudaMemsetAsync(scratch, 0, pa::kStatusBytes, s) != cudaSuccess ||
       cudaMemsetAsync(static_cast<unsigned char *>(scratch) + off[4], 0,
                       (size_t)num_seqs * num_heads * sizeof(int), s) != cudaSuccess))
    return PA_ERR_CUDA;
  return pa_v2_forward(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, num_blocks, block_size,
                       max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, scratch,
                       kNoAllocScratchBytes, stream);
}
