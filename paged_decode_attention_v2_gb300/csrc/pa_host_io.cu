// The per-step inputs of pa_forward_host read straight from pinned host
// memory.
//
// Pinned host memory is mapped into the device's address space, and on
// GB300 the host link is NVLink-C2C: SM loads over it need no copy-engine
// set-up per transfer, which at the sizes of one decode step (a few MB of
// queries and block tables) costs more than the bytes themselves.  One
// launch of this kernel copies the step's sequence lengths, block tables and
// queries from the caller's pinned buffers into the device staging buffer;
// the forward's last kernel then stores the output straight into the
// caller's pinned output buffer (see pa_forward_host).
#include "pa_device.cuh"

namespace pa {

template <typename V>
__device__ __forceinline__ void copy_units(const V *__restrict__ src, V *__restrict__ dst,
                                           long long n, long long tid, long long nth) {
  // Four loads in flight per thread before the stores: the link's latency is
  // microseconds, so each thread keeps several requests outstanding.
  long long i = tid;
  for (; i + 3 * nth < n; i += 4 * nth) {
    const V a = src[i], b = src[i + nth], c = src[i + 2 * nth], d = src[i + 3 * nth];
    dst[i] = a;
    dst[i + nth] = b;
    dst[i + 2 * nth] = c;
    dst[i + 3 * nth] = d;
  }
  for (; i < n; i += nth) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) pa_stage_in_kernel(const __grid_constant__ StageInParams p) {
  // The staging buffer may still be read by the previous call's kernels in
  // the stream: wait for them before writing it.  The attention kernel that
  // follows waits for this grid in turn, so it may start its prologue now.
  pdl_wait_primary();
  pdl_launch_dependents();
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nth = (long long)gridDim.x * blockDim.x;
#pragma unroll 1
  for (int seg = 0; seg < kStageInSegments; ++seg) {
    if (p.width[seg] == 16)
      copy_units(static_cast<const uint4 *>(p.src[seg]), static_cast<uint4 *>(p.dst[seg]),
                 p.units[seg], tid, nth);
    else
      copy_units(static_cast<const uint32_t *>(p.src[seg]), static_cast<uint32_t *>(p.dst[seg]),
                 p.units[seg], tid, nth);
  }
}

const void *stage_in_kernel() { return reinterpret_cast<const void *>(&pa_stage_in_kernel); }

}  // namespace pa
