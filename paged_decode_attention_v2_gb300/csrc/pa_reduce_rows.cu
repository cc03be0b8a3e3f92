// Phase 2 of V2 for short rows: the same cross-partition log-sum-exp reduce as
// pa_reduce.cu, per the "paged_attention_v2" commit note (project_6, commit
// 96f4baf "Dockerfile", section "Implementation", "Phase 2: Cross-partition
// reduction"):
//   M     = max_p max_logits[p]
//   r_p   = exp(max_logits[p] - M) * exp_sums[p]
//   out   = sum_p (r_p / sum_p' r_p') * tmp_out[p]
// for (sequence, head) rows whose partials fit in a few KB.
//
// A row's partial outputs are contiguous ([partition][D] fp32), so a warp
// takes them in one bulk copy (TMA engine, global -> shared) into one of its
// two buffers, and the next row's copy is in flight while it reduces the
// current one from shared memory.  With several KB a warp and dozens of warps
// an SM, the partials of the whole batch cross the memory system in about one
// round trip, where register loads in rounds of a few partitions a thread
// take several.  Lane i holds partition i's (max, sum) for the row's weights;
// a lane owns 4 output columns of every 128.
#include <math_constants.h>

#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kRowsWarps = kReduceRowsThreads / 32;  // warps a CTA
constexpr int kRowsChunks = 2;  // float4 columns a lane: D at most 256

__device__ __forceinline__ void bulk_load_row(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace

// Dynamic shared memory: kRowsWarps x 2 buffers of p.max_parts x D floats,
// then kRowsWarps x 2 mbarriers.  Rows with more partitions than 32 (one a
// lane) are not served here; the host picks the general kernel for them.
template <typename OutT>
__global__ void __launch_bounds__(kRowsWarps * 32)
    pa_v2_reduce_rows_kernel(const __grid_constant__ ReduceParams p) {
  extern __shared__ __align__(16) uint8_t smem_rows[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int D = p.head_size;
  const int P = p.max_parts;
  const size_t buf_floats = (size_t)P * D;
  float *bufs = reinterpret_cast<float *>(smem_rows) + (size_t)warp * 2 * buf_floats;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem_rows + (size_t)kRowsWarps * 2 * buf_floats * 4);
  const uint32_t bar0 = smem_u32(bars + 2 * warp);
  const long long nrows = (long long)p.num_seqs * p.num_heads;
  const long long rstride = (long long)gridDim.x * kRowsWarps;
  const uint64_t limit = kDrainLimitNs;

  if (lane == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    fence_mbar_init();
  }
  __syncwarp();
  long long row = (long long)blockIdx.x * kRowsWarps + warp;
  // seq_lens is an input, read before the wait (chunk mode: the rows' limits
  // are Phase 1 results, read after it)
  int np = row < nrows && !p.row_limit ? partitions_of_row(p, row) : 0;
  pdl_wait_primary();
  if (p.sched && blockIdx.x == 0 && threadIdx.x == 0) {  // Phase 1's work counters, for the next call
    p.sched[0] = 0;
    p.sched[1] = 0;
  }
  if (p.row_limit && row < nrows) np = partitions_of_row(p, row);
  pdl_launch_dependents();

  // a row's copy into buffer b, and its lane's (max, sum)
  auto issue = [&](long long r, int n, int b, float &ml, float &es) {
    const bool done = p.fuse_limit > 0 && n <= p.fuse_limit;  // finished by Phase 1
    ml = -CUDART_INF_F;
    es = 0.f;
    if (done || n <= 0) return;
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)n * (uint32_t)D * 4u;
      mbar_arrive_expect_tx(bar0 + 8 * b, bytes);
      bulk_load_row(smem_u32(bufs + (size_t)b * buf_floats), p.tmp_out + (size_t)r * P * D, bytes,
                    bar0 + 8 * b);
    }
    if (lane < n) {
      ml = __ldcg(p.max_logits + (size_t)r * P + lane);
      es = __ldcg(p.exp_sums + (size_t)r * P + lane);
    }
  };
  uint32_t phases = 0;  // bit b: the parity of buffer b's next copy
  int b = 0;
  float ml = -CUDART_INF_F, es = 0.f;
  if (row < nrows) issue(row, np, b, ml, es);
  bool ok = true;
  while (row < nrows) {
    const long long next = row + rstride;
    int np_next = 0;
    float ml_next = -CUDART_INF_F, es_next = 0.f;
    if (next < nrows) {
      np_next = partitions_of_row(p, next);
      issue(next, np_next, b ^ 1, ml_next, es_next);
    }
    const bool done = p.fuse_limit > 0 && np <= p.fuse_limit;
    if (!done) {
      OutT *out = static_cast<OutT *>(p.out) + row * D;
      if (np <= 0) {  // an empty sequence: zeros
        for (int c = 4 * lane; c < D; c += 128) store4(out + c, 0.f, 0.f, 0.f, 0.f);  // no shuffles
      } else {
        const bool w =
            lane == 0 ? mbar_wait(bar0 + 8 * b, (phases >> b) & 1u, limit, nullptr) : true;
        ok = __shfl_sync(0xffffffffu, w, 0) && ok;
        phases ^= 1u << b;
        // weights: r_i = exp(m_i - M) s_i over the row's partitions (lane i)
        float M = ml;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float r = ml == -CUDART_INF_F ? 0.f : expf(ml - M) * es;
        float S = r;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);
        const float inv = S > 0.f ? 1.f / S : 0.f;
        // every lane takes part in each weight's broadcast (a lane may own
        // no column: D 64); then its columns 4 lane + 128 k
        const float *src = bufs + (size_t)b * buf_floats;
        float4 acc[kRowsChunks];
#pragma unroll
        for (int k = 0; k < kRowsChunks; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < np; ++i) {
          const float wi = __shfl_sync(0xffffffffu, r, i);
#pragma unroll
          for (int k = 0; k < kRowsChunks; ++k) {
            const int c = 4 * lane + 128 * k;
            if (c < D) {
              const float4 v = *reinterpret_cast<const float4 *>(src + (size_t)i * D + c);
              acc[k].x = fmaf(wi, v.x, acc[k].x);
              acc[k].y = fmaf(wi, v.y, acc[k].y);
              acc[k].z = fmaf(wi, v.z, acc[k].z);
              acc[k].w = fmaf(wi, v.w, acc[k].w);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kRowsChunks; ++k) {
          const int c = 4 * lane + 128 * k;
          if (c < D) store4(out + c, acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
        }
        __syncwarp();  // every lane has read the buffer before its next copy is issued
      }
    }
    row = next;
    np = np_next;
    ml = ml_next;
    es = es_next;
    b ^= 1;
  }
  if (!ok && lane == 0) report(p.status, kStatusTimeout);
}

const void *reduce_rows_kernel(int dtype) {
  switch (dtype) {
    case 0: return reinterpret_cast<const void *>(&pa_v2_reduce_rows_kernel<float>);
    case 1: return reinterpret_cast<const void *>(&pa_v2_reduce_rows_kernel<__nv_bfloat16>);
    case 2: return reinterpret_cast<const void *>(&pa_v2_reduce_rows_kernel<__half>);
  }
  return nullptr;
}

size_t reduce_rows_smem_bytes(int max_parts, int head_size) {
  return (size_t)kRowsWarps * 2 * (size_t)max_parts * head_size * 4 + (size_t)kRowsWarps * 2 * 8;
}

}  // namespace pa
