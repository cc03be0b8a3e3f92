// Phase 2 of V2: cross-partition log-sum-exp reduce, per the
// "paged_attention_v2" commit note (project_6, commit 96f4baf "Dockerfile",
// section "Implementation", "Phase 2: Cross-partition reduction"):
//   M     = max_p max_logits[p]
//   r_p   = exp(max_logits[p] - M) * exp_sums[p]
//   out   = sum_p (r_p / sum_p' r_p') * tmp_out[p]
// One CTA per (sequence, query head) x column slice of the head.  The weights
// r_p go to shared memory once; the weighted sum of the tmp_out rows is
// spread over all threads with 16-byte loads, several partitions in flight
// per thread, then folded across thread rows in shared memory.
#include <math_constants.h>

#include "pa_device.cuh"

namespace pa {

constexpr int kReduceThreads = 256;

__device__ __forceinline__ float block_max(float v, float *scratch) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  v = lane < (int)(blockDim.x >> 5) ? scratch[lane] : -CUDART_INF_F;
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  return v;
}

__device__ __forceinline__ float block_sum(float v, float *scratch) {
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  v = lane < (int)(blockDim.x >> 5) ? scratch[lane] : 0.f;
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  return v;
}

template <typename OutT>
__global__ void __launch_bounds__(kReduceThreads)
    pa_v2_reduce_kernel(const __grid_constant__ ReduceParams p) {
  // With programmatic dependent launch this kernel may start before Phase 1
  // has finished; wait here until all of its results are visible.
  pdl_wait_primary();

  const int h = blockIdx.x % p.num_heads, s = blockIdx.x / p.num_heads;
  const int D = p.head_size;
  const int col0 = blockIdx.y * p.cols_per_cta;
  const int ncols = p.cols_per_cta;
  int L = p.seq_lens[s];
  L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);  // Phase 1 reported it
  const int np = (L + p.partition_size - 1) / p.partition_size;
  OutT *out = static_cast<OutT *>(p.out) + ((size_t)s * p.num_heads + h) * D + col0;
  if (np == 0) {
    for (int c = threadIdx.x; c < ncols; c += blockDim.x) out[c] = from_float<OutT>(0.f);
    return;
  }

  extern __shared__ float4 red_smem[];                       // [256] row partial sums
  float *w_s = reinterpret_cast<float *>(red_smem + kReduceThreads);  // [max_parts]
  __shared__ float scratch[32];

  const size_t row0 = ((size_t)s * p.num_heads + h) * p.max_parts;
  const float *ml = p.max_logits + row0;
  const float *es = p.exp_sums + row0;

  float mx = -CUDART_INF_F;
  for (int i = threadIdx.x; i < np; i += blockDim.x) mx = fmaxf(mx, ml[i]);
  mx = block_max(mx, scratch);
  float wsum = 0.f;
  for (int i = threadIdx.x; i < np; i += blockDim.x) {
    const float w = expf(ml[i] - mx) * es[i];
    w_s[i] = w;
    wsum += w;
  }
  wsum = block_sum(wsum, scratch);  // (ends with __syncthreads: w_s is visible)

  const int tpr = ncols / 4;                  // threads per tmp_out row (float4 each)
  const int rows_par = kReduceThreads / tpr;  // rows in flight
  const int c4 = threadIdx.x % tpr, r0 = threadIdx.x / tpr;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float *tmp = p.tmp_out + row0 * D + col0 + 4 * c4;
  int i = r0;
  for (; i + 3 * rows_par < np; i += 4 * rows_par) {
    float4 v[4];
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)(i + u * rows_par) * D));
      w[u] = w_s[i + u * rows_par];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x = fmaf(w[u], v[u].x, acc.x);
      acc.y = fmaf(w[u], v[u].y, acc.y);
      acc.z = fmaf(w[u], v[u].z, acc.z);
      acc.w = fmaf(w[u], v[u].w, acc.w);
    }
  }
  for (; i < np; i += rows_par) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)i * D));
    const float w = w_s[i];
    acc.x = fmaf(w, v.x, acc.x);
    acc.y = fmaf(w, v.y, acc.y);
    acc.z = fmaf(w, v.z, acc.z);
    acc.w = fmaf(w, v.w, acc.w);
  }
  red_smem[threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.x < tpr) {
    float4 t = red_smem[threadIdx.x];
    for (int r = 1; r < rows_par; ++r) {
      const float4 u = red_smem[r * tpr + threadIdx.x];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const float inv = 1.f / wsum;
    OutT *o = out + 4 * threadIdx.x;
    o[0] = from_float<OutT>(t.x * inv);
    o[1] = from_float<OutT>(t.y * inv);
    o[2] = from_float<OutT>(t.z * inv);
    o[3] = from_float<OutT>(t.w * inv);
  }
}

const void *reduce_kernel(int dtype) {
  switch (dtype) {
    case 0: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<float>);
    case 1: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__nv_bfloat16>);
    case 2: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__half>);
  }
  return nullptr;
}

}  // namespace pa
