// Phase 2 of V2: cross-partition log-sum-exp reduce, per the
// "paged_attention_v2" commit note (project_6, commit 96f4baf "Dockerfile",
// section "Implementation", "Phase 2: Cross-partition reduction"):
//   M     = max_p max_logits[p]
//   r_p   = exp(max_logits[p] - M) * exp_sums[p]
//   out   = sum_p (r_p / sum_p' r_p') * tmp_out[p]
//
// A group of `wph` warps (1, 2, 4 or 8) serves one (sequence, query head) and
// a slice of `cols_per_cta` columns of it; a 256-thread CTA holds 8 / wph such
// groups.  Every warp of a group finds M and sum r_p over all partitions by
// itself (warp shuffles, no block barrier), then takes every wph-th
// partition and accumulates r_p * tmp_out[p] over its columns with 16-byte
// loads, four partitions in flight.  With wph > 1 the warps' partial sums
// meet once in shared memory.  One warp per head suits batches whose
// sequences span few partitions; long sequences split their partitions over
// up to 8 warps (and their columns over several CTAs) to keep the load chain
// short.
#include <math_constants.h>

#include "pa_device.cuh"

namespace pa {

constexpr int kReduceThreads = 256;

template <typename OutT>
__global__ void __launch_bounds__(kReduceThreads)
    pa_v2_reduce_kernel(const __grid_constant__ ReduceParams p) {
  // With programmatic dependent launch this kernel may start before Phase 1
  // has finished; wait here until all of its results are visible.
  pdl_wait_primary();

  __shared__ float4 part_sum[kReduceThreads / 32][64];  // [warp][<= 256 cols / 4]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wph = p.warps_per_head;
  const int groups = (kReduceThreads / 32) / wph;
  const int g = warp / wph, wig = warp % wph;  // group in CTA, warp in group
  const long long pair = (long long)blockIdx.x * groups + g;
  const bool live = pair < (long long)p.num_seqs * p.num_heads;
  const int s = live ? (int)(pair / p.num_heads) : 0;
  const int h = live ? (int)(pair % p.num_heads) : 0;
  const int D = p.head_size;
  const int ncols = p.cols_per_cta;
  const int col0 = blockIdx.y * ncols;

  int np = 0;
  if (live) {
    int L = p.seq_lens[s];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);  // Phase 1 reported it
    np = (L + p.partition_size - 1) / p.partition_size;
  }
  OutT *out = static_cast<OutT *>(p.out) + ((size_t)s * p.num_heads + h) * D + col0;
  const size_t row0 = ((size_t)s * p.num_heads + h) * p.max_parts;
  const float *ml = p.max_logits + row0;
  const float *es = p.exp_sums + row0;

  // ---- M and the normaliser, per warp
  float mx = -CUDART_INF_F;
  for (int i = lane; i < np; i += 32) mx = fmaxf(mx, __ldcg(ml + i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float wsum = 0.f;
  for (int i = lane; i < np; i += 32) wsum += expf(__ldcg(ml + i) - mx) * __ldcg(es + i);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);

  // ---- weighted sum over this warp's partitions
  // lanes: `lpr` lanes per row (one float4 each, several if ncols > 128),
  // `rpi` rows per warp iteration
  const int c4 = ncols / 4;                // float4s per row
  const int lpr = c4 < 32 ? c4 : 32;       // lanes per row
  const int rpi = 32 / lpr;                // rows per iteration
  const int per_lane = c4 / lpr;           // float4s per lane (1 or 2)
  const int sub = lane / lpr, cl = lane % lpr;
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  const float *tmp = p.tmp_out + row0 * D + col0 + 4 * cl;
  const int stride = wph * rpi;
  int i = wig * rpi + sub;
  for (; i + 3 * stride < np; i += 4 * stride) {
    float4 v[4][2];
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = i + u * stride;
      w[u] = expf(__ldcg(ml + r) - mx) * __ldcg(es + r);
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < per_lane)
          v[u][k] = __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)r * D + 4 * lpr * k));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < per_lane) {
          acc[k].x = fmaf(w[u], v[u][k].x, acc[k].x);
          acc[k].y = fmaf(w[u], v[u][k].y, acc[k].y);
          acc[k].z = fmaf(w[u], v[u][k].z, acc[k].z);
          acc[k].w = fmaf(w[u], v[u][k].w, acc[k].w);
        }
  }
  for (; i < np; i += stride) {
    const float w = expf(__ldcg(ml + i) - mx) * __ldcg(es + i);
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (k < per_lane) {
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)i * D + 4 * lpr * k));
        acc[k].x = fmaf(w, v.x, acc[k].x);
        acc[k].y = fmaf(w, v.y, acc[k].y);
        acc[k].z = fmaf(w, v.z, acc[k].z);
        acc[k].w = fmaf(w, v.w, acc[k].w);
      }
  }
  // fold the rows handled by different lane groups of the warp
  for (int off = lpr; off < 32; off <<= 1)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      acc[k].x += __shfl_xor_sync(0xffffffffu, acc[k].x, off);
      acc[k].y += __shfl_xor_sync(0xffffffffu, acc[k].y, off);
      acc[k].z += __shfl_xor_sync(0xffffffffu, acc[k].z, off);
      acc[k].w += __shfl_xor_sync(0xffffffffu, acc[k].w, off);
    }
  if (wph > 1) {
    if (sub == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < per_lane) part_sum[warp][cl + lpr * k] = acc[k];
    }
    __syncthreads();
    if (wig != 0) return;
    if (sub == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < per_lane)
          for (int w2 = 1; w2 < wph; ++w2) {
            const float4 t = part_sum[warp + w2][cl + lpr * k];
            acc[k].x += t.x;
            acc[k].y += t.y;
            acc[k].z += t.z;
            acc[k].w += t.w;
          }
    }
  }
  if (!live || sub != 0) return;
  const float inv = np > 0 ? 1.f / wsum : 0.f;  // np == 0: empty sequence -> zeros
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (k < per_lane) {
      OutT *o = out + 4 * (cl + lpr * k);
      o[0] = from_float<OutT>(acc[k].x * inv);
      o[1] = from_float<OutT>(acc[k].y * inv);
      o[2] = from_float<OutT>(acc[k].z * inv);
      o[3] = from_float<OutT>(acc[k].w * inv);
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
