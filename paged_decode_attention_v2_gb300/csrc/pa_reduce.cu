// Phase 2 of V2: cross-partition log-sum-exp reduce, per the
// "paged_attention_v2" commit note (project_6, commit 96f4baf "Dockerfile",
// section "Implementation", "Phase 2: Cross-partition reduction"):
//   M     = max_p max_logits[p]
//   r_p   = exp(max_logits[p] - M) * exp_sums[p]
//   out   = sum_p (r_p / sum_p' r_p') * tmp_out[p]
//
// A group of `wph` warps (1, 2, 4 or 8) serves one (sequence, query head) and
// a slice of `cols_per_cta` columns of it; a 256-thread CTA holds 8 / wph such
// groups.  Lanes form row groups of `lpr` lanes (one 16-byte column chunk
// each); every row group walks its share of the partitions in one pass,
// four at a time with all loads issued up front, keeping an online
// log-sum-exp state: running max m, running sum S = sum r_p exp(-m) and the
// running weighted row sum.  Row groups, then warps (through shared memory),
// merge their states with the same rescale rule, so the result is the
// formula above up to rounding.
#include <math_constants.h>

#include "pa_device.cuh"

namespace pa {

constexpr int kReduceThreads = 256;

// Online LSE state of one lane: max, normaliser and up to 8 columns.
struct LseAcc {
  float m, S;
  float4 a[2];
};

__device__ __forceinline__ void lse_merge(LseAcc &x, float m2, float S2, const float4 (&a2)[2],
                                          int per_lane) {
  const float M = fmaxf(x.m, m2);
  const float f1 = M == -CUDART_INF_F ? 0.f : expf(x.m - M);
  const float f2 = M == -CUDART_INF_F ? 0.f : expf(m2 - M);
  x.S = x.S * f1 + S2 * f2;
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (k < per_lane) {
      x.a[k].x = x.a[k].x * f1 + a2[k].x * f2;
      x.a[k].y = x.a[k].y * f1 + a2[k].y * f2;
      x.a[k].z = x.a[k].z * f1 + a2[k].z * f2;
      x.a[k].w = x.a[k].w * f1 + a2[k].w * f2;
    }
  x.m = M;
}

template <typename OutT>
__global__ void __launch_bounds__(kReduceThreads)
    pa_v2_reduce_kernel(const __grid_constant__ ReduceParams p) {
  // With programmatic dependent launch this kernel may start before Phase 1
  // has finished; wait here until all of its results are visible.
  pdl_wait_primary();

  __shared__ float4 part_a[kReduceThreads / 32][64];  // [warp][<= 256 cols / 4]
  __shared__ float part_m[kReduceThreads / 32], part_S[kReduceThreads / 32];
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
  bool done = !live;  // sequences that Phase 1 finished are left alone
  if (live) {
    int L = p.seq_lens[s];
    L = L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);  // Phase 1 reported it
    np = (L + p.partition_size - 1) / p.partition_size;
    // With the combine fused (fuse_limit > 0) Phase 1 also wrote the zeros
    // of empty sequences; without it, this kernel writes them.
    if (p.fuse_limit > 0 && np <= p.fuse_limit) {
      done = true;
      np = 0;
    }
  }
  const size_t row0 = ((size_t)s * p.num_heads + h) * p.max_parts;
  const float *ml = p.max_logits + row0;
  const float *es = p.exp_sums + row0;

  const int c4 = ncols / 4;           // float4s per row
  const int lpr = c4 < 32 ? c4 : 32;  // lanes per row
  const int rpi = 32 / lpr;           // rows per warp iteration
  const int per_lane = c4 / lpr;      // float4s per lane (1 or 2)
  const int sub = lane / lpr, cl = lane % lpr;
  const float *tmp = p.tmp_out + row0 * D + col0 + 4 * cl;
  const int stride = wph * rpi;

  LseAcc acc;
  acc.m = -CUDART_INF_F;
  acc.S = 0.f;
  acc.a[0] = acc.a[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  int i = wig * rpi + sub;
  for (; i < np; i += 4 * stride) {
    float lm[4], le[4];
    float4 v[4][2];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = i + u * stride;
      const bool ok = r < np;
      lm[u] = ok ? __ldcg(ml + r) : -CUDART_INF_F;
      le[u] = ok ? __ldcg(es + r) : 0.f;
#pragma unroll
      for (int k = 0; k < 2; ++k)
        v[u][k] = (ok && k < per_lane)
                      ? __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)r * D + 4 * lpr * k))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float M = acc.m;
#pragma unroll
    for (int u = 0; u < 4; ++u) M = fmaxf(M, lm[u]);
    const float f = acc.m == -CUDART_INF_F ? 0.f : expf(acc.m - M);
    acc.S *= f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      acc.a[k].x *= f;
      acc.a[k].y *= f;
      acc.a[k].z *= f;
      acc.a[k].w *= f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = lm[u] == -CUDART_INF_F ? 0.f : expf(lm[u] - M) * le[u];
      acc.S += w;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        acc.a[k].x = fmaf(w, v[u][k].x, acc.a[k].x);
        acc.a[k].y = fmaf(w, v[u][k].y, acc.a[k].y);
        acc.a[k].z = fmaf(w, v[u][k].z, acc.a[k].z);
        acc.a[k].w = fmaf(w, v[u][k].w, acc.a[k].w);
      }
    }
    acc.m = M;
  }
  // merge the row groups of the warp (lanes with the same column chunk)
  for (int off = lpr; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, acc.m, off);
    const float S2 = __shfl_xor_sync(0xffffffffu, acc.S, off);
    float4 a2[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      a2[k].x = __shfl_xor_sync(0xffffffffu, acc.a[k].x, off);
      a2[k].y = __shfl_xor_sync(0xffffffffu, acc.a[k].y, off);
      a2[k].z = __shfl_xor_sync(0xffffffffu, acc.a[k].z, off);
      a2[k].w = __shfl_xor_sync(0xffffffffu, acc.a[k].w, off);
    }
    lse_merge(acc, m2, S2, a2, 2);
  }
  // merge the warps of the group
  if (wph > 1) {
    if (sub == 0) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        if (k < per_lane) part_a[warp][cl + lpr * k] = acc.a[k];
      if (lane == 0) {
        part_m[warp] = acc.m;
        part_S[warp] = acc.S;
      }
    }
    __syncthreads();
    if (wig != 0) return;
    if (sub == 0)
      for (int w2 = 1; w2 < wph; ++w2) {
        float4 a2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k)
          a2[k] = k < per_lane ? part_a[warp + w2][cl + lpr * k] : make_float4(0.f, 0.f, 0.f, 0.f);
        lse_merge(acc, part_m[warp + w2], part_S[warp + w2], a2, per_lane);
      }
  }
  if (done || sub != 0) return;
  OutT *out = static_cast<OutT *>(p.out) + ((size_t)s * p.num_heads + h) * D + col0;
  const float inv = np > 0 ? 1.f / acc.S : 0.f;  // np == 0: empty sequence -> zeros
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (k < per_lane) {
      OutT *o = out + 4 * (cl + lpr * k);
      o[0] = from_float<OutT>(acc.a[k].x * inv);
      o[1] = from_float<OutT>(acc.a[k].y * inv);
      o[2] = from_float<OutT>(acc.a[k].z * inv);
      o[3] = from_float<OutT>(acc.a[k].w * inv);
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
