// Phase 2 of V2: cross-partition log-sum-exp reduce, per the
// "paged_attention_v2" commit note (project_6, commit 96f4baf "Dockerfile",
// section "Implementation", "Phase 2: Cross-partition reduction"):
//   M     = max_p max_logits[p]
//   r_p   = exp(max_logits[p] - M) * exp_sums[p]
//   out   = sum_p (r_p / sum_p' r_p') * tmp_out[p]
//
// A task is one (sequence, query head) and a slice of its columns.  A team
// of W warps (1, 2, 4 or 8) serves one task at a time; a 256-thread CTA holds
// 8 / W teams, and the grid is no larger than what is resident on the GPU at
// once, so teams loop over tasks (persistent).  Inside a team, C lanes cover
// the slice's float4 columns of one partition and the team's 32 * W / C
// "slots" take the partitions slot, slot + S, ... (S slots); each thread
// issues the loads of up to NB of its partitions at once and folds them into
// an online log-sum-exp state: running max m, running sum S = sum r_p e^-m
// and the running weighted row.  The slots' states are then merged with the
// same rescale rule (shuffles inside a warp, shared memory across the team):
// the common maximum first, then each state rescaled once and summed, so
// the result is the formula above up to rounding.  The host sizes W and the
// column split so that one batch covers the longest sequence's partitions.
#include <math_constants.h>

#include "pa_device.cuh"

namespace pa {

constexpr int kReduceThreads = 256;

// Online LSE state of one thread: max, normaliser and VPT float4 columns.
template <int VPT>
struct LseAcc {
  float m, S;
  float4 a[VPT];
};

// Barrier of the W warps of team g (named barrier 1 + g; 0 is __syncthreads).
__device__ __forceinline__ void team_sync(int g, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(nthreads) : "memory");
}

template <typename OutT, int VPT>
__global__ void __launch_bounds__(kReduceThreads, 4)
    pa_v2_reduce_kernel(const __grid_constant__ ReduceParams p) {
  constexpr int NB = VPT == 1 ? 4 : 2;  // partitions per thread per batch of loads (no spills at 64 registers)
  __shared__ float4 part_a[kReduceThreads / 32][32 * VPT];  // [warp][slice float4s]
  __shared__ float part_m[kReduceThreads / 32], part_S[kReduceThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = p.warps_per_head;
  const int teams = (kReduceThreads / 32) / W;
  const int g = warp / W, wig = warp % W;  // team in CTA, warp in team
  const int D = p.head_size;
  const int ncols = p.cols_per_cta;
  const int C = ncols / (4 * VPT);  // lanes per partition row (<= 32)
  const int spw = 32 / C;           // partition slots per warp
  const int slot = wig * spw + lane / C, cl = lane % C;
  const int S = W * spw;            // partitions advance by S per round
  const int dsplit = D / ncols;
  const long long ntasks = (long long)p.num_seqs * p.num_heads * dsplit;
  const long long tstride = (long long)gridDim.x * teams;
  long long task = (long long)blockIdx.x * teams + g;

  // seq_lens is an input, not a Phase 1 result: read the first task's before
  // waiting for Phase 1 (programmatic dependent launch), later ones a task
  // ahead.
  // (in chunk mode the counts are Phase 1 results: read after the wait)
  int np_next = task < ntasks && !p.row_limit ? partitions_of_row(p, task / dsplit) : 0;
  pdl_wait_primary();
  // Phase 1 has completed: its work counters go back to zero for the next call
  if (p.sched && blockIdx.x == 0 && threadIdx.x == 0) {
    p.sched[0] = 0;
    p.sched[1] = 0;
  }
  if (p.row_limit && task < ntasks) np_next = partitions_of_row(p, task / dsplit);
  pdl_launch_dependents();  // the next kernel still waits for this grid to complete

  for (; task < ntasks; task += tstride) {
    const long long row = task / dsplit;  // s * num_heads + h
    const int col0 = (int)(task % dsplit) * ncols;
    int np = np_next;
    if (task + tstride < ntasks) np_next = partitions_of_row(p, (task + tstride) / dsplit);
    // With the combine fused into Phase 1 (fuse_limit > 0) it finished these
    // sequences, empty ones included; without it, this kernel writes the
    // zeros of empty sequences.
    const bool done = p.fuse_limit > 0 && np <= p.fuse_limit;
    if (done) np = 0;

    const float *ml = p.max_logits + row * p.max_parts;
    const float *es = p.exp_sums + row * p.max_parts;
    const float *tmp = p.tmp_out + row * p.max_parts * D + col0 + 4 * cl;

    LseAcc<VPT> acc;
    acc.m = -CUDART_INF_F;
    acc.S = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k) acc.a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i = slot; i < np; i += NB * S) {
      float lm[NB], le[NB];
      float4 v[NB][VPT];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int r = i + u * S;
        const bool ok = r < np;
        lm[u] = ok ? __ldcg(ml + r) : -CUDART_INF_F;
        le[u] = ok ? __ldcg(es + r) : 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          v[u][k] = ok ? __ldcg(reinterpret_cast<const float4 *>(tmp + (size_t)r * D + 4 * C * k))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float M = acc.m;
#pragma unroll
      for (int u = 0; u < NB; ++u) M = fmaxf(M, lm[u]);
      const float f = acc.m == -CUDART_INF_F ? 0.f : expf(acc.m - M);
      acc.S *= f;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        acc.a[k].x *= f;
        acc.a[k].y *= f;
        acc.a[k].z *= f;
        acc.a[k].w *= f;
      }
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const float w = lm[u] == -CUDART_INF_F ? 0.f : expf(lm[u] - M) * le[u];
        acc.S += w;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          acc.a[k].x = fmaf(w, v[u][k].x, acc.a[k].x);
          acc.a[k].y = fmaf(w, v[u][k].y, acc.a[k].y);
          acc.a[k].z = fmaf(w, v[u][k].z, acc.a[k].z);
          acc.a[k].w = fmaf(w, v[u][k].w, acc.a[k].w);
        }
      }
      acc.m = M;
    }
    // Merge the slots of the warp (lanes with the same column chunk), then
    // the warps of the team: first the common maximum, then one rescale per
    // state and plain sums, so that no merge waits on the one before it.
    float M = acc.m;
    for (int off = C; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    {
      const float f = M == -CUDART_INF_F ? 0.f : expf(acc.m - M);
      acc.S *= f;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        acc.a[k].x *= f;
        acc.a[k].y *= f;
        acc.a[k].z *= f;
        acc.a[k].w *= f;
      }
      acc.m = M;
    }
    for (int off = C; off < 32; off <<= 1) {
      acc.S += __shfl_xor_sync(0xffffffffu, acc.S, off);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        acc.a[k].x += __shfl_xor_sync(0xffffffffu, acc.a[k].x, off);
        acc.a[k].y += __shfl_xor_sync(0xffffffffu, acc.a[k].y, off);
        acc.a[k].z += __shfl_xor_sync(0xffffffffu, acc.a[k].z, off);
        acc.a[k].w += __shfl_xor_sync(0xffffffffu, acc.a[k].w, off);
      }
    }
    if (W > 1) {
      if (lane < C) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) part_a[warp][cl + C * k] = acc.a[k];
        if (lane == 0) {
          part_m[warp] = acc.m;
          part_S[warp] = acc.S;
        }
      }
      team_sync(g, W * 32);
      if (wig == 0 && lane < C) {
        float Mt = acc.m;
#pragma unroll
        for (int w2 = 1; w2 < 8; ++w2)
          if (w2 < W) Mt = fmaxf(Mt, part_m[warp + w2]);
        const float f0 = Mt == -CUDART_INF_F ? 0.f : expf(acc.m - Mt);
        acc.S *= f0;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          acc.a[k].x *= f0;
          acc.a[k].y *= f0;
          acc.a[k].z *= f0;
          acc.a[k].w *= f0;
        }
#pragma unroll
        for (int w2 = 1; w2 < 8; ++w2) {
          if (w2 >= W) break;
          const float f = Mt == -CUDART_INF_F ? 0.f : expf(part_m[warp + w2] - Mt);
          acc.S = fmaf(part_S[warp + w2], f, acc.S);
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            const float4 a2 = part_a[warp + w2][cl + C * k];
            acc.a[k].x = fmaf(a2.x, f, acc.a[k].x);
            acc.a[k].y = fmaf(a2.y, f, acc.a[k].y);
            acc.a[k].z = fmaf(a2.z, f, acc.a[k].z);
            acc.a[k].w = fmaf(a2.w, f, acc.a[k].w);
          }
        }
        acc.m = Mt;
      }
    }
    if (!done && wig == 0 && lane < C) {
      OutT *out = static_cast<OutT *>(p.out) + row * D + col0;
      const float inv = np > 0 ? 1.f / acc.S : 0.f;  // np == 0: empty sequence -> zeros
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        store4(out + 4 * (cl + C * k), acc.a[k].x * inv, acc.a[k].y * inv, acc.a[k].z * inv,
               acc.a[k].w * inv);
      }
    }
    if (W > 1) team_sync(g, W * 32);  // the shared slots are free for the next task
  }
}

const void *reduce_kernel(int dtype, int vpt) {
  if (vpt == 1) {
    switch (dtype) {
      case 0: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<float, 1>);
      case 1: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__nv_bfloat16, 1>);
      case 2: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__half, 1>);
    }
  } else if (vpt == 2) {
    switch (dtype) {
      case 0: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<float, 2>);
      case 1: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__nv_bfloat16, 2>);
      case 2: return reinterpret_cast<const void *>(&pa_v2_reduce_kernel<__half, 2>);
    }
  }
  return nullptr;
}

}  // namespace pa
