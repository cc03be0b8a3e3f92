// Paged decode attention kernel: V1 (whole sequence per work item) and
// Phase 1 of V2 (one partition per work item), per the "paged_attention_v2"
// commit note (project_6, commit 96f4baf "Dockerfile", section
// "Implementation", "Phase 1: Per-partition attention").
//
// A work item is one (sequence, KV head, token range): the range is a
// partition of partition_size tokens (V2) or the whole sequence (V1).  The
// item computes all G query heads that share the KV head, so every K/V byte
// of the range crosses HBM once.
//
// The kernel is persistent: a grid of about (CTAs per SM) x (SMs) CTAs pulls
// items from a device-wide counter until none are left.  Warp roles in a CTA:
//   warp NW        producer: takes the next item (atomic counter), locates it
//                  (a warp scan over seq_lens for V2), reads its block-table
//                  entries and issues TMA tile loads of whole KV pages
//                  (128-byte swizzled panels) into a ring of shared-memory
//                  stages, plus a bulk copy of the group's queries with the
//                  item's first stage.  Each stage carries a small header
//                  (item, first token, flags) written before its mbarrier
//                  arrive.  The producer runs ahead into the next item while
//                  the consumers finish the current one.
//   warps 0..NW-1  consumers: each takes 16 tokens of every stage and keeps
//                  its own online-softmax state (running max, sum, output).
//                  After an item's last stage they merge their states (the
//                  same log-sum-exp combine as Phase 2) and write either the
//                  final output (V1) or the partition's max_logits /
//                  exp_sums / normalised tmp_output (V2 Phase 1).
// The work counter goes back to zero for the next launch on the workspace:
// the Phase 2 kernel resets it after its wait, else the last CTA to finish
// does.
//
// Every wait is bounded (%globaltimer); a wait that runs out records
// PA_ERR_DEVICE_TIMEOUT, the CTA lets its own in-flight copies land, and
// returns without writing results.
#pragma once

#include <math_constants.h>

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kDebugStallConsumers = 1;

constexpr int kStageFirst = 1;  // first stage of an item (carries the queries)
constexpr int kStageLast = 2;   // last stage of an item (consumers write results)
constexpr int kStageEnd = 4;    // no more items: consumers leave

// Header of one ring stage, written by the producer before the stage's
// mbarrier arrive and read by the consumers after their wait.
struct StageInfo {
  int s, kvh, part;  // the work item
  int tok0;          // first token of the stage
  int tok_end;       // end of the item's token range
  int flags;         // kStage*
  int np;            // partitions of the item's sequence (V2)
  int pad;
};

// Largest partition count whose cross-partition combine may run inside this
// kernel: its scratch holds 3 floats per (head, partition).
constexpr int kFuseCap = kFuseLimitMax;

// Geometry of one K (or V) stage buffer as TMA writes it:
//   [unit][panel][unit_rows][128 bytes]
// where a unit is unit_rows consecutive tokens of one page, a panel is a
// 128-byte slice of the head dimension, and inside every 1024 bytes the
// 16-byte chunk index is XOR-ed with the row index mod 8 (TMA 128B swizzle).
struct StageGeom {
  int log2_unit_rows;
  int unit_rows_mask;
  uint32_t panel_bytes;  // unit_rows * 128
  uint32_t unit_bytes;   // panels * unit_rows * 128

  __device__ __forceinline__ uint32_t row_addr(uint32_t base, int tok) const {
    return base + (uint32_t)(tok >> log2_unit_rows) * unit_bytes +
           ((uint32_t)(tok & unit_rows_mask) << 7);
  }
  // 16-byte chunk `chunk` of the row that starts at row_addr(.., tok).
  __device__ __forceinline__ uint32_t chunk_addr(uint32_t row, int tok, int chunk) const {
    return row + (uint32_t)(chunk >> 3) * panel_bytes + ((uint32_t)((chunk & 7) ^ (tok & 7)) << 4);
  }
};

// ---------------------------------------------------------------------------
// Tensor-core math (bf16 / f16): per 16-token tile,
//   S^T[16 tok][8 heads] = K[16 tok][D] . Q^T[D][8 heads]     (mma m16n8k16)
//   O^T[D][8 heads]     += V^T[D][16 tok] . P^T[16 tok][8 heads]
// Q^T fragments stay in registers for the whole range; K comes in through
// ldmatrix, V through ldmatrix.trans, and P^T is turned from the S^T
// accumulator layout into the B-operand layout with movmatrix.trans.
// Accumulation is fp32.  P is rounded to the input type for the PV product
// and the running sum adds the rounded values, so the weights used and the
// normaliser agree.
template <typename T, int D, int NT, bool CHUNK = false>
struct TensorMath {
  static constexpr int KS = D / 16;
  static constexpr int GMAX = 8 * NT;
  // Query chunks (several tokens of a sequence per item, causal among them):
  // the columns are (token, head) rows, each with its own key limit.
  static constexpr bool kChunk = CHUNK;
  static constexpr bool kRowOwning = false;
  uint32_t qf[NT][KS][2];
  float o[NT][KS][4];
  float m[NT][2];
  float l[NT][2];
  int lim[CHUNK ? NT : 1][2];  // chunk mode: keys at or past lim[..] are hidden

  // Start an item: queries of the group from shared memory ([rows][D], input
  // type), fresh softmax state.  Chunk mode: row r belongs to the item's
  // (r / group)-th token, which sees the keys below lim_base + r / group + 1.
  __device__ __forceinline__ void begin_item(const uint8_t *q_smem, int rows, int lane, int,
                                             int lim_base = 0, int group = 1) {
    const T *q = reinterpret_cast<const T *>(q_smem);
    if constexpr (CHUNK) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = nt * 8 + 2 * (lane & 3) + j;  // this thread's S^T columns
          lim[nt][j] = c < rows ? lim_base + c / group + 1 : 0x7fffffff;
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + (lane >> 2);
      const bool live = h < rows;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const T *src = q + h * D + ks * 16 + 2 * (lane & 3);
        qf[nt][ks][0] = live ? *reinterpret_cast<const uint32_t *>(src) : 0u;
        qf[nt][ks][1] = live ? *reinterpret_cast<const uint32_t *>(src + 8) : 0u;
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[nt][mt][j] = 0.f;
      m[nt][0] = m[nt][1] = -CUDART_INF_F;
      l[nt][0] = l[nt][1] = 0.f;
    }
  }

  __device__ __forceinline__ void bind(float *, float *) {}

  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, const StageGeom &g, int tok0,
                                       int valid, int lane, float scale_log2, int abs0 = 0) {
    const int mi = lane >> 3, r = lane & 7;
    // ---- S^T = K Q^T
    // Two accumulators per n-tile (even / odd k-steps) halve the chain of
    // dependent mma instructions.
    float sacc[NT][4], sacc2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) sacc[nt][j] = sacc2[nt][j] = 0.f;
    {
      const int tokA = tok0 + r + ((mi & 1) << 3);
      const uint32_t rowA = g.row_addr(kbase, tokA);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(g.chunk_addr(rowA, tokA, 2 * ks + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (ks & 1)
            MmaOp<T>::run(sacc2[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
          else
            MmaOp<T>::run(sacc[nt], a0, a1, a2, a3, qf[nt][ks][0], qf[nt][ks][1]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) sacc[nt][j] += sacc2[nt][j];
    }
    // ---- online softmax on the tile (log2 domain)
    const int t_lo = lane >> 2, t_hi = t_lo + 8;
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float x0 = sacc[nt][0] * scale_log2, x1 = sacc[nt][1] * scale_log2;
      float x2 = sacc[nt][2] * scale_log2, x3 = sacc[nt][3] * scale_log2;
      if (t_lo >= valid) x0 = x1 = -CUDART_INF_F;
      if (t_hi >= valid) x2 = x3 = -CUDART_INF_F;
      if constexpr (CHUNK) {  // causal limits of the (token, head) columns
        const int k_lo = abs0 + t_lo, k_hi = abs0 + t_hi;
        if (k_lo >= lim[nt][0]) x0 = -CUDART_INF_F;
        if (k_lo >= lim[nt][1]) x1 = -CUDART_INF_F;
        if (k_hi >= lim[nt][0]) x2 = -CUDART_INF_F;
        if (k_hi >= lim[nt][1]) x3 = -CUDART_INF_F;
      }
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
      // chunk mode: a column that has seen no key yet keeps m = -inf; take
      // its exponents against 0 so that they come out 0, not NaN
      const float mb0 = CHUNK && mn0 == -CUDART_INF_F ? 0.f : mn0;
      const float mb1 = CHUNK && mn1 == -CUDART_INF_F ? 0.f : mn1;
      const float al0 = exp2f(m[nt][0] - mb0), al1 = exp2f(m[nt][1] - mb1);
      const uint32_t plo = MmaOp<T>::pack(exp2f(x0 - mb0), exp2f(x1 - mb1));
      const uint32_t phi = MmaOp<T>::pack(exp2f(x2 - mb0), exp2f(x3 - mb1));
      const float2 flo = MmaOp<T>::unpack(plo), fhi = MmaOp<T>::unpack(phi);
      l[nt][0] = l[nt][0] * al0 + (flo.x + fhi.x);
      l[nt][1] = l[nt][1] * al1 + (flo.y + fhi.y);
      // no column of the n-tile raised its max: every factor is exp2(0) = 1
      // and the rescale would change no bit
      const bool same = mn0 == m[nt][0] && mn1 == m[nt][1];
      m[nt][0] = mn0;
      m[nt][1] = mn1;
      pb[nt][0] = movmatrix_trans(plo);
      pb[nt][1] = movmatrix_trans(phi);
      if (!__all_sync(0xffffffffu, same)) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[nt][mt][0] *= al0;
          o[nt][mt][1] *= al1;
          o[nt][mt][2] *= al0;
          o[nt][mt][3] *= al1;
        }
      }
    }
    // ---- rows past the end of the range hold stale or foreign data: zero
    // them so that 0-weight x NaN cannot reach the accumulator.
    if (valid < 16) {
      constexpr int CPR = D * (int)sizeof(T) / 16;  // chunks per row
      const int n = (16 - valid) * CPR;
      for (int c = lane; c < n; c += 32) {
        const int tok = tok0 + valid + c / CPR;
        const uint32_t a = g.chunk_addr(g.row_addr(vbase, tok), tok, c % CPR);
        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(a), "r"(0u) : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
    }
    // ---- O^T += V^T P^T
    {
      const int tokB = tok0 + r + ((mi >> 1) << 3);
      const uint32_t rowB = g.row_addr(vbase, tokB);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(g.chunk_addr(rowB, tokB, 2 * mt + (mi & 1)), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          MmaOp<T>::run(o[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
  }

  // End of an item, step 1: this warp's max and sum per head -> m_w/l_w [GMAX].
  __device__ __forceinline__ void stats(float *m_w, float *l_w, int lane) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = l[nt][j];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (lane < 4) {
          const int h = nt * 8 + 2 * lane + j;
          m_w[h] = m[nt][j];
          l_w[h] = v;
        }
      }
  }

  // Step 2: with every warp's stats in m_s/l_s [NW][GMAX], scale this warp's
  // O by exp2(m_w - M) / L (log-sum-exp weight and final normaliser) and
  // store it to o_w [GMAX][D+4]; the sum over warps is then the output.
  // row_ml (one warp passes it): the merged (M, L) of every row, for the
  // partials.
  __device__ __forceinline__ void store_scaled(float *o_w, const float *m_s, const float *l_s,
                                               int nw, int lane, float2 *row_ml) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float f[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = nt * 8 + 2 * (lane & 3) + j;
        float M = -CUDART_INF_F;
        for (int w = 0; w < nw; ++w) M = fmaxf(M, m_s[w * GMAX + h]);
        float L = 0.f;
        for (int w = 0; w < nw; ++w) L += l_s[w * GMAX + h] * exp2f(m_s[w * GMAX + h] - M);
        if (row_ml && lane < 4) row_ml[h] = make_float2(M, L);
        f[j] = exp2f(m[nt][j] - M) / L;  // 0 for a warp that saw no token
        if constexpr (CHUNK) {
          if (!(L > 0.f)) f[j] = 0.f;  // a column that saw no key at all: zeros
        }
      }
      const int h0 = nt * 8 + 2 * (lane & 3);
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d = mt * 16 + (lane >> 2);
        o_w[h0 * (D + 4) + d] = o[nt][mt][0] * f[0];
        o_w[(h0 + 1) * (D + 4) + d] = o[nt][mt][1] * f[1];
        o_w[h0 * (D + 4) + d + 8] = o[nt][mt][2] * f[0];
        o_w[(h0 + 1) * (D + 4) + d + 8] = o[nt][mt][3] * f[1];
      }
    }
  }
};


// ---------------------------------------------------------------------------
// Query chunks with row-owning warps (bf16 / f16, D 64 or 128).  An item is
// up to 16 x NWC of the chunk's (token, head) rows; consumer warp w owns rows
// [16 w, 16 w + 16) of it and runs them over every key of each 64-key stage:
//   S[16 rows][64 keys] = Q[16][D] . K^T              (mma m16n8k16, A = Q)
//   O[16 rows][D]      += P[16][64 keys] . V[64][D]    (A = P, taken straight
//                                                       from S's accumulators)
// A row's statistics live in the four lanes of a quad, and no warp holds
// another's rows, so an item ends without a cross-warp merge: each warp
// writes its rows from registers, and the stage goes back to the producer as
// soon as its tile is done.  Each warp's tile carries 8 (S) and 16 (O)
// independent accumulator chains.  Accumulation is fp32; P is rounded to the
// input type for the PV product and the row sum adds the rounded values.
template <typename T, int D, int NWC>
struct RowMath {
  static constexpr bool kChunk = true;
  static constexpr bool kRowOwning = true;
  static constexpr int ST = 64;          // keys per stage
  // keys of one softmax step: at D = 128 a stage is taken in two halves, so
  // that S and P of only 32 keys are live beside O and the queries and a
  // thread fits in 168 registers (two CTAs an SM)
  static constexpr int SK = D >= 128 ? 32 : 64;
  static constexpr int KS = D / 16;      // k-steps of S = Q K^T
  static constexpr int NK = SK / 8;      // key n-tiles of S
  static constexpr int ND = D / 8;       // d n-tiles of O
  static constexpr int KK = SK / 16;     // key k-steps of O += P V
  static constexpr int GMAX = 16 * NWC;  // rows of an item
  uint32_t qa[KS][4];  // A fragments of this warp's 16 query rows
  float o[ND][4];
  float m[2], l[2];    // rows r0 = lane / 4 and r0 + 8 of the warp: running max (log2), sum
  int lim[2];          // keys at or past lim[i] are hidden from row i (0: not a row of the item)

  // Start an item: rows [0, rows) of the q slot (row-major [GMAX][D], input
  // type) are the item's; row r is the (r / group)-th token's head r % group,
  // which sees the keys below lim_base + r / group + 1.
  __device__ __forceinline__ void begin_item(const uint8_t *q_smem, int rows, int lane, int warp,
                                             int lim_base, int group) {
    // ldmatrix.x4 per k-step: lanes 0-15 give rows 0-15 at the k-step's first
    // 8 columns, lanes 16-31 the same rows at its last 8 (A layout a0..a3)
    const uint32_t a_row = smem_u32(q_smem) + (uint32_t)(16 * warp + (lane & 15)) * (D * sizeof(T)) +
                           (uint32_t)(lane >> 4) * 16u;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
      ldsm_x4(a_row + (uint32_t)ks * 32u, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r = 16 * warp + (lane >> 2) + 8 * i;
      lim[i] = r < rows ? lim_base + r / group + 1 : 0;
      m[i] = -CUDART_INF_F;
      l[i] = 0.f;
    }
#pragma unroll
    for (int d = 0; d < ND; ++d)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[d][j] = 0.f;
  }

  // One stage: keys [abs0, abs0 + valid) of the item, at positions 0.. of
  // the stage buffers, SK keys at a time.
  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, const StageGeom &g, int,
                                       int valid, int lane, float scale_log2, int abs0) {
#pragma unroll
    for (int k0 = 0; k0 < ST; k0 += SK)
      if (k0 < valid) step(kbase, vbase, g, k0, valid - k0, lane, scale_log2, abs0 + k0);
  }

  // Keys [abs0, abs0 + valid) at positions key0.. of the stage buffers (only
  // the first SK of them).
  __device__ __forceinline__ void step(uint32_t kbase, uint32_t vbase, const StageGeom &g, int key0,
                                       int valid, int lane, float scale_log2, int abs0) {
    const int mi = lane >> 3, r = lane & 7, q4 = lane & 3;
    // ---- S = Q K^T: matrix mi of an ldmatrix.x4 is keys 16 jp + r + 8 (mi >> 1)
    // at the k-step's 16-byte chunk 2 ks + (mi & 1): the B fragments of key
    // n-tiles 2 jp and 2 jp + 1
    float s[NK][4];
#pragma unroll
    for (int j = 0; j < NK; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[j][e] = 0.f;
    {
      uint32_t krow[NK / 2];
      int ktok[NK / 2];
#pragma unroll
      for (int jp = 0; jp < NK / 2; ++jp) {
        ktok[jp] = key0 + 16 * jp + r + ((mi >> 1) << 3);
        krow[jp] = g.row_addr(kbase, ktok[jp]);
      }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks)
#pragma unroll
        for (int jp = 0; jp < NK / 2; ++jp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(g.chunk_addr(krow[jp], ktok[jp], 2 * ks + (mi & 1)), b0, b1, b2, b3);
          MmaOp<T>::run(s[2 * jp], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          MmaOp<T>::run(s[2 * jp + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
    }
    // ---- online softmax per row (log2 domain); hidden keys get -inf
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < NK; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int kr = 8 * j + 2 * q4 + (e & 1);  // key within the step
        float x = s[j][e] * scale_log2;
        if (kr >= valid || abs0 + kr >= lim[e >> 1]) x = -CUDART_INF_F;
        s[j][e] = x;
        if (e < 2)
          mx0 = fmaxf(mx0, x);
        else
          mx1 = fmaxf(mx1, x);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    // a row that has seen no key yet keeps m = -inf: its exponents are taken
    // against 0 so that they come out 0, not NaN
    const float mb0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
    const float mb1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
    const float al0 = exp2f(m[0] - mb0), al1 = exp2f(m[1] - mb1);
    // P as the A fragments of the PV product: k-step kk takes key n-tiles
    // 2 kk (a0: row r0, a1: row r0 + 8) and 2 kk + 1 (a2, a3)
    uint32_t pa[KK][4];
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int j = 2 * kk + hf;
        const uint32_t lo = MmaOp<T>::pack(exp2f(s[j][0] - mb0), exp2f(s[j][1] - mb0));
        const uint32_t hi = MmaOp<T>::pack(exp2f(s[j][2] - mb1), exp2f(s[j][3] - mb1));
        const float2 fl = MmaOp<T>::unpack(lo), fh = MmaOp<T>::unpack(hi);
        ls0 += fl.x + fl.y;
        ls1 += fh.x + fh.y;
        pa[kk][2 * hf] = lo;
        pa[kk][2 * hf + 1] = hi;
      }
    l[0] = l[0] * al0 + ls0;
    l[1] = l[1] * al1 + ls1;
    m[0] = mn0;
    m[1] = mn1;
    if (al0 != 1.f || al1 != 1.f) {
#pragma unroll
      for (int d = 0; d < ND; ++d) {
        o[d][0] *= al0;
        o[d][1] *= al0;
        o[d][2] *= al1;
        o[d][3] *= al1;
      }
    }
    // ---- O += P V: matrix mi of an ldmatrix.x4.trans is keys 16 kk + r +
    // 8 (mi & 1) at d chunk 2 jd + (mi >> 1): the B fragments of d n-tiles
    // 2 jd and 2 jd + 1.  Keys past `valid` may hold stale bytes (NaN x 0
    // would reach O): their V halves are cleared in the fragments.
    const int k0 = 2 * q4;
#pragma unroll
    for (int kk = 0; kk < KK; ++kk) {
      const int tk = key0 + 16 * kk + r + ((mi & 1) << 3);
      const uint32_t vrow = g.row_addr(vbase, tk);
      uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;  // keys 16 kk + k0 (+1), and + 8
      if (valid < SK) {
        const int a = 16 * kk + k0;
        keep_lo = (a < valid ? 0x0000ffffu : 0u) | (a + 1 < valid ? 0xffff0000u : 0u);
        keep_hi = (a + 8 < valid ? 0x0000ffffu : 0u) | (a + 9 < valid ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int jd = 0; jd < ND / 2; ++jd) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(g.chunk_addr(vrow, tk, 2 * jd + (mi >> 1)), b0, b1, b2, b3);
        b0 &= keep_lo;
        b2 &= keep_lo;
        b1 &= keep_hi;
        b3 &= keep_hi;
        MmaOp<T>::run(o[2 * jd], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
        MmaOp<T>::run(o[2 * jd + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
      }
    }
  }

  // End of an item: this warp's rows from registers.  V2 writes the
  // partition's max logit (natural-log units), exp-sum and normalised output
  // row; V1 the output rows.  Rows of the item start at query row row0; row
  // r is token r / group, head kvh * group + r % group.
  __device__ __forceinline__ void finish(const AttnParams &p, int row0, int kvh, int part,
                                         int rows, int lane, int warp) const {
    const int q4 = lane & 3;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float lt = l[i];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      const int r = 16 * warp + (lane >> 2) + 8 * i;
      if (r >= rows) continue;
      const size_t orow = ((size_t)row0 + r / p.group) * p.num_heads + (size_t)kvh * p.group +
                          r % p.group;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      if (p.write_partials) {
        const size_t prow = orow * p.max_parts + part;
        float *dst = p.tmp_out + prow * D + 2 * q4;
#pragma unroll
        for (int d = 0; d < ND; ++d)
          *reinterpret_cast<float2 *>(dst + 8 * d) = make_float2(o[d][2 * i] * inv, o[d][2 * i + 1] * inv);
        if (q4 == 0) {
          p.max_logits[prow] = m[i] * 0.69314718055994530942f;  // back to natural-log units
          p.exp_sums[prow] = lt;
        }
      } else {
        T *dst = static_cast<T *>(p.out) + orow * D + 2 * q4;
#pragma unroll
        for (int d = 0; d < ND; ++d)
          *reinterpret_cast<uint32_t *>(dst + 8 * d) = MmaOp<T>::pack(o[d][2 * i] * inv, o[d][2 * i + 1] * inv);
      }
    }
  }
};

// ---------------------------------------------------------------------------
// CUDA-core fp32 math (any element type; the only path for f32).  Lane
// (tok = lane % 16, half = lane / 16) forms the dot products of one token
// with all G query heads over half of D; the halves are summed with one
// shuffle.  For PV each lane owns D/32 output columns of every head and
// reads the tile's probabilities from a small shared-memory table.
template <typename T, int D, int GMAX>
struct SimtMath {
  static constexpr bool kChunk = false;  // query chunks run on the tensor path only
  static constexpr bool kRowOwning = false;
  static constexpr int ELT = sizeof(T);
  static constexpr int CPR = D * ELT / 16;  // 16-byte chunks per row
  static constexpr int EPC = 16 / ELT;      // elements per chunk
  static constexpr int DPL = D / 32;        // output columns per lane
  static constexpr int QP = D + 8;          // q row pitch (floats)
  float acc[GMAX][DPL];
  float m[GMAX];
  float l[GMAX];
  const float *q_s;
  float *p_s;

  __device__ __forceinline__ static int qidx(int g, int d) {
    return g * QP + d + (d >= D / 2 ? 4 : 0);
  }

  __device__ __forceinline__ void bind(float *q_smem, float *p_smem) {
    q_s = q_smem;
    p_s = p_smem;
  }

  // Start an item: all consumer threads widen the group's queries ([G][D],
  // input type, in shared memory) into the fp32 table q_s (the caller then
  // synchronises the consumer warps).
  __device__ __forceinline__ void begin_item(const uint8_t *q_smem, int group, int,
                                             int ncons, int = 0, int = 1) {
    const T *q = reinterpret_cast<const T *>(q_smem);
    for (int i = threadIdx.x; i < GMAX * D; i += ncons) {
      const int g = i / D, d = i % D;
      const_cast<float *>(q_s)[qidx(g, d)] = g < group ? to_float(q[g * D + d]) : 0.f;
    }
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
      m[g] = -CUDART_INF_F;
      l[g] = 0.f;
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[g][j] = 0.f;
    }
  }

  __device__ __forceinline__ static void widen(const uint4 &c, float (&f)[EPC]) {
    if constexpr (ELT == 4) {
      chunk_to_float(c, f);
    } else if constexpr (sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value) {
      chunk_to_float_bf16(c, f);
    } else {
      chunk_to_float_f16(c, f);
    }
  }

  // This lane's DPL output columns of token `tok` (row address `row`).
  __device__ __forceinline__ void load_v(const StageGeom &g, uint32_t row, int tok, int lane,
                                         float (&v)[DPL]) const {
    constexpr int BYTES = DPL * ELT;  // 4, 8, 16 or 32
    const int byte0 = lane * BYTES;
    if constexpr (BYTES >= 16) {
#pragma unroll
      for (int c = 0; c < BYTES / 16; ++c) {
        uint4 raw;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                     : "r"(g.chunk_addr(row, tok, byte0 / 16 + c)));
        float f[EPC];
        widen(raw, f);
#pragma unroll
        for (int e = 0; e < EPC; ++e) v[c * EPC + e] = f[e];
      }
    } else {
      const uint32_t a = g.chunk_addr(row, tok, byte0 / 16) + (uint32_t)(byte0 % 16);
      uint32_t w[BYTES / 4];
      if constexpr (BYTES == 8) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "r"(a));
      } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[0]) : "r"(a));
      }
#pragma unroll
      for (int i = 0; i < BYTES / 4; ++i) {
        if constexpr (ELT == 4) {
          v[i] = __uint_as_float(w[i]);
        } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
          v[2 * i] = __uint_as_float(w[i] << 16);
          v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        } else {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
        }
      }
    }
  }

  __device__ __forceinline__ void tile(uint32_t kbase, uint32_t vbase, const StageGeom &g, int tok0,
                                       int valid, int lane, float scale_log2, int = 0) {
    const int tok = lane & 15, half = lane >> 4;
    float dot[GMAX];
#pragma unroll
    for (int gg = 0; gg < GMAX; ++gg) dot[gg] = 0.f;
    {
      const uint32_t row = g.row_addr(kbase, tok0 + tok);
      // Kept rolled: unrolled, every q load is loop-invariant and the
      // compiler would pin the whole query group in registers.
#pragma unroll 1
      for (int c = 0; c < CPR / 2; ++c) {
        const int chunk = half * (CPR / 2) + c;
        uint4 raw;
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                     : "r"(g.chunk_addr(row, tok0 + tok, chunk)));
        float kf[EPC];
        widen(raw, kf);
        const int d0 = chunk * EPC;
#pragma unroll
        for (int gg = 0; gg < GMAX; ++gg) {
#pragma unroll
          for (int e = 0; e < EPC; e += 4) {
            const float4 qv = *reinterpret_cast<const float4 *>(&q_s[qidx(gg, d0 + e)]);
            dot[gg] = fmaf(qv.x, kf[e], dot[gg]);
            dot[gg] = fmaf(qv.y, kf[e + 1], dot[gg]);
            dot[gg] = fmaf(qv.z, kf[e + 2], dot[gg]);
            dot[gg] = fmaf(qv.w, kf[e + 3], dot[gg]);
          }
        }
      }
    }
#pragma unroll
    for (int gg = 0; gg < GMAX; ++gg) {
      float x = dot[gg] + __shfl_xor_sync(0xffffffffu, dot[gg], 16);
      x = tok < valid ? x * scale_log2 : -CUDART_INF_F;
      float mx = x;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[gg], mx);
      const float al = exp2f(m[gg] - mn);
      const float pv = exp2f(x - mn);
      l[gg] = l[gg] * al + pv;
      m[gg] = mn;
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[gg][j] *= al;
      if (half == 0) p_s[tok * GMAX + gg] = pv;
    }
    __syncwarp();
    // ---- PV over the valid tokens only
    for (int t = 0; t < valid; ++t) {
      const int tk = tok0 + t;
      float v[DPL];
      load_v(g, g.row_addr(vbase, tk), tk, lane, v);
#pragma unroll
      for (int gg = 0; gg < GMAX; ++gg) {
        const float pg = p_s[t * GMAX + gg];
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[gg][j] = fmaf(pg, v[j], acc[gg][j]);
      }
    }
    __syncwarp();
  }

  __device__ __forceinline__ void stats(float *m_w, float *l_w, int lane) {
#pragma unroll
    for (int gg = 0; gg < GMAX; ++gg) {
      float v = l[gg];
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) {
        m_w[gg] = m[gg];
        l_w[gg] = v;
      }
    }
  }

  __device__ __forceinline__ void store_scaled(float *o_w, const float *m_s, const float *l_s,
                                               int nw, int lane, float2 *row_ml) {
#pragma unroll
    for (int gg = 0; gg < GMAX; ++gg) {
      float M = -CUDART_INF_F;
      for (int w = 0; w < nw; ++w) M = fmaxf(M, m_s[w * GMAX + gg]);
      float L = 0.f;
      for (int w = 0; w < nw; ++w) L += l_s[w * GMAX + gg] * exp2f(m_s[w * GMAX + gg] - M);
      if (row_ml && lane == 0) row_ml[gg] = make_float2(M, L);
      const float f = exp2f(m[gg] - M) / L;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o_w[gg * (D + 4) + lane * DPL + j] = acc[gg][j] * f;
    }
  }
};

// Register cap per thread: three CTAs of (NW + 1) warps must fit in one SM,
// i.e. at most four warps' registers per SM sub-partition (16K registers).
// Groups of more than 8 heads (and query chunks) keep twice the
// accumulators: at 4 consumer warps they are capped at 168, so that two CTAs
// (10 warps, three on some sub-partitions) fit: 3 x 168 x 32 <= 16K, while at
// 192 only two warps fit per sub-partition and the SM holds one CTA.  With
// fewer warps they are left uncapped.
template <int NW, int GMAX>
constexpr int kernel_max_regs() {
  return GMAX > 8 ? (NW == 4 ? 168 : 255) : (NW == 4 ? 128 : (NW == 2 ? 168 : 255));
}

// Row-owning query chunks: two CTAs of 5 warps put 3 warps on some
// schedulers, so 168 registers a thread at most (at 200 an SM held one CTA,
// one consumer warp per scheduler).
template <class Math, int NW, int GMAX>
constexpr int attn_max_regs() {
  return Math::kRowOwning ? (NW == 4 ? 168 : 255) : kernel_max_regs<NW, GMAX>();
}

// Tokens of one ring stage: 16 per consumer warp, or 64 for row-owning warps
// (which each run every key of the stage).
template <class Math, int NW>
constexpr int stage_tokens() {
  if constexpr (Math::kRowOwning)
    return Math::ST;
  else
    return NW * kTileTokens;
}

// ---------------------------------------------------------------------------
template <typename T, int D, int NW, int GMAX, class Math, bool SIMT>
__global__ void __launch_bounds__((NW + 1) * 32, 1) __maxnreg__((attn_max_regs<Math, NW, GMAX>()))
    pa_attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int ELT = sizeof(T);
  constexpr int ST = stage_tokens<Math, NW>();  // tokens per stage
  constexpr int ROW_BYTES = D * ELT;
  constexpr int NPANELS = ROW_BYTES / kPanelBytes;
  constexpr int HALF_BYTES = ST * ROW_BYTES;  // K (or V) bytes of one stage
  constexpr int NCONS = NW * 32;
  constexpr int QBYTES = GMAX * D * ELT;      // queries of one item
  // A stage is its K and V bytes followed by its query slot (padded to keep
  // the next stage's TMA destinations 1024-byte aligned for the 128B swizzle).
  constexpr int QSLOT = (QBYTES + 1023) & ~1023;
  constexpr int STAGE_BYTES = 2 * HALF_BYTES + QSLOT;
  // The consumer warps merge their states in an item's last stage (K, V and
  // query bytes, dead by then: the queries were taken into registers or the
  // fp32 table when the item began); the stage goes back to the producer
  // after the merge.
  constexpr int MERGE_BYTES_STATE = NW * GMAX * (D + 4) * 4 + NW * GMAX * 2 * 4 + GMAX * 8;
  constexpr int MERGE_BYTES_FUSE = (3 * GMAX * kFuseCap + 4) * 4;  // fused combine scratch
  static_assert(Math::kRowOwning ||
                    (MERGE_BYTES_STATE <= STAGE_BYTES && MERGE_BYTES_FUSE <= STAGE_BYTES),
                "the merge fits in one stage");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NST = p.num_stages;

  // ---- shared memory carve-up (sizes mirrored by attn_smem_bytes)
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *ring = smem;  // NST x [K | V | queries]
  StageInfo *info = reinterpret_cast<StageInfo *>(ring + (size_t)NST * STAGE_BYTES);
  uint64_t *bars = reinterpret_cast<uint64_t *>(info + NST);
  volatile int *flags = reinterpret_cast<volatile int *>(bars + 2 * NST + 2);
  float *simt_q = reinterpret_cast<float *>(
      (reinterpret_cast<uintptr_t>(flags) + 16 + 15) & ~uintptr_t(15));
  float *simt_p = simt_q + GMAX * (D + 8);
  const uint32_t ring_u32 = smem_u32(ring);
  const uint32_t full0 = smem_u32(bars), empty0 = full0 + 8 * NST, never = full0 + 16 * NST;
  const uint32_t cons_bar = never + 8;  // consumer-warp barrier (bounded waits)

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, NW);
    }
    mbar_init(never, 1);
    mbar_init(cons_bar, NW);
    flags[0] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Launched with programmatic dependent launch: everything above touched
  // only shared memory; wait here until the previous kernel in the stream has
  // finished and its writes are visible (it may have produced the queries or
  // the cache, or still be reading what this kernel writes).
  pdl_wait_primary();

  const StageGeom geom{p.log2_unit_rows, p.unit_rows - 1, (uint32_t)p.unit_rows * kPanelBytes,
                       (uint32_t)(NPANELS * p.unit_rows * kPanelBytes)};
  const uint64_t limit = p.wait_limit_ns;
  const int qbytes = p.group * D * ELT;

  if (warp == NW) {
    // ======================= producer warp =======================
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
      // The block-table entries of a CTA's first item are read right after
      // seq_lens (which locates the item): fetch them into L2 meanwhile, so
      // that the first K/V copy waits one DRAM round trip less.  V1: the
      // item's sequence is blockIdx / Hkv.  V2: the first items of all CTAs
      // lie at the head of the table, so CTA b fetches its b-th 128-byte line.
      const char *bt0 = reinterpret_cast<const char *>(p.block_tables);
      if (!p.write_partials && !Math::kChunk) {
        const int s0 = (int)blockIdx.x / p.num_kv_heads;
        if (s0 < p.num_seqs && p.max_blocks_per_seq > 0)
          prefetch_l2(bt0 + (size_t)s0 * p.max_blocks_per_seq * sizeof(int32_t));
      } else {
        const size_t bytes = (size_t)p.num_seqs * p.max_blocks_per_seq * sizeof(int32_t);
        if ((size_t)blockIdx.x * 128 < bytes) prefetch_l2(bt0 + (size_t)blockIdx.x * 128);
      }
    }
    const int U = p.unit_rows;
    const int units_per_stage = ST / U;
    // Every K/V byte is read once: let those lines leave L2 first.
    const uint64_t kv_policy = l2_policy_evict_first();
    // V2 locates an item through the running count of items per sequence;
    // the cursor (a chunk of 32 sequences, scanned once) only moves forward
    // because every CTA takes items in increasing order.
    int cs = 0, cbase = 0, c_cnt = 0, c_incl = 0, c_L = 0, c_total = 0;
    int c_qs = 0, c_n = 0, c_nrg = 0;  // chunk mode: first query row, chunk tokens, row groups
    bool c_loaded = false;
    auto load_chunk = [&]() {
      const int sl = cs + lane;
      c_L = 0;
      if (sl < p.num_seqs) {
        c_L = __ldg(p.seq_lens + sl);
        if (c_L < 0 || c_L > p.max_seq_len) {
          report(p.status, kStatusBadInput);
          c_L = c_L < 0 ? 0 : p.max_seq_len;
        }
      }
      // With the cross-partition combine fused into this kernel, an empty
      // sequence gets one item per KV head that writes zeros; lanes past the
      // last sequence count none.
      const int c_np = (c_L + p.range_tokens - 1) / p.range_tokens;
      // V2 may be asked for a range of partitions only (context parallelism:
      // the rest belong to other GPUs): [part_begin, part_end) of each sequence
      const int c_nr = max(0, min(c_np, p.part_end) - p.part_begin);
      c_cnt = sl >= p.num_seqs ? 0
                               : p.num_kv_heads * (c_np == 0 && p.fuse_limit > 0 ? 1 : c_nr);
      if constexpr (Math::kChunk) {
        // the sequence's query chunk: its last c_n tokens, query rows from c_qs;
        // items: (KV head, partition, group of chunk_tokens tokens)
        c_qs = 0;
        c_n = 0;
        if (sl < p.num_seqs) {
          c_qs = __ldg(p.q_start + sl);
          const int qe = __ldg(p.q_start + sl + 1);
          c_n = qe - c_qs;
          if (c_qs < 0 || c_n < 0 || c_n > c_L || qe > p.num_rows) {
            report(p.status, kStatusBadInput);  // its rows get no items
            c_n = 0;
          }
        }
        c_nrg = (c_n + p.chunk_tokens - 1) / p.chunk_tokens;
        c_cnt = sl >= p.num_seqs ? 0 : p.num_kv_heads * c_np * c_nrg;
      }
      c_incl = c_cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, c_incl, off);
        if (lane >= off) c_incl += t;
      }
      c_total = __shfl_sync(0xffffffffu, c_incl, 31);
      c_loaded = true;
    };
    // The first item of a CTA is its own index; later ones come from the
    // counter, offset by the number of CTAs that take items.  Lane 0 issues
    // the atomic one item ahead and the value is broadcast only when that
    // item is located.
    int takers = (int)gridDim.x;
    int item = blockIdx.x;
    if (p.write_partials && p.num_seqs <= 32) {
      // A batch of at most 32 sequences is counted in one chunk, so every CTA
      // knows the number of items N.  When N is not a multiple of the grid
      // (say 1.7 items per CTA) the CTAs that take one more item than the
      // rest set the pace; so only ceil(N / ceil(N / grid)) CTAs take items,
      // each the same number, and the others leave at once.
      load_chunk();
      const int per = (c_total + (int)gridDim.x - 1) / (int)gridDim.x;
      takers = per > 0 ? (c_total + per - 1) / per : 0;
      if ((int)blockIdx.x >= takers) item = c_total;  // past the last item: none
    }
    // Predicated in PTX so that nothing consumes the result until the item
    // ends: every CTA takes its first item at the same moment, and a select
    // on the result (lane == 0 ? atomicAdd(..) : 0) would hold the producer
    // for the whole round trip of atomics queued on one address.
    auto grab_issue = [&]() -> int { return atomic_add_lane0(p.sched, lane); };
    auto grab_value = [&](int raw) -> int {
      return takers + __shfl_sync(0xffffffffu, raw, 0);
    };
    int i = 0;  // stages issued by this CTA
    bool ok = true;
    while (true) {
      // ---- locate the item: (s, kvh, part, L)
      int s = 0, kvh = 0, part = 0, L = 0, np_s = 1;
      int nrg = 0, qs = 0, n_s = 0, rg = 0;  // chunk mode
      bool found = false;
      if (item < 0) {  // a corrupted work counter: stop rather than guess
        if (lane == 0) report(p.status, kStatusBadInput);
      } else if (!p.write_partials && !Math::kChunk) {  // V1: Hkv items per sequence, empty ones too
        s = item / p.num_kv_heads;
        if (s < p.num_seqs) {
          found = true;
          kvh = item % p.num_kv_heads;
          L = __ldg(p.seq_lens + s);
          if (L < 0 || L > p.max_seq_len) {
            if (lane == 0) report(p.status, kStatusBadInput);
            L = L < 0 ? 0 : p.max_seq_len;
          }
        }
      } else {
        while (true) {
          if (!c_loaded) load_chunk();
          if (item < cbase + c_total) {
            const unsigned hit = __ballot_sync(0xffffffffu, cbase + c_incl > item);
            const int ls = __ffs(hit) - 1;
            s = cs + ls;
            L = __shfl_sync(0xffffffffu, c_L, ls);
            const int first = cbase + __shfl_sync(0xffffffffu, c_incl - c_cnt, ls);
            np_s = (L + p.range_tokens - 1) / p.range_tokens;
            if constexpr (Math::kChunk) {
              // (KV head, partition, row group); the row groups of one
              // partition are neighbours, so their K/V re-reads hit L2
              nrg = __shfl_sync(0xffffffffu, c_nrg, ls);
              qs = __shfl_sync(0xffffffffu, c_qs, ls);
              n_s = __shfl_sync(0xffffffffu, c_n, ls);
              const int per_head = np_s * nrg;
              kvh = (item - first) / per_head;
              const int rem = (item - first) % per_head;
              part = rem / nrg;
              rg = rem % nrg;
            } else {
              const int nr = max(0, min(np_s, p.part_end) - p.part_begin);
              const int items_per_head = nr > 0 ? nr : 1;
              kvh = (item - first) / items_per_head;
              part = p.part_begin + (item - first) % items_per_head;
            }
            found = s < p.num_seqs;  // always, by the count above; never write past the batch
            break;
          }
          if (cs + 32 >= p.num_seqs) break;
          cs += 32;
          cbase += c_total;
          c_loaded = false;
        }
      }
      if (!found) break;
      // The next item is taken from the counter once this item's first copies
      // are issued: nothing needs it before the item ends, and every CTA
      // reaches this point at about the same moment, so the atomics queue on
      // one address for a while.
      int next_raw = 0;

      const int tok_begin = part * p.range_tokens;
      int tok_end = min(tok_begin + p.range_tokens, L);
      // chunk mode: the item's tokens, its output rows and key limits
      int row0 = 0, rows = 0, lim_base = 0, ntok = 0;
      if constexpr (Math::kChunk) {
        const int t_first = rg * p.chunk_tokens;
        ntok = min(p.chunk_tokens, n_s - t_first);
        rows = ntok * p.group;
        lim_base = L - n_s + t_first;  // keys below lim_base + i + 1 for token i of the group
        row0 = qs + t_first;
        tok_end = min(tok_end, lim_base + ntok);
        // Phase 2 needs each row's count of visible keys: the partition-0
        // items (one per KV head, all equal) record it
        if (part == 0 && p.row_limit)
          for (int t = lane; t < ntok; t += 32) p.row_limit[row0 + t] = lim_base + t + 1;
        if (tok_end <= tok_begin) {  // the partition lies past every token of the group
          item = grab_value(grab_issue());
          continue;
        }
      }
      if (tok_end <= tok_begin) {  // empty sequence (V1, or V2 with the fused combine): zeros
        T *o = static_cast<T *>(p.out) + ((size_t)s * p.num_heads + (size_t)kvh * p.group) * D;
        for (int e = lane; e < p.group * D; e += 32) o[e] = from_float<T>(0.f);
        item = grab_value(grab_issue());
        continue;
      }
      // A window of 64 block-table entries: lane j holds pages win0+j (cur)
      // and win0+32+j (nxt); it slides by 32 pages when a stage reaches nxt.
      const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
      const int last_page = (tok_end - 1) >> p.log2_block_size;
      auto load_entry = [&](int page) -> int {
        return (page >= 0 && page <= last_page) ? __ldg(bt + page) : -1;
      };
      int win0 = tok_begin >> p.log2_block_size;
      int cur = load_entry(win0 + lane);
      int nxt = load_entry(win0 + 32 + lane);
      const int n_st = (tok_end - tok_begin + ST - 1) / ST;
      for (int j = 0; j < n_st; ++j) {
        const int st = i % NST;
        if (i >= NST) {
          bool w = true;
          if (lane == 0) w = mbar_wait(empty0 + 8 * st, ((i / NST) - 1) & 1, limit, flags);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
        }
        const int stage_tok0 = tok_begin + j * ST;
        const int n_units = min(units_per_stage, (tok_end - stage_tok0 + U - 1) / U);
        const int tok = stage_tok0 + lane * U;
        const int rel = ((lane < n_units ? tok : stage_tok0) >> p.log2_block_size) - win0;
        const int a = __shfl_sync(0xffffffffu, cur, rel & 31);
        const int b = __shfl_sync(0xffffffffu, nxt, rel & 31);
        int y = -1;
        if (lane < n_units) {
          const int blk = rel < 32 ? a : b;
          if ((unsigned)blk >= (unsigned)p.num_blocks) {
            report(p.status, kStatusBadInput);
          } else {
            y = (blk * p.num_kv_heads + kvh) * p.block_size + (tok & (p.block_size - 1));
          }
        }
        const unsigned valid_mask = __ballot_sync(0xffffffffu, y >= 0);
        const bool first = j == 0;
        if (lane == 0) {
          StageInfo &h = info[st];
          h.s = s;
          h.kvh = kvh;
          h.part = part;
          h.tok0 = stage_tok0;
          h.tok_end = tok_end;
          h.flags = (first ? kStageFirst : 0) | (j == n_st - 1 ? kStageLast : 0);
          h.np = np_s;
          const uint32_t q_in = Math::kChunk ? (uint32_t)(ntok * qbytes) : (uint32_t)qbytes;
          if constexpr (Math::kChunk) {
            h.s = row0;     // first output row
            h.np = rows;    // (token, head) rows
            h.pad = lim_base;
          }
          mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)__popc(valid_mask) * U * ROW_BYTES * 2 +
                                                    (first ? q_in : 0u));
        }
        __syncwarp();
        if (y >= 0) {
          const uint32_t kdst = ring_u32 + (uint32_t)st * STAGE_BYTES + (uint32_t)lane * geom.unit_bytes;
          const uint32_t vdst = kdst + HALF_BYTES;
          // one copy per page and tensor: all panels of the unit's rows
          if constexpr (Math::kChunk) {  // the next row group re-reads these pages: keep them
            tma_load_3d(kdst, &tmap_k, 0, y, 0, full0 + 8 * st);
            tma_load_3d(vdst, &tmap_v, 0, y, 0, full0 + 8 * st);
          } else {
            tma_load_3d_hint(kdst, &tmap_k, 0, y, 0, full0 + 8 * st, kv_policy);
            tma_load_3d_hint(vdst, &tmap_v, 0, y, 0, full0 + 8 * st, kv_policy);
          }
        }
        if constexpr (Math::kChunk) {
          // one copy per token: its G heads are contiguous
          for (int t = lane; first && t < ntok; t += 32) {
            const T *q = static_cast<const T *>(p.query) +
                         ((size_t)(row0 + t) * p.num_heads + (size_t)kvh * p.group) * D;
            bulk_load(ring_u32 + (uint32_t)st * STAGE_BYTES + 2 * HALF_BYTES + (uint32_t)(t * qbytes), q,
                      (uint32_t)qbytes, full0 + 8 * st);
          }
        } else if (first && lane == 0) {
          const T *q = static_cast<const T *>(p.query) +
                       ((size_t)s * p.num_heads + (size_t)kvh * p.group) * D;
          bulk_load(ring_u32 + (uint32_t)st * STAGE_BYTES + 2 * HALF_BYTES, q, (uint32_t)qbytes,
                    full0 + 8 * st);
        }
        if (j == 0) next_raw = grab_issue();
        ++i;
        const int next_rel = ((stage_tok0 + ST) >> p.log2_block_size) - win0;
        if (next_rel >= 32) {
          cur = nxt;
          win0 += 32;
          nxt = load_entry(win0 + 32 + lane);
        }
      }
      if (!ok) break;
      item = grab_value(next_raw);
    }
    // Every copy of this CTA is issued: let the next kernel (Phase 2) be
    // scheduled once every CTA has come this far.  Its CTAs then take the
    // SMs that the first CTAs to finish leave free and sit in their own
    // dependency wait, which still holds them until this grid has completed,
    // instead of being launched only after the last CTA's epilogue.
    pdl_launch_dependents();
    if (ok) {  // tell the consumers there is nothing more
      const int st = i % NST;
      if (i >= NST) {
        bool w = true;
        if (lane == 0) w = mbar_wait(empty0 + 8 * st, ((i / NST) - 1) & 1, limit, flags);
        ok = __shfl_sync(0xffffffffu, w, 0);
      }
      if (ok && lane == 0) {
        info[st].flags = kStageEnd;
        mbar_arrive(full0 + 8 * st);
      }
      if (ok) ++i;
    }
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    // Let every copy this CTA started land before the CTA can retire.
    if (lane == 0) {
      const int first = i > NST ? i - NST : 0;
      for (int j = first; j < i; ++j)
        mbar_wait(full0 + 8 * (j % NST), (j / NST) & 1, kDrainLimitNs, nullptr);
    }
    __syncwarp();
  } else if constexpr (Math::kRowOwning) {
    // ============ consumer warps, each owning 16 rows of an item ============
    Math math;
    bool ok = true;
    if (p.debug_flags & kDebugStallConsumers) {
      // Wait on a barrier that nothing releases: the bound must end it.
      ok = mbar_wait(never, 0, limit, flags);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; ok; ++i) {
      const int st = i % NST;
      const bool w = mbar_wait(full0 + 8 * st, (i / NST) & 1, limit, flags);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      const StageInfo h = info[st];
      if (h.flags & kStageEnd) break;
      const uint32_t kbase = ring_u32 + (uint32_t)st * STAGE_BYTES;
      // h.np = the item's rows, h.pad = the key limit base of its first token
      if (h.flags & kStageFirst)
        math.begin_item(ring + (size_t)st * STAGE_BYTES + 2 * HALF_BYTES, h.np, lane, warp, h.pad,
                        p.group);
      math.tile(kbase, kbase + HALF_BYTES, geom, 0, min(ST, h.tok_end - h.tok0), lane,
                p.scale_log2, h.tok0);
      // nothing of the stage is read after the tile: hand it back at once
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      if (h.flags & kStageLast) math.finish(p, h.s, h.kvh, h.part, h.np, lane, warp);
    }
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    pdl_launch_dependents();
  } else {
    // ======================= consumer warps =======================
    Math math;
    math.bind(simt_q, simt_p + warp * kTileTokens * GMAX);
    // Barrier of the NW consumer warps on an mbarrier, so that its wait is
    // bounded like every other wait (a plain bar.sync could not give up).
    int cons_phase = 0;
    auto cons_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(cons_bar);
      const bool w = mbar_wait(cons_bar, cons_phase & 1, limit, flags);
      ++cons_phase;
      return __all_sync(0xffffffffu, w);
    };
    bool ok = true;
    if (p.debug_flags & kDebugStallConsumers) {
      // Wait on a barrier that nothing releases: the bound must end it.
      ok = mbar_wait(never, 0, limit, flags);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; ok; ++i) {
      const int st = i % NST;
      const bool w = mbar_wait(full0 + 8 * st, (i / NST) & 1, limit, flags);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      const StageInfo h = info[st];
      if (h.flags & kStageEnd) break;
      if (h.flags & kStageFirst) {
        if constexpr (Math::kChunk)  // rows = (token, head) pairs; h.pad = first token's key limit
          math.begin_item(ring + (size_t)st * STAGE_BYTES + 2 * HALF_BYTES, h.np, lane, NCONS,
                          h.pad, p.group);
        else
          math.begin_item(ring + (size_t)st * STAGE_BYTES + 2 * HALF_BYTES, p.group, lane, NCONS);
        if constexpr (SIMT) {
          ok = cons_sync();  // the shared fp32 query table is complete
          if (!ok) break;
        }
      }
      const int tile_tok0 = h.tok0 + warp * kTileTokens;
      const int valid = max(0, min(kTileTokens, h.tok_end - tile_tok0));
      if (valid > 0) {
        const uint32_t kbase = ring_u32 + (uint32_t)st * STAGE_BYTES;
        math.tile(kbase, kbase + HALF_BYTES, geom, warp * kTileTokens, valid, lane, p.scale_log2,
                  tile_tok0);
      }
      __syncwarp();
      if (!(h.flags & kStageLast)) {
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
        continue;
      }

      // ---- item done: merge the consumer warps' states (log-sum-exp), write
      uint8_t *mb = ring + (size_t)st * STAGE_BYTES;
      float *m_s = reinterpret_cast<float *>(mb);
      float *l_s = m_s + NW * GMAX;
      float *o_s = l_s + NW * GMAX;
      ok = cons_sync();  // every warp is done with the slot's K/V (and the previous merge)
      if (!ok) break;
      math.stats(m_s + warp * GMAX, l_s + warp * GMAX, lane);
      ok = cons_sync();
      if (!ok) break;
      // warp 0 also records each row's merged (M, L) for the partials
      float2 *row_ml = reinterpret_cast<float2 *>(o_s + (size_t)NW * GMAX * (D + 4));
      math.store_scaled(o_s + (size_t)warp * GMAX * (D + 4), m_s, l_s, NW, lane,
                        warp == 0 ? row_ml : nullptr);
      ok = cons_sync();
      if (!ok) break;
      // out[h][d] = sum over warps of the scaled partial outputs (16 bytes a thread)
      const int G = p.group;
      const size_t head0 = (size_t)h.s * p.num_heads + (size_t)h.kvh * G;
      // output rows of the item: the group's G heads, or in chunk mode h.np
      // (token, head) rows starting at query row h.s
      const int rows = Math::kChunk ? h.np : G;
      for (int idx = threadIdx.x; idx < rows * (D / 4); idx += NCONS) {
        const int hh = idx / (D / 4), d = 4 * (idx % (D / 4));
        const size_t orow = Math::kChunk ? ((size_t)h.s + hh / G) * p.num_heads +
                                               (size_t)h.kvh * G + hh % G
                                         : head0 + hh;
        float4 acc = *reinterpret_cast<const float4 *>(&o_s[(size_t)hh * (D + 4) + d]);
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) {
          const float4 v =
              *reinterpret_cast<const float4 *>(&o_s[((size_t)w2 * GMAX + hh) * (D + 4) + d]);
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        if (p.write_partials) {
          const size_t row = orow * p.max_parts + h.part;
          *reinterpret_cast<float4 *>(p.tmp_out + row * D + d) = acc;
          if (d == 0) {
            const float2 ml = row_ml[hh];
            p.max_logits[row] = ml.x * 0.69314718055994530942f;  // back to natural-log units
            p.exp_sums[row] = ml.y;
          }
        } else {
          store4(static_cast<T *>(p.out) + orow * D + d, acc.x, acc.y, acc.z, acc.w);
        }
      }
      if (!Math::kChunk && p.write_partials && h.np <= p.fuse_limit) {
        // Phase 2 inside Phase 1 for a sequence of few partitions: the last
        // CTA to finish one of them (per KV head) combines them all, with the
        // same log-sum-exp rule as the Phase 2 kernel.
        __threadfence();  // this partition's partials are visible device-wide
        ok = cons_sync();
        if (!ok) break;
        int *cnt = p.group_count + (size_t)h.s * p.num_kv_heads + h.kvh;
        volatile int *last = reinterpret_cast<volatile int *>(mb);
        if (threadIdx.x == 0) {
          // The barrier above ordered every consumer thread's partial writes
          // before this point; the fence and the acq_rel increment publish
          // them device-wide to the CTA that finds the final count.
          __threadfence();
          *last = atomic_add_acq_rel_gpu(cnt, 1) == h.np - 1 ? 1 : 0;
        }
        ok = cons_sync();
        if (!ok) break;
        if (*last) {
          __threadfence();  // the other CTAs' partials are visible to our reads
          const int np = h.np;
          float *mlv = reinterpret_cast<float *>(mb) + 4;  // [G][np]
          float *wts = mlv + GMAX * kFuseCap;              // [G][np]
          float *esv = wts + GMAX * kFuseCap;              // [G][np]
          for (int k = threadIdx.x; k < G * np; k += NCONS) {
            const size_t r = (head0 + k / np) * p.max_parts + k % np;
            mlv[k] = __ldcg(p.max_logits + r);
            esv[k] = __ldcg(p.exp_sums + r);
          }
          ok = cons_sync();
          if (!ok) break;
          for (int hh = threadIdx.x; hh < G; hh += NCONS) {
            float M = -CUDART_INF_F;
            for (int j = 0; j < np; ++j) M = fmaxf(M, mlv[hh * np + j]);
            float sum = 0.f;
            for (int j = 0; j < np; ++j) {
              const float r = esv[hh * np + j] * expf(mlv[hh * np + j] - M);
              wts[hh * np + j] = r;
              sum += r;
            }
            const float inv = 1.f / sum;
            for (int j = 0; j < np; ++j) wts[hh * np + j] *= inv;
          }
          ok = cons_sync();
          if (!ok) break;
          for (int idx = threadIdx.x; idx < G * (D / 4); idx += NCONS) {
            const int hh = idx / (D / 4), d = 4 * (idx % (D / 4));
            const float *src = p.tmp_out + (head0 + hh) * p.max_parts * D + d;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < np; j += 4) {
              float4 v[4];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                v[u] = j + u < np ? __ldcg(reinterpret_cast<const float4 *>(src + (size_t)(j + u) * D))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float w = j + u < np ? wts[hh * np + j + u] : 0.f;
                acc.x = fmaf(w, v[u].x, acc.x);
                acc.y = fmaf(w, v[u].y, acc.y);
                acc.z = fmaf(w, v[u].z, acc.z);
                acc.w = fmaf(w, v[u].w, acc.w);
              }
            }
            store4(static_cast<T *>(p.out) + (head0 + hh) * D + d, acc.x, acc.y, acc.z, acc.w);
          }
          if (threadIdx.x == 0) *cnt = 0;  // ready for the next launch
        }
      }
      {
        // hand the stage back to the producer; its next TMA writes come after
        // our generic-proxy writes
        fence_proxy_async_smem();
        ok = cons_sync();
        if (!ok) break;
      }
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
    }
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    // The producer normally triggered the next kernel already; this covers a
    // producer that left early.  (Triggered at the start instead, Phase 2's
    // CTAs would crowd onto the few SMs that have room while every CTA still
    // streams.)
    pdl_launch_dependents();
  }

  // ---- the work counter goes back to zero for the next launch: in the
  // Phase 2 kernel after its wait, else here, by the last CTA out (a fence
  // and an atomic round trip at the end of every CTA, which the Phase 2 reset
  // takes off the critical path)
  if (!p.sched_reset_later) {
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(p.sched, 0);
        atomicExch(p.sched + 1, 0);
      }
    }
  }
}

template <typename T, int D, int NW, int GMAX, class Math, bool SIMT>
AttnKernelInfo attn_info() {
  return AttnKernelInfo{reinterpret_cast<const void *>(&pa_attn_kernel<T, D, NW, GMAX, Math, SIMT>),
                        NW, stage_tokens<Math, NW>(), GMAX};
}

// Consumer warps per CTA: a stage is NW x 16 tokens; keep it at 32 KB of K+V
// for rows of 256 bytes or more (4, 2 or 1 warps), so that two stages (the
// host's choice for up to 8 heads a group) leave room for three CTAs on an SM.
template <typename T, int D>
constexpr int consumer_warps() {
  return D * (int)sizeof(T) <= 256 ? 4 : (D * (int)sizeof(T) <= 512 ? 2 : 1);
}

template <typename T>
AttnKernelInfo select_tensor(int D, int group) {
  if (group <= 8) {
    switch (D) {
      case 64: return attn_info<T, 64, consumer_warps<T, 64>(), 8, TensorMath<T, 64, 1>, false>();
      case 128: return attn_info<T, 128, consumer_warps<T, 128>(), 8, TensorMath<T, 128, 1>, false>();
      case 256: return attn_info<T, 256, consumer_warps<T, 256>(), 8, TensorMath<T, 256, 1>, false>();
    }
  } else if (group <= 16) {
    switch (D) {
      case 64: return attn_info<T, 64, consumer_warps<T, 64>(), 16, TensorMath<T, 64, 2>, false>();
      case 128: return attn_info<T, 128, consumer_warps<T, 128>(), 16, TensorMath<T, 128, 2>, false>();
      case 256: return attn_info<T, 256, consumer_warps<T, 256>(), 16, TensorMath<T, 256, 2>, false>();
    }
  }
  return AttnKernelInfo{nullptr, 0, 0, 0};
}

// Query chunks on mma.sync.  (At D 128 the host sends chunks of more than 16
// rows per KV head to the tcgen05 kernel, unless told not to; these kernels
// then serve D 64 and 256, up to 16 rows at D 128, and that comparison.)
// Chunks of more than 32 (token, head) rows per KV head run on row-owning
// warps (64 keys a stage, items of 64 rows, four consumer warps) for D 64 and
// 128 when the group divides 64; measured on GB300, that is 1.3x the
// two-n-tile path at 16 and 64 tokens of 8 heads, while 32-row items (two
// consumer warps, one per SM sub-partition) were slower than it at 4 tokens.
// Everything else runs on the two-n-tile tensor path, 16 rows an item.
template <typename T>
AttnKernelInfo select_chunk(int D, int group, int max_rows) {
  if ((D == 64 || D == 128) && 64 % group == 0 && max_rows > 32) {
    switch (D) {
      case 64: return attn_info<T, 64, 4, 64, RowMath<T, 64, 4>, false>();
      case 128: return attn_info<T, 128, 4, 64, RowMath<T, 128, 4>, false>();
    }
  }
  switch (D) {
    case 64: return attn_info<T, 64, consumer_warps<T, 64>(), 16, TensorMath<T, 64, 2, true>, false>();
    case 128: return attn_info<T, 128, consumer_warps<T, 128>(), 16, TensorMath<T, 128, 2, true>, false>();
    case 256: return attn_info<T, 256, consumer_warps<T, 256>(), 16, TensorMath<T, 256, 2, true>, false>();
  }
  return AttnKernelInfo{nullptr, 0, 0, 0};
}

template <typename T, int D>
AttnKernelInfo select_simt_d(int group) {
  constexpr int NW = consumer_warps<T, D>();
  if (group <= 4) return attn_info<T, D, NW, 4, SimtMath<T, D, 4>, true>();
  if (group <= 8) return attn_info<T, D, NW, 8, SimtMath<T, D, 8>, true>();
  if (group <= 16) return attn_info<T, D, NW, 16, SimtMath<T, D, 16>, true>();
  return AttnKernelInfo{nullptr, 0, 0, 0};
}

template <typename T>
AttnKernelInfo select_simt(int D, int group) {
  switch (D) {
    case 64: return select_simt_d<T, 64>(group);
    case 128: return select_simt_d<T, 128>(group);
    case 256: return select_simt_d<T, 256>(group);
  }
  return AttnKernelInfo{nullptr, 0, 0, 0};
}

}  // namespace pa
