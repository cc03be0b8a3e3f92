// Internal launch parameters shared by the host planner and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kTileTokens = 16;     // tokens per warp tile (mma M / N extent)
constexpr int kPanelBytes = 128;    // TMA box width: one 128-byte swizzle span
constexpr int kStatusBytes = 256;   // status block at the head of the workspace
constexpr uint64_t kDefaultWaitLimitNs = 1000000000ull;  // 1 s
constexpr uint64_t kDrainLimitNs = 1000000000ull;        // drain of own copies
constexpr int kFuseLimitMax = 16;  // most partitions a fused combine handles

// Parameters of the attention kernel (Phase 1 of V2, or V1).
struct AttnParams {
  const void *query;           // [B][H][D]
  void *out;                   // [B][H][D] (V1) — dtype
  const int32_t *block_tables; // [B][max_blocks_per_seq]
  const int32_t *seq_lens;     // [B]
  float *max_logits;           // [B][H][max_parts]   (V2)
  float *exp_sums;             // [B][H][max_parts]   (V2)
  float *tmp_out;              // [B][H][max_parts][D] (V2)
  int *status;                 // workspace status word
  int *sched;                  // [0] next work item, [1] CTAs finished
  int sched_reset_later;       // 1: the Phase 2 launch that follows zeroes sched;
                               // 0: the last CTA out does
  int num_seqs, num_heads, num_kv_heads, group;  // group = H / Hkv
  int block_size, log2_block_size;
  int unit_rows, log2_unit_rows;  // rows per TMA box: min(block_size, stage tokens)
  int max_blocks_per_seq, max_seq_len, num_blocks;
  int range_tokens;   // tokens per work item: partition_size (V2) or max_seq_len (V1)
  int max_parts;      // partitions per (seq, head) in the workspace layout
  int part_begin, part_end;  // V2: partitions [part_begin, part_end) of each
                             // sequence only (0, INT_MAX: all of them)
  int write_partials; // 1: V2 Phase 1 outputs, 0: V1 final output
  int fuse_limit;     // V2: sequences of at most this many partitions get the
                      // cross-partition combine inside this kernel (0 = none)
  int *group_count;   // V2 fused combine: finished partitions per (seq, kv head)
  // Query chunks (pa_chunks_forward): the chunk of sequence s is query rows
  // q_start[s] .. q_start[s+1]-1, its last tokens; an item takes up to
  // chunk_tokens of them (x group rows <= 16).  Null q_start: one query per
  // sequence.
  const int32_t *q_start;
  int num_rows;
  int chunk_tokens;
  int *row_limit;     // V2 chunk mode: keys visible to each query row (for Phase 2)
  int num_stages;
  int cluster;        // tcgen05 chunk kernel: CTAs of a thread-block cluster (1: none)
  int debug_flags;
  float scale_log2;   // scale * log2(e)
  uint64_t wait_limit_ns;
};

// Parameters of the Phase 2 (log-sum-exp) reduce kernel.
struct ReduceParams {
  void *out;
  const float *max_logits, *exp_sums, *tmp_out;
  const int32_t *seq_lens;
  int *status;
  int num_seqs, num_heads, head_size, max_parts, partition_size, max_seq_len;
  int fuse_limit;      // sequences of at most this many partitions were
                       // finished by Phase 1 (0 = none)
  const int *row_limit; // chunk mode: keys visible to each query row (null: the
                        // sequence's length, rows being sequences)
  int cols_per_cta;    // columns of one task: head_size / (column split)
  int warps_per_head;  // warps of the team that serves one task: 1, 2, 4 or 8
  int *sched;          // non-null: Phase 1's work counters, zeroed after the wait
};

// Parameters of the kernel that reads pa_forward_host's inputs from pinned
// host memory: segment i is units[i] elements of width[i] bytes (16 or 4)
// from src[i] (a device-side address of host memory) to dst[i] (staging).
constexpr int kStageInSegments = 3;
struct StageInParams {
  const void *src[kStageInSegments];
  void *dst[kStageInSegments];
  long long units[kStageInSegments];
  int width[kStageInSegments];
};

enum MathKind { kMathSimt = 1, kMathTensor = 2 };

// Static description of one compiled attention kernel.
struct AttnKernelInfo {
  const void *fn;     // __global__ function
  int consumer_warps; // warps computing; one more warp produces (TMA)
  int stage_tokens;   // tokens of one ring stage
                      // (consumer_warps * kTileTokens, or 64 for row-owning warps)
  int max_group;      // largest H / Hkv it handles (query chunks: rows of an item)
  int umma;           // tcgen05 kernels (their own layouts and launches): 1 the
                      // query-chunk kernel (rows on M), 2 the kernel of small
                      // items (keys on M)
};

// Query chunks on tcgen05: D 128, 16-bit, more than 16 rows per KV head.  A
// 128-row item costs about the same however many of its rows are live, and
// the two-n-tile kernel needs one 16-row item per 16 rows: measured on GB300
// (the 256-sequence cache, 8 heads a group) the tcgen05 kernel is ahead from
// 32 rows (0.260 against 0.293 ms at 4 tokens, 0.258 against 0.426 at 8) and
// behind at 16 (0.258 against 0.193 ms).
inline bool umma_chunk_ok(int head_size, int group, long long max_rows) {
  return head_size == 128 && group >= 1 && 128 % group == 0 && max_rows > 16;
}
// clustered: the instantiation launched in thread-block clusters
AttnKernelInfo attn_kernel_umma_chunk(int dtype_bf16, bool clustered);
size_t umma_chunk_smem_bytes();
// Items of at most 16 query rows on tcgen05, the keys on the MMA's M (decode
// with up to 16 heads a KV head, short query chunks): D 128, 16-bit.
inline bool umma_keys_ok(int head_size, long long item_rows) {
  return head_size == 128 && item_rows >= 1 && item_rows <= 16;
}
AttnKernelInfo attn_kernel_umma_keys(int dtype_bf16);
size_t umma_keys_smem_bytes();
constexpr int kUmmaStagesHost = 2;
constexpr int kUmmaTmemColsHost = 256;     // tensor-memory columns per CTA (of 512 per SM)
constexpr int kUmmaKeysTmemColsHost = 64;  // the same for the kernel of small items

// Dynamic shared memory the attention kernel needs for `stages` stages (the
// kernel's carve-up, in order: the ring of stages, each its K and V bytes and
// a query slot padded to 1024 bytes; stage headers; mbarriers; flags;
// CUDA-core tables).  The consumer warps merge inside an item's last stage, so
// the merge takes no bytes of its own.
inline size_t attn_smem_bytes(int head_size, int elt, int stage_tokens, int consumer_warps,
                              int max_group, int stages, bool simt) {
  const size_t kv = (size_t)stage_tokens * head_size * elt * 2;
  const size_t qslot = ((size_t)max_group * head_size * elt + 1023) & ~(size_t)1023;
  size_t ring = (kv + qslot) * stages;
  size_t headers = 32 * (size_t)stages;
  size_t bars = 8 * (2 * (size_t)stages + 2);  // full, empty, never-set, consumer barrier
  size_t flags = 16 + 16;                      // flags + alignment
  size_t simt_extra = 0;
  if (simt) {
    simt_extra = (size_t)max_group * (head_size + 8) * 4 +               // q (fp32)
                 (size_t)consumer_warps * kTileTokens * max_group * 4;  // p tiles
  }
  return 1024 /* alignment slack */ + ring + headers + bars + flags + simt_extra;
}

// Kernel tables, one per translation unit (see pa_attn_*.cu).
AttnKernelInfo attn_kernel_tensor_bf16(int head_size, int group);
AttnKernelInfo attn_kernel_tensor_f16(int head_size, int group);
AttnKernelInfo attn_kernel_simt_f32(int head_size, int group);
AttnKernelInfo attn_kernel_simt_bf16(int head_size, int group);
AttnKernelInfo attn_kernel_simt_f16(int head_size, int group);
AttnKernelInfo attn_kernel_chunk_bf16(int head_size, int group, int max_rows);
AttnKernelInfo attn_kernel_chunk_f16(int head_size, int group, int max_rows);
const void *reduce_kernel(int dtype, int float4_per_thread);
// Phase 2 for rows whose partials fit in a few KB (bulk copies into shared
// memory, four warps a CTA, one row a warp at a time)
constexpr int kReduceRowsThreads = 128;
const void *reduce_rows_kernel(int dtype);
size_t reduce_rows_smem_bytes(int max_parts, int head_size);
const void *stage_in_kernel();

}  // namespace pa
