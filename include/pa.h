/*
 * libpa — paged decode attention for NVIDIA GB300 (sm_103a), C ABI.
 *
 * One decode step of attention for a batch of sequences whose keys and
 * values live in a paged KV cache addressed through a per-sequence block
 * table.  Two algorithms compute the same result:
 *
 *   V1  one pass over each sequence (one CTA per sequence and KV head);
 *   V2  the partitioned form of the "paged_attention_v2" commit note
 *       (project_6, commit 96f4baf "Dockerfile", section "Implementation"):
 *       Phase 1 computes, for every (sequence, head, partition of
 *       partition_size tokens), the max logit, the exp-sum and the
 *       normalised weighted V sum; Phase 2 merges the partitions with the
 *       log-sum-exp rescale (global max, rescale by exp(m_p - M) times the
 *       partition's exp-sum, normalised sum of the partials).
 *
 * Both reach out[s][h] = softmax_t(scale * q[s][h] . K_t) @ V over the
 * seq_lens[s] tokens of sequence s, kvh = h / (num_heads / num_kv_heads).
 *
 * Layouts (row-major, contiguous, device memory):
 *   query, out         [num_seqs][num_heads][head_size]          (dtype)
 *   key_cache,
 *   value_cache        [num_blocks][num_kv_heads][block_size][head_size]
 *   block_tables       int32 [num_seqs][max_blocks_per_seq]; entry j of row s
 *                      is the physical block holding tokens
 *                      [j*block_size, (j+1)*block_size) of sequence s.
 *                      Entries past ceil(seq_lens[s]/block_size) are never read.
 *   seq_lens           int32 [num_seqs], each in [0, max_seq_len]
 *
 * Ownership: the caller owns every buffer and the stream.  The library
 * allocates no device memory, never synchronises in the forward calls, and
 * only enqueues kernels on `stream` (a cudaStream_t passed as void*; NULL is
 * the legacy default stream).  Calls on one workspace must not overlap.
 *
 * Errors: argument problems are found on the host and returned before any
 * launch.  A failed launch returns PA_ERR_CUDA (see pa_last_cuda_error).
 * Problems in the data, found by the kernels (a block-table entry outside
 * [0, num_blocks), a sequence length outside [0, max_seq_len]) or a bounded
 * device wait that ran out, are recorded in the workspace's status word and
 * read with pa_read_device_status.  Kernels never trap.
 *
 * Supported: dtype f32, bf16, f16 (query, caches and out share it);
 * head_size 64, 128, 256; block_size 8, 16, 32, 64; num_heads / num_kv_heads
 * in [1, 16]; partition_size a multiple of 64 and of block_size, at most
 * 8192.  K and V caches, query and out 16-byte aligned; workspace 256-byte
 * aligned; num_blocks * num_kv_heads * block_size < 2^31.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,         /* bad pointer, size or combination      */
  PA_ERR_UNSUPPORTED = 2,         /* legal but not built (dtype, sizes)    */
  PA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < pa_workspace_bytes  */
  PA_ERR_CUDA = 4,                /* a CUDA runtime call failed            */
  PA_ERR_DEVICE_BAD_INPUT = 5,    /* kernel saw a bad block id / length    */
  PA_ERR_DEVICE_TIMEOUT = 6       /* a bounded device wait ran out         */
} pa_status_t;

typedef enum { PA_DTYPE_F32 = 0, PA_DTYPE_BF16 = 1, PA_DTYPE_F16 = 2 } pa_dtype_t;

typedef enum { PA_VARIANT_AUTO = 0, PA_VARIANT_V1 = 1, PA_VARIANT_V2 = 2 } pa_variant_t;

/* Arithmetic of QK^T and PV.  AUTO: tensor cores (mma, fp32 accumulate) for
 * bf16/f16, CUDA-core fp32 FMA for f32.  SIMT forces the CUDA-core path. */
typedef enum { PA_MATH_AUTO = 0, PA_MATH_SIMT = 1, PA_MATH_TENSOR = 2 } pa_math_t;

/* Optional knobs for pa_forward.  Zero-initialise, then set what you need. */
typedef struct {
  int32_t variant;        /* pa_variant_t                                   */
  int32_t math;           /* pa_math_t                                      */
  int32_t num_stages;     /* KV pipeline depth per CTA, 0 = library choice  */
  int32_t debug_flags;    /* PA_DEBUG_*; 0 in production                    */
  uint64_t wait_limit_ns; /* bound on each device wait, 0 = 1 second        */
  void *phase1_event;     /* cudaEvent_t or NULL: for V2, recorded on the
                             stream between the Phase 1 and Phase 2 kernels
                             (lets a caller time the phases with events)   */
  int32_t ctas_per_sm;    /* persistent CTAs per SM, 0 = as many as fit     */
  int32_t fuse_partitions;/* V2: sequences of at most this many partitions
                             (capped at 16) get the cross-partition combine
                             inside the Phase 1 kernel; 0 (the default) or
                             negative = never: the Phase 2 kernel does it */
  int32_t share_kv;       /* query chunks on the tcgen05 kernel (head_size
                             128, more than 16 rows per KV head) with 256 or
                             more rows per KV head: 1 = the CTAs of the row
                             groups of the same keys form a thread-block
                             cluster (of 2 or 4) and share every K/V stage
                             through multicast copies, so that K/V cross HBM
                             once instead of once per row group; slower on
                             GB300 when HBM is not the limit (measured
                             2.5-10 %); 0 (the default) = each CTA loads its
                             own */
} pa_options_t;

/* Debug: every consumer warp waits on a barrier that nothing ever releases,
 * so the bounded wait runs out and the kernel reports PA_ERR_DEVICE_TIMEOUT
 * (after letting its own in-flight copies land).  Used to test the timeout
 * path without hanging or faulting the GPU. */
#define PA_DEBUG_STALL_CONSUMERS 1

/* Debug: query chunks never take the tcgen05 kernel (chunks of more than 16
 * rows per KV head at head_size 128 then run on the mma.sync row-owning
 * kernel), for comparisons of the two. */
#define PA_DEBUG_NO_TCGEN05 2

/* Option: every call that the tcgen05 kernel of small items can serve takes
 * it: head_size 128, bf16/f16, at most 16 query rows per KV head and item
 * (decode with any group, query chunks of up to 16 / group tokens an item),
 * without the fused combine.  The keys of a stage are the MMA's M and the
 * item's rows its N, so no tensor-core lane computes a missing row.  Off by
 * default: on GB300 the mma.sync kernels are faster on every such workload
 * measured (decode with 16 query heads a KV head: 0.116-0.146 ms against
 * 0.098 ms a step).  PA_DEBUG_NO_TCGEN05 wins over it. */
#define PA_DEBUG_TCGEN05_KEYS 4


/* Bytes of workspace that pa_v2_forward needs (V1 needs only the 256-byte
 * status block).  The partials are the three per-partition arrays that the
 * "paged_attention_v2" commit note (project_6, commit 96f4baf "Dockerfile",
 * section "Implementation", "Phase 1") has Phase 1 store for Phase 2:
 * tmp_output, exp_sums and max_logits, kept in fp32 here.
 * Layout, each part 256-byte aligned, in this order:
 *   status      int32 status word + work-queue counters (a 256-byte block)
 *   max_logits  f32 [num_seqs][num_heads][max_parts]   Phase 1 max logit
 *   exp_sums    f32 [num_seqs][num_heads][max_parts]   sum exp(logit - max)
 *   tmp_out     f32 [num_seqs][num_heads][max_parts][head_size]  normalised
 *   counters    int32 [num_seqs][num_heads]: partitions finished per
 *               (sequence, KV head), for the fused cross-partition combine
 * with max_parts = ceil(max_seq_len / partition_size).  Returns 0 on bad
 * arguments. */
size_t pa_workspace_bytes(int num_seqs, int num_heads, int head_size,
                          int max_seq_len, int partition_size);

/* Byte offsets of the five workspace parts above (offsets[0..4]); returns
 * PA_ERR_INVALID_ARG on bad arguments.  Lets callers read Phase 1 results. */
pa_status_t pa_workspace_layout(int num_seqs, int num_heads, int head_size,
                                int max_seq_len, int partition_size,
                                size_t offsets[5]);

/* Zero a new workspace (enqueued on `stream`).  Call once after allocating
 * it, and again after a call reported a device error.  Kernels only ever
 * set the status word to a nonzero code; the work-queue and combine
 * counters are left at zero by every launch that completes. */
pa_status_t pa_workspace_init(void *workspace, size_t workspace_bytes,
                              void *stream);

/* V1: single pass over each whole sequence, the kernel the "paged_attention_v2"
 * commit note (project_6, commit 96f4baf "Dockerfile") opens with: "V1
 * limitation" describes it as one launch over the entire KV sequence, and its
 * "Integration" list keeps it for sequences of up to 8192 tokens.  Here a
 * work item is one (sequence, KV head), computing all num_heads/num_kv_heads
 * query heads of the group with an online softmax; items are spread over a
 * persistent grid.  partition_size is validated but otherwise unused.
 * The workspace needs >= 256 bytes (its status block). */
pa_status_t pa_v1_forward(void *out, const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_heads,
                          int num_kv_heads, int head_size, int num_blocks,
                          int block_size, int max_blocks_per_seq,
                          int max_seq_len, float scale, int partition_size,
                          int dtype, void *workspace, size_t workspace_bytes,
                          void *stream);

/* V2: the Phase 1 kernel computes every (sequence, KV head, partition) and
 * writes max_logits / exp_sums / tmp_out into the workspace; then the
 * log-sum-exp combine (Phase 2 kernel) writes out.  With
 * pa_options_t.fuse_partitions = n > 0, for a sequence of at most min(n, 16)
 * partitions the last Phase 1 work item of each (sequence, KV head) does
 * that combine instead, and the Phase 2 kernel is launched only if
 * max_seq_len allows a longer sequence.  Same arguments
 * as V1; the workspace must hold pa_workspace_bytes(...) bytes. */
pa_status_t pa_v2_forward(void *out, const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_heads,
                          int num_kv_heads, int head_size, int num_blocks,
                          int block_size, int max_blocks_per_seq,
                          int max_seq_len, float scale, int partition_size,
                          int dtype, void *workspace, size_t workspace_bytes,
                          void *stream);

/* The same call with the V1/V2 choice made by pa_choose_v2 (the device's SM
 * count is queried once per device), or forced through `opts` (NULL = all
 * defaults).  For V2 the workspace must hold pa_workspace_bytes(...). */
pa_status_t pa_forward(void *out, const void *query, const void *key_cache,
                       const void *value_cache, const int32_t *block_tables,
                       const int32_t *seq_lens, int num_seqs, int num_heads,
                       int num_kv_heads, int head_size, int num_blocks,
                       int block_size, int max_blocks_per_seq, int max_seq_len,
                       float scale, int partition_size, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream,
                       const pa_options_t *opts);

/* The two phases of V2 as separate calls, for splitting long sequences over
 * several GPUs (context parallelism).  The "paged_attention_v2" commit note
 * (project_6, commit 96f4baf "Dockerfile", section "Implementation") defines
 * Phase 1 per partition and Phase 2 as the log-sum-exp reduction over a
 * sequence's partitions; the partitions are independent until Phase 2, so
 * GPU r can run Phase 1 over its own range of partitions, the GPUs exchange
 * their partials (one all-gather of max_logits, exp_sums and tmp_out slots,
 * done by the caller), and Phase 2 over the gathered slots gives the
 * single-GPU result.
 *
 * pa_v2_partials: Phase 1 only, for the partitions p with
 *   part_begin <= p < min(part_end, ceil(seq_lens[s] / partition_size))
 * of every sequence s.  It writes their max_logits / exp_sums / tmp_out
 * slots of the workspace (the layout of pa_workspace_layout, sized by
 * pa_workspace_bytes for the whole sequences) and nothing else: slots of
 * other partitions keep their contents, and there is no output.  Block-table
 * entries of pages outside the range are never read, so a GPU that holds only
 * its own range's pages may pass -1 there.  The arguments are those of
 * pa_v2_forward (seq_lens are the whole lengths), without out, plus
 * 0 <= part_begin <= part_end (PA_ERR_INVALID_ARG otherwise; part_end may
 * exceed the partition count).  [0, INT32_MAX) is Phase 1 of pa_v2_forward.
 * Errors as pa_v2_forward; device-detected ones land in this workspace's
 * status word. */
pa_status_t pa_v2_partials(const void *query, const void *key_cache,
                           const void *value_cache, const int32_t *block_tables,
                           const int32_t *seq_lens, int num_seqs, int num_heads,
                           int num_kv_heads, int head_size, int num_blocks,
                           int block_size, int max_blocks_per_seq,
                           int max_seq_len, float scale, int partition_size,
                           int dtype, int part_begin, int part_end,
                           void *workspace, size_t workspace_bytes,
                           void *stream);

/* pa_v2_combine: Phase 2 only.  For every sequence s and head h, the
 * log-sum-exp combine of the slots of partitions 0 .. ceil(seq_lens[s] /
 * partition_size) - 1 in the workspace, written to out[s][h] in dtype (zeros
 * for an empty sequence).  Every one of those slots must hold a Phase 1
 * result (pa_v2_partials here, or slots copied in from other GPUs); the
 * workspace is only read.  seq_lens and out on the device, layouts and the
 * other arguments as pa_v2_forward; head_size, dtype and partition_size are
 * checked as there.  Enqueued on `stream` after whatever precedes it. */
pa_status_t pa_v2_combine(void *out, const int32_t *seq_lens, int num_seqs,
                          int num_heads, int head_size, int max_seq_len,
                          int partition_size, int dtype, const void *workspace,
                          size_t workspace_bytes, void *stream);

/* Multi-token queries over the paged cache: the query of sequence s is a
 * chunk of its LAST n_s = q_start[s+1] - q_start[s] cached tokens (for
 * example draft tokens to verify, or a small prefill chunk whose keys and
 * values are already in the cache), rows q_start[s] .. q_start[s+1]-1 of
 * query and out ([num_rows][num_heads][head_size]).  Chunk token i, at cache
 * position L - n_s + i with L = seq_lens[s], attends causally to the cache
 * tokens [0, L - n_s + i].  The pages give no formula for this; it is the
 * plain causal reading of attention over a paged prefix (the prefill patch
 * of project_6 tunes such a kernel).
 *
 * q_start: device int32 [num_seqs + 1], non-decreasing, q_start[0] = 0,
 * q_start[num_seqs] = num_rows, 0 <= n_s <= min(seq_lens[s], max_chunk).
 * The other arguments as pa_forward (opts->variant picks V1/V2/auto); the V2
 * workspace is sized as pa_workspace_bytes(num_rows, ...).  bf16 and f16 only
 * (PA_ERR_UNSUPPORTED for f32).  An item covers 16 / (num_heads /
 * num_kv_heads) tokens of a chunk, so longer chunks re-read their prefix once
 * per such group (from L2 when the groups of a partition run together).  A
 * chunk that breaks the rules above is reported as PA_ERR_DEVICE_BAD_INPUT
 * and its rows hold no meaningful values (the other sequences' rows are
 * computed as usual). */
pa_status_t pa_chunks_forward(void *out, const void *query,
                              const void *key_cache, const void *value_cache,
                              const int32_t *block_tables,
                              const int32_t *seq_lens, const int32_t *q_start,
                              int num_seqs, int num_rows, int max_chunk,
                              int num_heads, int num_kv_heads, int head_size,
                              int num_blocks, int block_size,
                              int max_blocks_per_seq, int max_seq_len,
                              float scale, int partition_size, int dtype,
                              void *workspace, size_t workspace_bytes,
                              void *stream, const pa_options_t *opts);

/* Device bytes of the staging buffer pa_forward_host needs: the query and
 * the output ([num_seqs][num_heads][head_size] in the dtype), the block
 * tables and seq_lens, each part 256-byte aligned.  Returns 0 on bad
 * arguments. */
size_t pa_host_staging_bytes(int num_seqs, int num_heads, int head_size,
                             int max_blocks_per_seq, int dtype);

/* pa_forward with the per-step data in HOST memory: query_host,
 * block_tables_host and seq_lens_host are read from the host and out_host is
 * written on the host (same layouts as pa_forward).  The KV caches and the
 * workspace stay on the device.  `staging` is a caller-owned device buffer of
 * at least pa_host_staging_bytes(...) bytes, 256-byte aligned.
 *
 * When all four host buffers are pinned (page-locked, hence mapped into the
 * device's address space; out_host 16-byte aligned), nothing goes through a
 * copy engine: one kernel reads the lengths, block tables and queries from
 * the host buffers into the staging buffer over the host link, and the last
 * kernel of the forward stores the output straight into out_host.  Otherwise
 * the call enqueues one host-to-device cudaMemcpyAsync each of seq_lens, the
 * block tables and the query into the staging buffer, the kernels of
 * pa_forward, and one device-to-host copy of the output (pageable buffers
 * make those copies synchronise the host with the stream).
 *
 * Either way it returns when everything is enqueued on `stream`: synchronise
 * the stream before reading out_host.  The host buffers and the staging
 * buffer must stay untouched until the stream reaches the end of the call.
 * Errors: as pa_forward, plus PA_ERR_INVALID_ARG for a null host pointer or
 * a staging buffer that is null, misaligned or smaller than
 * pa_host_staging_bytes(...); argument errors come back before anything is
 * enqueued. */
pa_status_t pa_forward_host(void *out_host, const void *query_host,
                            const void *key_cache, const void *value_cache,
                            const int32_t *block_tables_host,
                            const int32_t *seq_lens_host, int num_seqs,
                            int num_heads, int num_kv_heads, int head_size,
                            int num_blocks, int block_size,
                            int max_blocks_per_seq, int max_seq_len,
                            float scale, int partition_size, int dtype,
                            void *staging, size_t staging_bytes,
                            void *workspace, size_t workspace_bytes,
                            void *stream, const pa_options_t *opts);

/* V2 for callers that cannot allocate device memory, for example a plug-in
 * whose host framework owns all device memory and forbids cudaMalloc while
 * it serves a request, or a serving loop that must not pay cudaMalloc's
 * implicit synchronisation.  The paged_attention_v2 pages have no
 * counterpart: this entry point exists only for such callers.
 *
 * Same arguments as pa_v2_forward, minus the workspace.  V2's scratch comes
 * from a fixed 32 MiB array in device memory owned by the library.  Every
 * GPU that loads the library holds the array until the process exits.
 * Requests whose pa_workspace_bytes(...) exceeds 32 MiB return
 * PA_ERR_WORKSPACE_TOO_SMALL.  The call allocates nothing and calls no
 * allocating routine.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls on a device share the one array and each overwrites what the last
 * left there, so calls whose kernels overlap on the GPU race: serialise
 * them.  Device-detected data errors land in the shared array's status word,
 * which each call clears; callers that need pa_read_device_status use
 * pa_v2_forward with their own workspace. */
pa_status_t pa_v2_forward_noalloc(void *out, const void *query,
                                  const void *key_cache,
                                  const void *value_cache,
                                  const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs,
                                  int num_heads, int num_kv_heads,
                                  int head_size, int num_blocks,
                                  int block_size, int max_blocks_per_seq,
                                  int max_seq_len, float scale,
                                  int partition_size, int dtype, void *stream);

/* Host heuristic: 1 if V2 should serve this batch on a GPU with sm_count
 * SMs, 0 for V1.  The pages switch on sequence length alone: the commit note
 * for computility-run.yaml (project_6, commit a2a5dd8) lists the decode path
 * as V1 up to 8192 tokens and V2 above, and GROUND_TRUTH_STATUS_v2.md
 * (project_6_baseline5, section "路径 3") says the partitioning should follow
 * the SM count.  Here: V1 when every sequence fits in one partition;
 * otherwise V2 unless the batch alone fills the GPU several times over with
 * short sequences (the length bound and the fill factor are set from
 * measurements on GB300). */
int pa_choose_v2(int num_seqs, int num_kv_heads, int max_seq_len,
                 int partition_size, int sm_count);

/* The same heuristic for query chunks (pa_chunks_forward with the automatic
 * variant): 1 for V2, 0 for V1, for chunks of at most max_chunk tokens.  V1
 * when every sequence fits in one partition; with at most 8 (token, head)
 * rows per KV head, pa_choose_v2's answer; otherwise V1 when the batch has
 * at least 8 work items per SM (4 on the tcgen05 kernel), counting an item
 * per (sequence, KV head) and row group as the chunk kernels cut them (128
 * rows on the tcgen05 kernel: more than 16 rows per KV head at head_size
 * 128; 64 on the row-owning kernel: more than 32 rows per KV head at
 * head_size 64, a group dividing 64; else 16), V2 below (measured on GB300).
 * Pure host arithmetic on its arguments. */
int pa_choose_v2_chunks(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                        int max_chunk, int max_seq_len, int partition_size, int sm_count);

/* Synchronise `stream`, return the workspace's status word as a pa_status_t
 * (PA_OK if no kernel reported a problem) and reset it to 0.  The pages have
 * no counterpart: this is how the library reports data errors its kernels
 * find (a block-table entry outside [0, num_blocks), a length outside
 * [0, max_seq_len]) or a bounded device wait that ran out, since kernels
 * never trap.  Not for use inside a stream capture (it synchronises). */
pa_status_t pa_read_device_status(void *workspace, void *stream);

/* Static English text for a status code. */
const char *pa_status_string(int status);

/* Text of the last CUDA error seen by this thread inside the library. */
const char *pa_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
