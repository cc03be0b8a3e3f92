// libpa C ABI: argument checks, the V1/V2 choice, the launch plan (pipeline
// depth, grids, TMA descriptors) and the kernel launches.
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

using namespace pa;

thread_local char g_last_error[512] = "";

pa_status_t fail_cuda(const char *what, const char *detail) {
  snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, detail);
  return PA_ERR_CUDA;
}
pa_status_t fail_cuda(const char *what, cudaError_t e) {
  return fail_cuda(what, cudaGetErrorString(e));
}

int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int elt_size(int dtype) { return dtype == PA_DTYPE_F32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// Per-device facts, queried once.
struct DeviceFacts {
  bool ready = false;
  int sm_count = 0;
  int max_smem_optin = 0;
  int smem_per_sm = 0, reserved_smem = 0, regs_per_sm = 0, threads_per_sm = 0;
};
constexpr int kMaxDevices = 64;
DeviceFacts g_devices[kMaxDevices];
std::mutex g_mutex;

pa_status_t device_facts(DeviceFacts **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda("cudaGetDevice", "device ordinal too large");
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceFacts &f = g_devices[dev];
  if (!f.ready) {
    e = cudaDeviceGetAttribute(&f.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(SM count)", e);
    e = cudaDeviceGetAttribute(&f.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(smem)", e);
    e = cudaDeviceGetAttribute(&f.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(smem per SM)", e);
    e = cudaDeviceGetAttribute(&f.reserved_smem, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(reserved smem)", e);
    e = cudaDeviceGetAttribute(&f.regs_per_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(registers)", e);
    e = cudaDeviceGetAttribute(&f.threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
    if (e != cudaSuccess) return fail_cuda("cudaDeviceGetAttribute(threads)", e);
    f.ready = true;
  }
  *out = &f;
  return PA_OK;
}

// CTAs of a kernel one SM holds by its registers (whole warps, 256-register
// allocation units), shared memory (with the per-block reservation) and
// threads.
pa_status_t resource_ctas_per_sm(const void *fn, int threads, size_t smem, const DeviceFacts *dev,
                                 int *out) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) return fail_cuda("cudaFuncGetAttributes", e);
  const long long warps = (threads + 31) / 32;
  const long long regs_per_warp = ((long long)fa.numRegs * 32 + 255) / 256 * 256;
  long long n = regs_per_warp > 0 ? dev->regs_per_sm / (warps * regs_per_warp) : 0;
  const long long per_block = (long long)smem + fa.sharedSizeBytes + dev->reserved_smem;
  if (per_block > 0 && dev->smem_per_sm / per_block < n) n = dev->smem_per_sm / per_block;
  if (dev->threads_per_sm / threads < n) n = dev->threads_per_sm / threads;
  *out = (int)(n > 0 ? n : 0);
  return PA_OK;
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
struct SmemSetting {
  const void *fn;
  int dev;
  int bytes;
};
SmemSetting g_smem_settings[256];
int g_num_smem_settings = 0;

pa_status_t ensure_smem(const void *fn, size_t bytes) {
  if (bytes <= 48 * 1024) return PA_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int i = 0; i < g_num_smem_settings; ++i)
    if (g_smem_settings[i].fn == fn && g_smem_settings[i].dev == dev &&
        g_smem_settings[i].bytes >= (int)bytes)
      return PA_OK;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return fail_cuda("cudaFuncSetAttribute(max dynamic smem)", e);
  for (int i = 0; i < g_num_smem_settings; ++i)
    if (g_smem_settings[i].fn == fn && g_smem_settings[i].dev == dev) {
      g_smem_settings[i].bytes = (int)bytes;
      return PA_OK;
    }
  if (g_num_smem_settings < 256) g_smem_settings[g_num_smem_settings++] = {fn, dev, (int)bytes};
  return PA_OK;
}

// Resident CTAs per SM of a kernel at a given block size and dynamic smem,
// remembered per (kernel, smem, device).
struct OccupancyEntry {
  const void *fn;
  int dev, threads;
  size_t smem;
  int per_sm;
};
OccupancyEntry g_occupancy[256];
int g_num_occupancy = 0;

pa_status_t occupancy(const void *fn, int threads, size_t smem, int *per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda("cudaGetDevice", e);
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int i = 0; i < g_num_occupancy; ++i) {
    const OccupancyEntry &o = g_occupancy[i];
    if (o.fn == fn && o.dev == dev && o.threads == threads && o.smem == smem) {
      *per_sm = o.per_sm;
      return PA_OK;
    }
  }
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem);
  if (e != cudaSuccess) return fail_cuda("cudaOccupancyMaxActiveBlocksPerMultiprocessor", e);
  if (g_num_occupancy < 256) g_occupancy[g_num_occupancy++] = {fn, dev, threads, smem, n};
  *per_sm = n;
  return PA_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

pa_status_t get_encoder(PFN_cuTensorMapEncodeTiled_v12000 *fn) {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return fail_cuda("cudaGetDriverEntryPointByVersion", e);
    if (q != cudaDriverEntryPointSuccess || !p)
      return fail_cuda("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled not found");
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  *fn = g_encode;
  return PA_OK;
}

// A 3-D view of a cache: (128-byte panel slice, token row, panel), the rows
// being the num_blocks * num_kv_heads * block_size token rows of head_size
// elements; the box is a whole unit of unit_rows rows (every panel), landing
// in shared memory as [panel][row][128 bytes] with the 128-byte swizzle.
pa_status_t encode_cache_map(CUtensorMap *map, const void *base, int dtype, int head_size,
                             long long rows, int unit_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  pa_status_t st = get_encoder(&enc);
  if (st != PA_OK) return st;
  const int elt = elt_size(dtype);
  CUtensorMapDataType dt = dtype == PA_DTYPE_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                           : dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int panel = kPanelBytes / elt;  // elements of a 128-byte panel
  const int panels = head_size / panel;
  cuuint64_t gdim[3] = {(cuuint64_t)panel, (cuuint64_t)rows, (cuuint64_t)panels};
  cuuint64_t gstride[2] = {(cuuint64_t)head_size * elt, (cuuint64_t)kPanelBytes};
  cuuint32_t box[3] = {(cuuint32_t)panel, (cuuint32_t)unit_rows, (cuuint32_t)panels};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void *>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof msg, "CUresult %d", (int)r);
    return fail_cuda("cuTensorMapEncodeTiled", msg);
  }
  return PA_OK;
}

// ---------------------------------------------------------------------------
struct Call {
  void *out;
  const void *query, *key_cache, *value_cache;
  const int32_t *block_tables, *seq_lens;
  int num_seqs, num_heads, num_kv_heads, head_size, num_blocks, block_size;
  int max_blocks_per_seq, max_seq_len;
  float scale;
  int partition_size, dtype;
  void *workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  // query chunks (pa_chunks_forward); q_start == nullptr: one query a sequence
  const int32_t *q_start;
  int num_rows;
  int max_chunk;
  // V2 split into its phases (pa_v2_partials / pa_v2_combine): the phases to
  // run (bit 0: Phase 1, bit 1: Phase 2) and Phase 1's range of partitions
  int phases = 3;
  int part_begin = 0, part_end = INT_MAX;
};

// Rows of query (and output) and of the V2 workspace: sequences, or the query
// chunks' rows.
int query_rows(const Call &c) { return c.q_start ? c.num_rows : c.num_seqs; }

// Chunk mode: tokens of one item (its (token, head) rows fill the 16 columns
// of the two-n-tile tensor path).
int chunk_tokens_of(const Call &c) { return 16 / (c.num_heads / c.num_kv_heads); }

int max_parts_of(int max_seq_len, int partition_size) {
  return (max_seq_len + partition_size - 1) / partition_size;
}

constexpr int kMaxReduceParts = 1 << 20;  // bound on partitions per sequence

// Checks that need no device.  need_v2: the workspace must hold the partials.
pa_status_t check_args(const Call &c, bool need_v2) {
  if (c.dtype != PA_DTYPE_F32 && c.dtype != PA_DTYPE_BF16 && c.dtype != PA_DTYPE_F16)
    return PA_ERR_INVALID_ARG;
  if (c.num_seqs < 0 || c.num_heads < 1 || c.num_kv_heads < 1 || c.num_blocks < 1 ||
      c.max_blocks_per_seq < 1 || c.max_seq_len < 0 || c.block_size < 1 || c.partition_size < 1)
    return PA_ERR_INVALID_ARG;
  if (c.num_heads % c.num_kv_heads) return PA_ERR_INVALID_ARG;
  if (!isfinite(c.scale)) return PA_ERR_INVALID_ARG;
  if ((long long)c.max_seq_len > (long long)c.max_blocks_per_seq * c.block_size)
    return PA_ERR_INVALID_ARG;
  if (c.head_size != 64 && c.head_size != 128 && c.head_size != 256) return PA_ERR_UNSUPPORTED;
  if (c.block_size != 8 && c.block_size != 16 && c.block_size != 32 && c.block_size != 64)
    return PA_ERR_UNSUPPORTED;
  if (c.num_heads / c.num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  if (c.partition_size % 64 || c.partition_size % c.block_size || c.partition_size > 8192)
    return PA_ERR_UNSUPPORTED;
  if ((long long)c.num_blocks * c.num_kv_heads * c.block_size >= (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  if (c.q_start) {
    if (c.num_rows < 0 || c.max_chunk < 1 || c.max_chunk > c.max_seq_len) return PA_ERR_INVALID_ARG;
    if (c.dtype == PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;  // tensor path only
    if (!aligned(c.q_start, 4)) return PA_ERR_INVALID_ARG;
  }
  const long long groups =
      c.q_start ? (c.max_chunk + chunk_tokens_of(c) - 1) / chunk_tokens_of(c) : 1;
  if ((long long)c.num_seqs * c.num_kv_heads * max_parts_of(c.max_seq_len, c.partition_size) *
          groups >= (1ll << 31))
    return PA_ERR_UNSUPPORTED;
  if (need_v2 && max_parts_of(c.max_seq_len, c.partition_size) > kMaxReduceParts)
    return PA_ERR_UNSUPPORTED;
  if (c.part_begin < 0 || c.part_end < c.part_begin) return PA_ERR_INVALID_ARG;
  if ((c.part_begin != 0 || c.part_end != INT_MAX) && (!need_v2 || c.q_start))
    return PA_ERR_INVALID_ARG;  // a range of partitions is a V2 decode notion
  if (!c.out || !c.query || !c.key_cache || !c.value_cache || !c.block_tables || !c.seq_lens ||
      !c.workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned(c.out, 16) || !aligned(c.query, 16) || !aligned(c.key_cache, 16) ||
      !aligned(c.value_cache, 16) || !aligned(c.block_tables, 4) || !aligned(c.seq_lens, 4) ||
      !aligned(c.workspace, 256))
    return PA_ERR_INVALID_ARG;
  const size_t need = need_v2 ? pa_workspace_bytes(query_rows(c), c.num_heads, c.head_size,
                                                   c.max_seq_len, c.partition_size)
                              : (size_t)kStatusBytes;
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (c.workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  return PA_OK;
}

// Checks of a Phase-2-only call (pa_v2_combine): no query, caches or tables.
pa_status_t check_combine_args(const Call &c) {
  if (c.dtype != PA_DTYPE_F32 && c.dtype != PA_DTYPE_BF16 && c.dtype != PA_DTYPE_F16)
    return PA_ERR_INVALID_ARG;
  if (c.num_seqs < 0 || c.num_heads < 1 || c.max_seq_len < 0 || c.partition_size < 1)
    return PA_ERR_INVALID_ARG;
  if (c.head_size != 64 && c.head_size != 128 && c.head_size != 256) return PA_ERR_UNSUPPORTED;
  if (c.partition_size % 64 || c.partition_size > 8192) return PA_ERR_UNSUPPORTED;
  if (max_parts_of(c.max_seq_len, c.partition_size) > kMaxReduceParts) return PA_ERR_UNSUPPORTED;
  if (!c.out || !c.seq_lens || !c.workspace) return PA_ERR_INVALID_ARG;
  if (!aligned(c.out, 16) || !aligned(c.seq_lens, 4) || !aligned(c.workspace, 256))
    return PA_ERR_INVALID_ARG;
  const size_t need = pa_workspace_bytes(c.num_seqs, c.num_heads, c.head_size, c.max_seq_len,
                                         c.partition_size);
  if (need == 0) return PA_ERR_INVALID_ARG;
  if (c.workspace_bytes < need) return PA_ERR_WORKSPACE_TOO_SMALL;
  return PA_OK;
}

AttnKernelInfo pick_kernel(int math, int dtype, int head_size, int group) {
  if (math == kMathTensor) {
    if (dtype == PA_DTYPE_BF16) return attn_kernel_tensor_bf16(head_size, group);
    if (dtype == PA_DTYPE_F16) return attn_kernel_tensor_f16(head_size, group);
  } else {
    if (dtype == PA_DTYPE_F32) return attn_kernel_simt_f32(head_size, group);
    if (dtype == PA_DTYPE_BF16) return attn_kernel_simt_bf16(head_size, group);
    if (dtype == PA_DTYPE_F16) return attn_kernel_simt_f16(head_size, group);
  }
  return AttnKernelInfo{nullptr, 0, 0, 0};
}

// The cache as TMA sees it for the tcgen05 chunk kernel: (128-byte panel
// slice, row within an 8-row group, panel, 8-row group), so that one box of
// (64 elements, 8 rows, every panel, unit_rows / 8 groups) brings all panels
// of a page's rows and lands as [group][panel][8 rows][128 bytes]: each
// 8-row group of a panel is one 1024-byte swizzle atom, and the matrix
// descriptors step 2048 bytes (D 128) from group to group.
pa_status_t encode_cache_map_umma(CUtensorMap *map, const void *base, int dtype, int head_size,
                                  long long rows, int unit_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  pa_status_t st = get_encoder(&enc);
  if (st != PA_OK) return st;
  const int elt = elt_size(dtype);
  const int panel = kPanelBytes / elt;
  const int panels = head_size / panel;
  CUtensorMapDataType dt = dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t gdim[4] = {(cuuint64_t)panel, 8, (cuuint64_t)panels, (cuuint64_t)(rows / 8)};
  cuuint64_t gstride[3] = {(cuuint64_t)head_size * elt, (cuuint64_t)kPanelBytes,
                           (cuuint64_t)head_size * elt * 8};
  cuuint32_t box[4] = {(cuuint32_t)panel, 8, (cuuint32_t)panels, (cuuint32_t)(unit_rows / 8)};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = enc(map, dt, 4, const_cast<void *>(base), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof msg, "CUresult %d", (int)r);
    return fail_cuda("cuTensorMapEncodeTiled", msg);
  }
  return PA_OK;
}

// The queries as TMA sees them for the tcgen05 kernel of small items:
// (element of D, head, query row), so that a box of (64, group, tokens) at
// (64 p, kv_head * group, row) brings panel p of an item's tokens x group
// rows, landing as [token][head][128 bytes] (row n = token * group + head) in
// the 128-byte swizzle.
pa_status_t encode_query_map(CUtensorMap *map, const void *query, int dtype, int head_size,
                             int num_heads, long long rows, int group, int tokens) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  pa_status_t st = get_encoder(&enc);
  if (st != PA_OK) return st;
  const int elt = elt_size(dtype);
  CUtensorMapDataType dt = dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t gdim[3] = {(cuuint64_t)head_size, (cuuint64_t)num_heads,
                        (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t gstride[2] = {(cuuint64_t)head_size * elt, (cuuint64_t)num_heads * head_size * elt};
  cuuint32_t box[3] = {(cuuint32_t)(kPanelBytes / elt), (cuuint32_t)group, (cuuint32_t)tokens};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void *>(query), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[64];
    snprintf(msg, sizeof msg, "CUresult %d", (int)r);
    return fail_cuda("cuTensorMapEncodeTiled", msg);
  }
  return PA_OK;
}

// Phase 2 of one call: kernel, grid and parameters.  It is planned before
// Phase 1 is enqueued, so that nothing can fail between the two launches.
struct Phase2Plan {
  ReduceParams r;
  const void *fn = nullptr;
  long long ctas = 0;
  int threads = 256;
  size_t smem = 0;  // dynamic shared memory
};

pa_status_t plan_phase2(const Call &c, const AttnParams &p, const DeviceFacts *dev,
                        long long prows, Phase2Plan *out) {
  ReduceParams &r = out->r;
  memset(&r, 0, sizeof r);
  r.out = c.out;
  r.max_logits = p.max_logits;
  r.exp_sums = p.exp_sums;
  r.tmp_out = p.tmp_out;
  r.seq_lens = c.seq_lens;
  r.status = p.status;
  r.num_seqs = query_rows(c);  // Phase 2 rows: (query row, head)
  r.num_heads = c.num_heads;
  r.head_size = c.head_size;
  r.max_parts = p.max_parts;
  r.partition_size = c.partition_size;
  r.max_seq_len = c.max_seq_len;
  r.fuse_limit = p.fuse_limit;
  r.row_limit = p.row_limit;
  // Rows whose partials fit in 8 KB (and 32 partitions, one a lane): a warp
  // takes each row's partials in one bulk copy, the next row's in flight
  // while it reduces the current one, so that the whole batch crosses the
  // memory system in about one round trip (measured on GB300, the
  // 256-sequence decode batch: see the kernel's notes).
  if (p.max_parts <= 32 && (size_t)p.max_parts * c.head_size * 4 <= 8192) {
    const void *fn = reduce_rows_kernel(c.dtype);
    if (!fn) return PA_ERR_UNSUPPORTED;
    const size_t smem = reduce_rows_smem_bytes(p.max_parts, c.head_size);
    pa_status_t st = ensure_smem(fn, smem);
    if (st != PA_OK) return st;
    int occ_r = 0;
    st = occupancy(fn, kReduceRowsThreads, smem, &occ_r);
    if (st != PA_OK) return st;
    if (occ_r < 1) return PA_ERR_UNSUPPORTED;
    long long ctas = (prows + kReduceRowsThreads / 32 - 1) / (kReduceRowsThreads / 32);
    if (ctas > (long long)occ_r * dev->sm_count) ctas = (long long)occ_r * dev->sm_count;
    out->fn = fn;
    out->ctas = ctas;
    out->threads = kReduceRowsThreads;
    out->smem = smem;
    return PA_OK;
  }
  // Team size W (warps per task) and column split: the pair that minimises
  // the chain of the longest task (1 + its rounds of loads, a round being one
  // batch of NB partitions per thread) plus 2 for every further wave of
  // tasks (the typical task, with sequences of mixed lengths, takes one
  // round).  Only max_seq_len is known here, so the longest task is sized
  // from it.
  int occ = 0;
  {
    const void *probe = reduce_kernel(c.dtype, 1);
    pa_status_t so = occupancy(probe, 256, 0, &occ);
    if (so != PA_OK) return so;
    if (occ < 1) return PA_ERR_UNSUPPORTED;
  }
  const long long resident_warps = (long long)occ * dev->sm_count * 8;
  int best_w = 1, best_ds = 1, best_vpt = 1;
  long long best_cost = -1;
  for (int w = 1; w <= 8; w *= 2) {
    for (int ds = 1; c.head_size / 4 / ds >= 4; ds *= 2) {
      const int f4 = c.head_size / 4 / ds;  // float4 columns per task
      const int vpt = f4 > 32 ? f4 / 32 : 1;
      if (vpt > 2) continue;
      const int lanes = f4 / vpt;
      const long long slots = (long long)w * (32 / lanes);
      const long long nb = vpt == 1 ? 4 : 2;  // the kernel's batch (NB)
      const long long rounds = (p.max_parts + slots * nb - 1) / (slots * nb);
      const long long conc = resident_warps / w;
      const long long waves = (prows * ds + conc - 1) / conc;
      const long long cost = (1 + rounds) + 2 * (waves - 1);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best_w = w;
        best_ds = ds;
        best_vpt = vpt;
      }
    }
  }
  r.cols_per_cta = c.head_size / best_ds;
  r.warps_per_head = best_w;
  const void *rfn = reduce_kernel(c.dtype, best_vpt);
  if (!rfn) return PA_ERR_UNSUPPORTED;
  out->fn = rfn;
  int occ_k = 0;
  {
    pa_status_t so = occupancy(rfn, 256, 0, &occ_k);
    if (so != PA_OK) return so;
    if (occ_k < 1) return PA_ERR_UNSUPPORTED;
  }
  // persistent: never more CTAs than are resident at once
  const long long teams_per_cta = 8 / best_w;
  long long ctas = (prows * best_ds + teams_per_cta - 1) / teams_per_cta;
  if (ctas > (long long)occ_k * dev->sm_count) ctas = (long long)occ_k * dev->sm_count;
  out->ctas = ctas;
  return PA_OK;
}

// Launch a planned Phase 2 kernel, chained to the previous kernel of the
// stream by programmatic dependent launch (its own wait holds it until that
// kernel has completed).
pa_status_t launch_phase2(const Phase2Plan &plan, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)plan.ctas, 1, 1);
  cfg.blockDim = dim3((unsigned)plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ReduceParams r = plan.r;
  void *rargs[1] = {&r};
  cudaError_t e = cudaLaunchKernelExC(&cfg, plan.fn, rargs);
  if (e != cudaSuccess) return fail_cuda("launch reduce kernel", e);
  return PA_OK;
}

pa_status_t launch(const Call &c, bool v2, const pa_options_t &opt) {
  DeviceFacts *dev = nullptr;
  pa_status_t st = device_facts(&dev);
  if (st != PA_OK) return st;

  const int group = c.num_heads / c.num_kv_heads;
  int math = opt.math;
  if (math == PA_MATH_AUTO) math = c.dtype == PA_DTYPE_F32 ? kMathSimt : kMathTensor;
  if (math != kMathSimt && math != kMathTensor) return PA_ERR_INVALID_ARG;
  if (math == kMathTensor && c.dtype == PA_DTYPE_F32) return PA_ERR_UNSUPPORTED;
  const bool chunk = c.q_start != nullptr;
  if (chunk && math != kMathTensor) return PA_ERR_UNSUPPORTED;
  const bool tc = math == kMathTensor && !(opt.debug_flags & PA_DEBUG_NO_TCGEN05);
  // Items of at most 16 rows on tcgen05 with the keys on the MMA's M, when
  // asked for (PA_DEBUG_TCGEN05_KEYS), unless the combine is to be fused
  // into Phase 1, which only the mma.sync kernels do.  Not the default:
  // measured on GB300 (16 heads a group on the 256-sequence cache) it takes
  // 0.123-0.146 ms (V2) / 0.116-0.126 ms (V1) a step, on two boxes, against
  // the two-n-tile mma.sync kernel's 0.098 ms: one CTA an SM does not cover
  // its item boundaries.
  const long long item_rows = chunk ? (long long)c.max_chunk * group : group;
  const bool keys = tc && (opt.debug_flags & PA_DEBUG_TCGEN05_KEYS) &&
                    umma_keys_ok(c.head_size, item_rows) && aligned(c.query, 16) &&
                    !(v2 && !chunk && opt.fuse_partitions > 0);
  const bool umma = chunk && tc && umma_chunk_ok(c.head_size, group, item_rows);
  // tcgen05 chunks of several 128-row groups per KV head, when asked
  // (share_kv): a cluster of 2 or 4 CTAs takes them together, sharing each
  // stage's K/V by multicast.  Off by default: measured on GB300 (the
  // 256-sequence cache, V1) it reads K/V from HBM once instead of 1.66 times
  // but takes 10 % longer at 4 CTAs (64-token chunks) and 2.5 % at 2.
  int cl = 1;
  if (umma && opt.share_kv > 0) {
    const long long rg = ((long long)c.max_chunk * group + 127) / 128;
    cl = rg >= 4 ? 4 : rg >= 2 ? 2 : 1;
  }
  const AttnKernelInfo k =
      keys    ? attn_kernel_umma_keys(c.dtype == PA_DTYPE_BF16 ? 1 : 0)
      : umma  ? attn_kernel_umma_chunk(c.dtype == PA_DTYPE_BF16 ? 1 : 0, cl > 1)
      : chunk ? (c.dtype == PA_DTYPE_BF16
                     ? attn_kernel_chunk_bf16(c.head_size, group, c.max_chunk * group)
                     : attn_kernel_chunk_f16(c.head_size, group, c.max_chunk * group))
              : pick_kernel(math, c.dtype, c.head_size, group);
  if (!k.fn) return PA_ERR_UNSUPPORTED;

  const int elt = elt_size(c.dtype);
  const size_t stage_bytes = (size_t)k.stage_tokens * c.head_size * elt * 2;
  const bool simt = math == kMathSimt;
  const int threads = (k.consumer_warps + 1) * 32;
  // Pipeline depth: the number of stages that keeps the most K/V bytes in
  // flight per SM (resident CTAs x stages x stage bytes); on a tie the
  // shallower ring, whose extra CTAs cover one another's start-up and
  // epilogue (measured on GB300: three CTAs of two 32 KB stages stream faster
  // than two CTAs of three).
  int stages = opt.num_stages > 0 ? opt.num_stages : 0;
  if (stages > 0 && (stages < 2 || stages > 16)) return PA_ERR_INVALID_ARG;
  if (k.umma) stages = kUmmaStagesHost;  // a fixed layout
  if (stages == 0) {
    long long best = 0;
    for (int n = 2; n <= 8; ++n) {
      const size_t b = attn_smem_bytes(c.head_size, elt, k.stage_tokens, k.consumer_warps,
                                       k.max_group, n, simt);
      if (b > (size_t)dev->max_smem_optin) break;
      st = ensure_smem(k.fn, b);
      if (st != PA_OK) return st;
      int fit = 0;
      st = occupancy(k.fn, threads, b, &fit);
      if (st != PA_OK) return st;
      const long long flight = (long long)fit * n * (long long)stage_bytes;
      if (flight > best) {
        best = flight;
        stages = n;
      }
    }
    if (stages <= 0) return PA_ERR_UNSUPPORTED;
  }
  size_t smem = k.umma == 2 ? umma_keys_smem_bytes()
                 : k.umma    ? umma_chunk_smem_bytes()
                             : attn_smem_bytes(c.head_size, elt, k.stage_tokens, k.consumer_warps,
                                        k.max_group, stages, simt);
  if (smem > (size_t)dev->max_smem_optin) return PA_ERR_UNSUPPORTED;

  const int unit_rows = c.block_size < k.stage_tokens ? c.block_size : k.stage_tokens;
  const long long rows = (long long)c.num_blocks * c.num_kv_heads * c.block_size;
  CUtensorMap tmap_k, tmap_v;
  auto encode = k.umma ? encode_cache_map_umma : encode_cache_map;
  st = encode(&tmap_k, c.key_cache, c.dtype, c.head_size, rows, unit_rows);
  if (st != PA_OK) return st;
  st = encode(&tmap_v, c.value_cache, c.dtype, c.head_size, rows, unit_rows);
  if (st != PA_OK) return st;
  // the kernel of small items: an item's tokens (of its query chunk), at
  // most 16 rows with its heads, and never more than there are query rows
  long long item_tokens = 1;
  if (chunk) {
    item_tokens = k.max_group / group;
    if (item_tokens > c.max_chunk) item_tokens = c.max_chunk;
    if (item_tokens > c.num_rows) item_tokens = c.num_rows;
    if (item_tokens < 1) item_tokens = 1;
  }
  CUtensorMap tmap_q;
  memset(&tmap_q, 0, sizeof tmap_q);
  if (k.umma == 2) {
    st = encode_query_map(&tmap_q, c.query, c.dtype, c.head_size, c.num_heads, query_rows(c), group,
                          (int)item_tokens);
    if (st != PA_OK) return st;
  }

  uint8_t *ws = static_cast<uint8_t *>(c.workspace);
  const int max_parts = v2 ? max_parts_of(c.max_seq_len, c.partition_size) : 1;
  size_t off[5] = {0, 0, 0, 0, 0};
  if (v2) {
    if (pa_workspace_layout(query_rows(c), c.num_heads, c.head_size, c.max_seq_len,
                            c.partition_size, off) != PA_OK)
      return PA_ERR_INVALID_ARG;
  }

  AttnParams p;
  memset(&p, 0, sizeof p);
  p.query = c.query;
  p.out = c.out;
  p.block_tables = c.block_tables;
  p.seq_lens = c.seq_lens;
  p.status = reinterpret_cast<int *>(ws);
  p.sched = reinterpret_cast<int *>(ws) + 1;
  if (v2) {
    p.max_logits = reinterpret_cast<float *>(ws + off[1]);
    p.exp_sums = reinterpret_cast<float *>(ws + off[2]);
    p.tmp_out = reinterpret_cast<float *>(ws + off[3]);
  }
  p.num_seqs = c.num_seqs;
  p.num_heads = c.num_heads;
  p.num_kv_heads = c.num_kv_heads;
  p.group = group;
  p.block_size = c.block_size;
  p.log2_block_size = ilog2(c.block_size);
  p.unit_rows = unit_rows;
  p.log2_unit_rows = ilog2(unit_rows);
  p.max_blocks_per_seq = c.max_blocks_per_seq;
  p.max_seq_len = c.max_seq_len;
  p.num_blocks = c.num_blocks;
  p.range_tokens = v2 ? c.partition_size : (c.max_seq_len > 0 ? c.max_seq_len : 1);
  p.max_parts = max_parts > 0 ? max_parts : 1;
  p.write_partials = v2 ? 1 : 0;
  p.part_begin = c.part_begin;
  p.part_end = c.part_end;
  const bool phase1 = (c.phases & 1) != 0;
  const bool phase2 = (c.phases & 2) != 0;
  if (v2) {
    // Off unless asked for: on the workloads measured so far the separate
    // Phase 2 kernel costs less than the per-item handshake of the fused one.
    const int fuse = opt.fuse_partitions > 0 ? opt.fuse_partitions : 0;
    p.fuse_limit = fuse > kFuseLimitMax ? kFuseLimitMax : fuse;
    if (!phase1 || !phase2) p.fuse_limit = 0;  // the phases run apart
    p.group_count = reinterpret_cast<int *>(ws + off[4]);
    // chunk mode: no fused combine; the counters region holds the rows' limits
    if (chunk) {
      p.fuse_limit = 0;
      p.row_limit = reinterpret_cast<int *>(ws + off[4]);
    }
  }
  if (chunk) {
    p.q_start = c.q_start;
    p.num_rows = c.num_rows;
    // tokens of an item: its rows / heads per token
    p.chunk_tokens = k.umma == 2 ? (int)item_tokens : k.max_group / group;
  }
  p.num_stages = stages;
  p.debug_flags = opt.debug_flags;
  p.scale_log2 = (float)((double)c.scale * 1.4426950408889634);
  p.wait_limit_ns = opt.wait_limit_ns ? opt.wait_limit_ns : kDefaultWaitLimitNs;

  // Phase 2 runs unless there are no rows, or the combine is fused and covers
  // every sequence (Phase 1 then also writes the empty ones' zeros).  When it
  // runs, it returns Phase 1's work counter to zero after its wait, so that
  // Phase 1's CTAs can retire without a last-CTA-out handshake.
  const long long prows = (long long)query_rows(c) * c.num_heads;
  const bool run_p2 =
      v2 && phase2 && prows > 0 &&
      !(p.fuse_limit > 0 && max_parts_of(c.max_seq_len, c.partition_size) <= p.fuse_limit);
  Phase2Plan plan;
  if (run_p2) {
    st = plan_phase2(c, p, dev, prows, &plan);
    if (st != PA_OK) return st;
    if (phase1) {
      plan.r.sched = p.sched;
      p.sched_reset_later = 1;
    }
  }

  st = ensure_smem(k.fn, smem);
  if (st != PA_OK) return st;

  // Persistent grid: as many CTAs as fit on the GPU (or the requested number
  // per SM), never more than there can be work items.
  int per_sm = 0;
  st = occupancy(k.fn, threads, smem, &per_sm);
  if (st != PA_OK) return st;
  if (per_sm < 1) return PA_ERR_UNSUPPORTED;
  if (opt.ctas_per_sm > 0 && opt.ctas_per_sm < per_sm) per_sm = opt.ctas_per_sm;
  if (k.umma) {
    // The occupancy query answers 1 for these kernels whatever its shared
    // memory (measured on GB300: at 20 KB too), while two CTAs fit its
    // registers, shared memory and tensor memory and do run side by side
    // (1.5x the throughput of one).  So its CTAs per SM come from those
    // resources, never more than the 512 tensor-memory columns hold.  A CTA
    // the SM cannot place would only start late: CTAs never wait on others.
    int est = 0;
    st = resource_ctas_per_sm(k.fn, threads, smem, dev, &est);
    if (st != PA_OK) return st;
    if (est > per_sm) per_sm = est;
    if (opt.ctas_per_sm > 0 && opt.ctas_per_sm < per_sm) per_sm = opt.ctas_per_sm;
    const int tmem_cols = k.umma == 2 ? kUmmaKeysTmemColsHost : kUmmaTmemColsHost;
    if (per_sm * tmem_cols > 512) per_sm = 512 / tmem_cols;
  }
  const long long range_parts =
      v2 ? (long long)(c.part_end < p.max_parts ? c.part_end : p.max_parts) - c.part_begin
         : p.max_parts;
  const long long groups = chunk ? (c.max_chunk + p.chunk_tokens - 1) / p.chunk_tokens : 1;
  p.cluster = cl;
  const long long max_items = (long long)c.num_seqs * c.num_kv_heads *
                              (range_parts > 0 ? range_parts : 0) * ((groups + cl - 1) / cl) * cl;
  long long grid = (long long)per_sm * dev->sm_count;
  if (grid > max_items) grid = max_items;
  grid = grid / cl * cl;  // whole clusters
  if (phase1 && grid > 0) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = c.stream;
    // Programmatic dependent launch: the kernel's launch and shared-memory
    // set-up overlap the tail of the previous kernel in the stream; the
    // kernel waits for that kernel before its first global access.
    cudaLaunchAttribute pattr[2];
    pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pattr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pattr;
    cfg.numAttrs = 1;
    if (cl > 1) {
      pattr[1].id = cudaLaunchAttributeClusterDimension;
      pattr[1].val.clusterDim.x = (unsigned)cl;
      pattr[1].val.clusterDim.y = 1;
      pattr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
    }
    void *args[4] = {&p, &tmap_k, &tmap_v, &tmap_q};  // the query map: small-item kernel only
    cudaError_t e = cudaLaunchKernelExC(&cfg, k.fn, args);
    if (e != cudaSuccess) return fail_cuda("launch attention kernel", e);
  }
  if (!run_p2) return PA_OK;

  if (opt.phase1_event && phase1) {
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(opt.phase1_event), c.stream);
    if (e != cudaSuccess) {
      cudaMemsetAsync(p.sched, 0, 2 * sizeof(int), c.stream);  // Phase 2 will not reset it
      return fail_cuda("cudaEventRecord(phase1_event)", e);
    }
  }
  st = launch_phase2(plan, c.stream);
  if (st != PA_OK && phase1) cudaMemsetAsync(p.sched, 0, 2 * sizeof(int), c.stream);  // see above
  return st;
}

// Phase 2 alone (pa_v2_combine): the partials are already in the workspace,
// written by Phase 1 here or gathered from other GPUs.
pa_status_t launch_combine(const Call &c) {
  DeviceFacts *dev = nullptr;
  pa_status_t st = device_facts(&dev);
  if (st != PA_OK) return st;
  const long long prows = (long long)c.num_seqs * c.num_heads;
  if (prows == 0) return PA_OK;
  size_t off[5];
  if (pa_workspace_layout(c.num_seqs, c.num_heads, c.head_size, c.max_seq_len, c.partition_size,
                          off) != PA_OK)
    return PA_ERR_INVALID_ARG;
  uint8_t *ws = static_cast<uint8_t *>(c.workspace);
  AttnParams p;
  memset(&p, 0, sizeof p);
  p.status = reinterpret_cast<int *>(ws);
  p.max_logits = reinterpret_cast<float *>(ws + off[1]);
  p.exp_sums = reinterpret_cast<float *>(ws + off[2]);
  p.tmp_out = reinterpret_cast<float *>(ws + off[3]);
  const int mp = max_parts_of(c.max_seq_len, c.partition_size);
  p.max_parts = mp > 0 ? mp : 1;
  Phase2Plan plan;
  st = plan_phase2(c, p, dev, prows, &plan);
  if (st != PA_OK) return st;
  return launch_phase2(plan, c.stream);
}

Call make_call(void *out, const void *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_heads,
               int num_kv_heads, int head_size, int num_blocks, int block_size,
               int max_blocks_per_seq, int max_seq_len, float scale, int partition_size,
               int dtype, void *workspace, size_t workspace_bytes, void *stream) {
  return Call{out,          query,         key_cache,          value_cache, block_tables,
              seq_lens,     num_seqs,      num_heads,          num_kv_heads, head_size,
              num_blocks,   block_size,    max_blocks_per_seq, max_seq_len, scale,
              partition_size, dtype,       workspace,          workspace_bytes,
              static_cast<cudaStream_t>(stream)};
}

// The variant a call runs (V1 or V2) and the full argument check for it;
// nothing is enqueued.
pa_status_t resolve(const Call &c, int variant, bool *v2) {
  if (variant == PA_VARIANT_V1) {
    *v2 = false;
  } else if (variant == PA_VARIANT_V2) {
    *v2 = true;
  } else if (variant == PA_VARIANT_AUTO) {
    pa_status_t st0 = check_args(c, false);
    if (st0 != PA_OK) return st0;
    *v2 = false;
    if (c.num_seqs == 0) return PA_OK;
    DeviceFacts *dev = nullptr;
    pa_status_t st = device_facts(&dev);
    if (st != PA_OK) return st;
    *v2 = (c.q_start ? pa_choose_v2_chunks(c.num_seqs, c.num_heads, c.num_kv_heads, c.head_size,
                                           c.max_chunk, c.max_seq_len, c.partition_size,
                                           dev->sm_count)
                     : pa_choose_v2(c.num_seqs, c.num_kv_heads, c.max_seq_len,
                                    c.partition_size, dev->sm_count)) != 0;
  } else {
    return PA_ERR_INVALID_ARG;
  }
  return check_args(c, *v2);
}

pa_status_t run(const Call &c, int variant, const pa_options_t &opt) {
  bool v2 = false;
  pa_status_t st = resolve(c, variant, &v2);
  if (st != PA_OK) return st;
  if (c.num_seqs == 0) return PA_OK;
  return launch(c, v2, opt);
}

// The device-side address of host memory, if it is pinned (page-locked and
// mapped into the current device's address space); false for pageable
// memory, which only the copy engines may read.
bool device_view(const void *host, const void **dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of an unknown pointer
    return false;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return false;
  *dev = a.devicePointer;
  return true;
}
bool device_view(void *host, void **dev) {
  const void *d = nullptr;
  if (!device_view(static_cast<const void *>(host), &d)) return false;
  *dev = const_cast<void *>(d);
  return true;
}

// Enqueue the kernel that copies pa_forward_host's inputs (three segments:
// lengths, block tables, queries) from mapped host memory into staging.
pa_status_t stage_in(const void *s0, void *d0, size_t b0, const void *s1, void *d1, size_t b1,
                     const void *s2, void *d2, size_t b2, cudaStream_t stream) {
  DeviceFacts *dev = nullptr;
  pa_status_t st = device_facts(&dev);
  if (st != PA_OK) return st;
  StageInParams p;
  memset(&p, 0, sizeof p);
  const void *src[3] = {s0, s1, s2};
  void *dst[3] = {d0, d1, d2};
  const size_t bytes[3] = {b0, b1, b2};
  long long units16 = 0;
  for (int i = 0; i < kStageInSegments; ++i) {
    const bool wide = aligned(src[i], 16) && aligned(dst[i], 16) && bytes[i] % 16 == 0;
    p.src[i] = src[i];
    p.dst[i] = dst[i];
    p.width[i] = wide ? 16 : 4;  // every segment is a whole number of 4-byte words
    p.units[i] = (long long)(bytes[i] / p.width[i]);
    units16 += (long long)((bytes[i] + 15) / 16);
  }
  // about four 16-byte units per thread, at most four CTAs per SM
  long long ctas = (units16 + 4 * 256 - 1) / (4 * 256);
  if (ctas > 4LL * dev->sm_count) ctas = 4LL * dev->sm_count;
  if (ctas < 1) ctas = 1;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)ctas, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[1] = {&p};
  cudaError_t e = cudaLaunchKernelExC(&cfg, stage_in_kernel(), args);
  if (e != cudaSuccess) return fail_cuda("launch stage-in kernel", e);
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_workspace_bytes(int num_seqs, int num_heads, int head_size, int max_seq_len,
                          int partition_size) {
  size_t off[5];
  if (pa_workspace_layout(num_seqs, num_heads, head_size, max_seq_len, partition_size, off) !=
      PA_OK)
    return 0;
  return off[4] + align256((size_t)num_seqs * num_heads * 4);
}

pa_status_t pa_workspace_layout(int num_seqs, int num_heads, int head_size, int max_seq_len,
                                int partition_size, size_t offsets[5]) {
  if (!offsets || num_seqs < 0 || num_heads < 1 || head_size < 1 || max_seq_len < 0 ||
      partition_size < 1)
    return PA_ERR_INVALID_ARG;
  const size_t parts = (size_t)max_parts_of(max_seq_len, partition_size);
  const size_t stats = align256((size_t)num_seqs * num_heads * parts * 4);
  offsets[0] = 0;
  offsets[1] = kStatusBytes;
  offsets[2] = offsets[1] + stats;
  offsets[3] = offsets[2] + stats;
  offsets[4] = offsets[3] + align256((size_t)num_seqs * num_heads * parts * head_size * 4);
  return PA_OK;
}

pa_status_t pa_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace || workspace_bytes < (size_t)kStatusBytes || !aligned(workspace, 256))
    return PA_ERR_INVALID_ARG;
  cudaError_t e =
      cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda("cudaMemsetAsync(workspace)", e);
  return PA_OK;
}

pa_status_t pa_v1_forward(void *out, const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                          int head_size, int num_blocks, int block_size, int max_blocks_per_seq,
                          int max_seq_len, float scale, int partition_size, int dtype,
                          void *workspace, size_t workspace_bytes, void *stream) {
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  return run(make_call(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, num_blocks, block_size,
                       max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, workspace,
                       workspace_bytes, stream),
             PA_VARIANT_V1, opt);
}

pa_status_t pa_v2_forward(void *out, const void *query, const void *key_cache,
                          const void *value_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                          int head_size, int num_blocks, int block_size, int max_blocks_per_seq,
                          int max_seq_len, float scale, int partition_size, int dtype,
                          void *workspace, size_t workspace_bytes, void *stream) {
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  return run(make_call(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, num_blocks, block_size,
                       max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, workspace,
                       workspace_bytes, stream),
             PA_VARIANT_V2, opt);
}

pa_status_t pa_forward(void *out, const void *query, const void *key_cache,
                       const void *value_cache, const int32_t *block_tables,
                       const int32_t *seq_lens, int num_seqs, int num_heads, int num_kv_heads,
                       int head_size, int num_blocks, int block_size, int max_blocks_per_seq,
                       int max_seq_len, float scale, int partition_size, int dtype,
                       void *workspace, size_t workspace_bytes, void *stream,
                       const pa_options_t *opts) {
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  if (opts) opt = *opts;
  return run(make_call(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                       num_heads, num_kv_heads, head_size, num_blocks, block_size,
                       max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, workspace,
                       workspace_bytes, stream),
             opt.variant, opt);
}

pa_status_t pa_v2_partials(const void *query, const void *key_cache, const void *value_cache,
                           const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                           int num_heads, int num_kv_heads, int head_size, int num_blocks,
                           int block_size, int max_blocks_per_seq, int max_seq_len, float scale,
                           int partition_size, int dtype, int part_begin, int part_end,
                           void *workspace, size_t workspace_bytes, void *stream) {
  // `out` is never written in this mode; the query stands in for it in the
  // argument checks (it has the same size and alignment rules).
  Call c = make_call(const_cast<void *>(query), query, key_cache, value_cache, block_tables,
                     seq_lens, num_seqs, num_heads, num_kv_heads, head_size, num_blocks,
                     block_size, max_blocks_per_seq, max_seq_len, scale, partition_size, dtype,
                     workspace, workspace_bytes, stream);
  c.phases = 1;
  c.part_begin = part_begin;
  c.part_end = part_end;
  pa_status_t st = check_args(c, true);
  if (st != PA_OK) return st;
  if (num_seqs == 0 || part_begin >= part_end) return PA_OK;
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  return launch(c, true, opt);
}

pa_status_t pa_v2_combine(void *out, const int32_t *seq_lens, int num_seqs, int num_heads,
                          int head_size, int max_seq_len, int partition_size, int dtype,
                          const void *workspace, size_t workspace_bytes, void *stream) {
  Call c = make_call(out, nullptr, nullptr, nullptr, nullptr, seq_lens, num_seqs, num_heads, 1,
                     head_size, 1, 16, 1, max_seq_len, 1.0f, partition_size, dtype,
                     const_cast<void *>(workspace), workspace_bytes, stream);
  c.phases = 2;
  pa_status_t st = check_combine_args(c);
  if (st != PA_OK) return st;
  return launch_combine(c);
}

pa_status_t pa_chunks_forward(void *out, const void *query, const void *key_cache,
                              const void *value_cache, const int32_t *block_tables,
                              const int32_t *seq_lens, const int32_t *q_start, int num_seqs,
                              int num_rows, int max_chunk, int num_heads, int num_kv_heads,
                              int head_size, int num_blocks, int block_size,
                              int max_blocks_per_seq, int max_seq_len, float scale,
                              int partition_size, int dtype, void *workspace,
                              size_t workspace_bytes, void *stream, const pa_options_t *opts) {
  if (!q_start) return PA_ERR_INVALID_ARG;
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  if (opts) opt = *opts;
  Call c = make_call(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                     num_heads, num_kv_heads, head_size, num_blocks, block_size,
                     max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, workspace,
                     workspace_bytes, stream);
  c.q_start = q_start;
  c.num_rows = num_rows;
  c.max_chunk = max_chunk;
  if (num_rows == 0) return check_args(c, false);
  return run(c, opt.variant, opt);
}

size_t pa_host_staging_bytes(int num_seqs, int num_heads, int head_size,
                             int max_blocks_per_seq, int dtype) {
  if (num_seqs < 0 || num_heads < 1 || head_size < 1 || max_blocks_per_seq < 1 ||
      (dtype != PA_DTYPE_F32 && dtype != PA_DTYPE_BF16 && dtype != PA_DTYPE_F16))
    return 0;
  const size_t qo = align256((size_t)num_seqs * num_heads * head_size * elt_size(dtype));
  return 2 * qo + align256((size_t)num_seqs * max_blocks_per_seq * 4) +
         align256((size_t)num_seqs * 4) + (num_seqs == 0 ? 256 : 0);
}

pa_status_t pa_forward_host(void *out_host, const void *query_host, const void *key_cache,
                            const void *value_cache, const int32_t *block_tables_host,
                            const int32_t *seq_lens_host, int num_seqs, int num_heads,
                            int num_kv_heads, int head_size, int num_blocks, int block_size,
                            int max_blocks_per_seq, int max_seq_len, float scale,
                            int partition_size, int dtype, void *staging, size_t staging_bytes,
                            void *workspace, size_t workspace_bytes, void *stream,
                            const pa_options_t *opts) {
  if (!out_host || !query_host || !block_tables_host || !seq_lens_host || !staging ||
      !aligned(staging, 256))
    return PA_ERR_INVALID_ARG;
  const size_t need =
      pa_host_staging_bytes(num_seqs, num_heads, head_size, max_blocks_per_seq, dtype);
  if (need == 0 || staging_bytes < need) return PA_ERR_INVALID_ARG;
  pa_options_t opt;
  memset(&opt, 0, sizeof opt);
  if (opts) opt = *opts;
  // staging: query | out | block tables | seq_lens
  const size_t qbytes = (size_t)num_seqs * num_heads * head_size * elt_size(dtype);
  const size_t tbytes = (size_t)num_seqs * max_blocks_per_seq * 4;
  uint8_t *st = static_cast<uint8_t *>(staging);
  void *q_dev = st;
  void *out_dev = st + align256(qbytes);
  int32_t *bt_dev = reinterpret_cast<int32_t *>(st + 2 * align256(qbytes));
  int32_t *sl_dev = reinterpret_cast<int32_t *>(st + 2 * align256(qbytes) + align256(tbytes));
  Call c = make_call(out_dev, q_dev, key_cache, value_cache, bt_dev, sl_dev, num_seqs,
                     num_heads, num_kv_heads, head_size, num_blocks, block_size,
                     max_blocks_per_seq, max_seq_len, scale, partition_size, dtype, workspace,
                     workspace_bytes, stream);
  // Pinned host buffers are mapped into the device: then a kernel reads the
  // inputs and the last kernel writes the output in place (no copy engine).
  void *out_map = nullptr;
  const void *q_map = nullptr, *bt_map = nullptr, *sl_map = nullptr;
  const bool mapped = device_view(out_host, &out_map) && device_view(query_host, &q_map) &&
                      device_view(block_tables_host, &bt_map) &&
                      device_view(seq_lens_host, &sl_map) && aligned(out_map, 16);
  if (mapped) c.out = out_map;
  // argument problems are reported before anything is enqueued
  bool v2 = false;
  pa_status_t chk = resolve(c, opt.variant, &v2);
  if (chk != PA_OK) return chk;
  if (num_seqs == 0) return PA_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (mapped) {
    pa_status_t r = stage_in(sl_map, sl_dev, (size_t)num_seqs * 4, bt_map, bt_dev, tbytes, q_map,
                             q_dev, qbytes, s);
    if (r != PA_OK) return r;
    return launch(c, v2, opt);
  }
  cudaError_t e = cudaMemcpyAsync(sl_dev, seq_lens_host, (size_t)num_seqs * 4,
                                  cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_cuda("cudaMemcpyAsync(seq_lens)", e);
  e = cudaMemcpyAsync(bt_dev, block_tables_host, tbytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_cuda("cudaMemcpyAsync(block_tables)", e);
  e = cudaMemcpyAsync(q_dev, query_host, qbytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return fail_cuda("cudaMemcpyAsync(query)", e);
  pa_status_t r = launch(c, v2, opt);
  if (r != PA_OK) return r;
  e = cudaMemcpyAsync(out_host, out_dev, qbytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return fail_cuda("cudaMemcpyAsync(out)", e);
  return PA_OK;
}

int pa_choose_v2(int num_seqs, int num_kv_heads, int max_seq_len, int partition_size,
                 int sm_count) {
  // Every sequence in one partition: V2 would only add the reduce.
  if (partition_size < 1 || max_seq_len <= partition_size) return 0;
  if (sm_count <= 0) return 1;
  // V1 has one work item per (sequence, KV head).  Measured on GB300 (bf16,
  // D 128, 32 q / 4 kv heads, lengths uniform in [L/2, L], consecutive steps
  // with the K/V cold in L2), V1 is ahead:
  //   - with at least 16 items per SM, at every length (2-6 %): the items
  //     balance over the persistent CTAs and V2's partials and reduce are
  //     pure overhead;
  //   - with 8 to 16 items per SM, up to 2 partitions of length;
  //   - with 2 to 3 items per SM, i.e. one item per resident CTA with at
  //     least two CTAs streaming on every SM, up to 4 partitions of length.
  // Everywhere else (one CTA per SM, or a second round of uneven items)
  // V2's finer items win.
  const long long items = (long long)num_seqs * num_kv_heads;
  const long long sm = sm_count;
  if (items >= 16 * sm) return 0;
  if (items >= 8 * sm && max_seq_len <= 2LL * partition_size) return 0;
  if (items >= 2 * sm && items <= 3 * sm && max_seq_len <= 4LL * partition_size) return 0;
  return 1;
}

int pa_choose_v2_chunks(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                        int max_chunk, int max_seq_len, int partition_size, int sm_count) {
  if (partition_size < 1 || max_seq_len <= partition_size) return 0;
  if (sm_count <= 0 || num_kv_heads < 1 || num_heads < num_kv_heads || max_chunk < 1) return 1;
  const int group = num_heads / num_kv_heads;
  const long long rows = (long long)max_chunk * group;
  // Up to 8 (token, head) rows per KV head the item costs what a decode item
  // does: the decode rule holds.
  if (rows <= 8)
    return pa_choose_v2(num_seqs, num_kv_heads, max_seq_len, partition_size, sm_count);
  // Items as the chunk kernels cut them: 128 rows on tcgen05, 64 on
  // row-owning warps, else 16.
  const bool umma = umma_chunk_ok(head_size, group, rows);
  const bool row_owning = (head_size == 64 || head_size == 128) && 64 % group == 0 && rows > 32;
  const int tokens = (umma ? 128 : row_owning ? 64 : 16) / group;
  const long long groups = (max_chunk + tokens - 1) / tokens;
  const long long items = (long long)num_seqs * num_kv_heads * groups;
  // Measured on GB300 (bf16, D 128, 32 q / 4 kv heads; 256 sequences of up
  // to 3584 tokens with 2 to 64 tokens a chunk, 8 of up to 8192 and one of
  // 100,000; consecutive steps).  On the 16- and 64-row kernels V1 is ahead
  // from 2048 items (13.5 per SM: 1.23x at 4 tokens), V2 at 1024 and fewer
  // (6.7 per SM: 1.02x at 2 tokens, 1.12x at 8).  On the tcgen05 kernel V1 is
  // ahead from 1024 items (1.36x at 16 tokens, 1.67x at 64), V2 at 128 and
  // fewer.  A chunk item's epilogue costs more than a decode item's, and V1
  // pays it once per sequence; each switch sits between the measured counts.
  if (items >= (umma ? 4LL : 8LL) * sm_count) return 0;
  return 1;
}

pa_status_t pa_read_device_status(void *workspace, void *stream) {
  if (!workspace || !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_cuda("cudaStreamSynchronize", e);
  int v = 0;
  e = cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda("cudaMemcpy(status)", e);
  if (v != 0) {
    e = cudaMemset(workspace, 0, sizeof v);
    if (e != cudaSuccess) return fail_cuda("cudaMemset(status)", e);
  }
  return static_cast<pa_status_t>(v);
}

const char *pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE_BAD_INPUT: return "kernel found a bad block-table entry or sequence length";
    case PA_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
  }
  return "unknown status";
}

const char *pa_last_cuda_error(void) { return g_last_error; }

int pa_version(void) { return 100; }

}  // extern "C"
