// Attention for items of at most 16 query rows on the 5th-generation tensor
// cores (tcgen05, sm_103a), D = 128, 16-bit inputs: decode with up to 16 query
// heads a KV head, and query chunks of up to 16 (token, head) rows per KV head.
//
// The keys take the MMA's M, the few query rows its N, so no lane of the
// tensor core computes a query row that does not exist:
//   S^T[128 keys][16 rows]  = K[128][D] . Q^T         (both K-major)
//   O^T[D][16 rows]        += V^T[D][128 keys] . P^T  (V MN-major, P^T K-major)
// with fp32 accumulators in tensor memory.  A softmax thread owns one key of
// the stage (its tensor-memory lane) and sees that key's score for every
// row; the rows' running maxima are common to all threads and raised lazily:
// an exchange among the four softmax warps tells whether any score of the
// stage exceeds its row's maximum in use by more than 2^8 (exponent units),
// and only then are the stage's row maxima formed and O^T and the partial
// sums rescaled, which is exact because the final normaliser uses the same
// maxima.  Each thread keeps its own partial row sums; they are added across
// the threads once per item, as are the true maxima the partials record.  A
// thread of the epilogue owns one column d of O^T for all rows; the outputs
// leave through the TMA engine (bulk copies from shared memory), as the
// plain stores of a CTA whose copies keep HBM busy each wait for the memory
// system.
//
// Warps: 0-3 softmax and output, 4 producer (TMA of K/V pages and of each
// item's queries, work items), 5 MMA issuer (and the tensor-memory
// allocation).  One CTA an SM; every wait is bounded.
//
// Taken only when asked for (PA_DEBUG_TCGEN05_KEYS): on GB300 the 16-row
// mma.sync kernel, two CTAs an SM, is faster on decode with 16 query heads a
// KV head (0.098 against 0.116-0.146 ms a step on the 256-sequence cache).
// Measured there, with a per-CTA %globaltimer trace: a stage streams at about
// the HBM rate within an item, but the producer issues a 4 KB page copy about
// every 65 ns (near the 16 a stage that HBM needs), and each item boundary
// costs microseconds (the next item's lookup and block-table loads, which
// wait for the memory system while the CTA's own copies keep HBM busy, and
// the epilogue) that a second CTA would cover but the shared memory of the
// 128-key ring leaves no room for.
#include <type_traits>

#include "pa_attn.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kKeysStage = 128;  // keys of a stage: the S MMA's M, the PV MMAs' K
constexpr int kKeysM = kKeysStage;
constexpr int kKeysN = 16;       // query rows of an item: the MMAs' N
constexpr int kKeysD = 128;      // head size
constexpr int kKeysTmemCols = 64;  // S^T at columns 0 and 16 (two buffers), O^T at 32
constexpr int kKeysKSlots = 3;
constexpr int kKeysVSlots = 3;
// A K (or V) slot holds 128 keys as [8-key group][panel][8 keys][128 B], each
// 8-key piece of a panel one 1024-byte swizzle atom; a page's rows arrive in
// one 4-D copy.
constexpr int kKeysGroup = (kKeysD * 2 / 128) * 1024;
constexpr int kKeysSlot = (kKeysStage / 8) * kKeysGroup;  // 32 KB
// Q of an item: [panel][16 rows][128 B], 2 KB a panel; P^T of a stage: two
// such panels (64 keys each)
constexpr int kKeysTilePanel = kKeysN * 128;
constexpr int kKeysTile = (kKeysD * 2 / 128) * kKeysTilePanel;
constexpr int kKeysPTile = (kKeysStage * 2 / 128) * kKeysTilePanel;
constexpr int kKeysOTile = kKeysN * kKeysD * 4;  // an item's output rows, fp32
constexpr float kKeysMargin = 8.f;  // log2 units

struct KeysStage {
  int row0, kvh, part;  // the item: first query row, KV head, partition
  int tok0;             // key of the stage's first row
  int valid;            // keys of the stage in the item's range
  int flags;            // kStage*
  int rows;             // (token, head) rows of the item
  int lim_base;         // row n sees keys below lim_base + n / group + 1
  int qb;               // the item's query buffer
  int pad[3];
};

// One value per row (16) in every lane of a warp, reduced over the warp's 32
// lanes: each of five exchange steps halves the rows a lane keeps, so the
// lanes 2c and 2c + 1 end with row c, after 16 shuffles in all.
template <bool MAX>
__device__ __forceinline__ float op2(float a, float b) {
  return MAX ? fmaxf(a, b) : a + b;
}
template <bool MAX>
__device__ __forceinline__ float warp_rows_reduce(const float (&v)[kKeysN], int lane) {
  float a8[8], a4[4], a2[2];
  const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4, h1 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float send = h4 ? v[j] : v[8 + j];
    const float keep = h4 ? v[8 + j] : v[j];
    a8[j] = op2<MAX>(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = h3 ? a8[j] : a8[4 + j];
    const float keep = h3 ? a8[4 + j] : a8[j];
    a4[j] = op2<MAX>(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = h2 ? a4[j] : a4[2 + j];
    const float keep = h2 ? a4[2 + j] : a4[j];
    a2[j] = op2<MAX>(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  float a1;
  {
    const float send = h1 ? a2[0] : a2[1];
    const float keep = h1 ? a2[1] : a2[0];
    a1 = op2<MAX>(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  return op2<MAX>(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from shared to global memory through the TMA engine, in this thread's
// current bulk group.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(dst)),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// this thread's bulk copies have read their shared-memory sources
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// this thread's bulk copies are complete
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <typename T>
__device__ __forceinline__ unsigned short to_bits16(float x) {
  const T h = from_float<T>(x);
  return *reinterpret_cast<const unsigned short *>(&h);
}

}  // namespace

// One CTA an SM (its shared memory allows no second).
template <typename T>
__global__ void __launch_bounds__(192, 1)
    pa_umma_keys_kernel(const __grid_constant__ AttnParams p,
                        const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ CUtensorMap tmap_q) {
  constexpr int D = kKeysD;
  constexpr int NK = kKeysKSlots, NV = kKeysVSlots;
  constexpr int NPANELS = D * (int)sizeof(T) / 128;
  constexpr uint32_t kIdescS = instr_desc<T>(kKeysM, kKeysN, false, false);
  constexpr uint32_t kIdescPV = instr_desc<T>(kKeysD, kKeysN, false, true);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The 128-byte swizzle needs every tile 1024-byte aligned.  The kernel's
  // shared memory leaves no room for alignment slack, so it relies on the
  // dynamic shared memory starting 1024-byte aligned (right after the 1 KB
  // the system reserves) and checks it.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) report(p.status, kStatusBadInput);
    return;
  }
  uint8_t *kring = smem_raw;                    // NK x [16 groups][panel][8 keys][128 B]
  uint8_t *vring = kring + NK * kKeysSlot;      // NV x the same
  uint8_t *qbuf = vring + NV * kKeysSlot;       // 2 x [panel][16 rows][128 B]
  uint8_t *pbuf = qbuf + 2 * kKeysTile;         // 2 x [key panel][16 rows][128 B]
  float *obuf = reinterpret_cast<float *>(pbuf + 2 * kKeysPTile);  // [16 rows][D] outputs
  KeysStage *info = reinterpret_cast<KeysStage *>(reinterpret_cast<uint8_t *>(obuf) + kKeysOTile);
  // the softmax warps' exchanges: 2 x [4 warps][32 floats]
  float *xbuf = reinterpret_cast<float *>(info + NK);
  uint64_t *bars = reinterpret_cast<uint64_t *>(xbuf + 2 * 4 * 32);
  // fullK[NK], emptyK[NK], fullV[NV], emptyV[NV], q_full[2], q_empty[2],
  // s_full[2], p_full[2], o_done, drain, never, grp
  constexpr int NBARS = 2 * NK + 2 * NV + 12;
  volatile int *flags = reinterpret_cast<volatile int *>(bars + NBARS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS) + 4;
  const uint32_t kring_u32 = smem_u32(kring), vring_u32 = smem_u32(vring);
  const uint32_t q_u32 = smem_u32(qbuf), p_u32 = smem_u32(pbuf);
  const uint32_t fullk0 = smem_u32(bars), emptyk0 = fullk0 + 8 * NK;
  const uint32_t fullv0 = emptyk0 + 8 * NK, emptyv0 = fullv0 + 8 * NV;
  const uint32_t q_full = emptyv0 + 8 * NV, q_empty = q_full + 16, s_full = q_empty + 16,
                 p_full = s_full + 16, o_done = p_full + 16, drain = o_done + 8,
                 never = drain + 8, grp = never + 8;
  const uint64_t limit = p.wait_limit_ns;
  const int G = p.group;
  const bool decode = p.q_start == nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NK; ++i) {
      mbar_init(fullk0 + 8 * i, 1);
      mbar_init(emptyk0 + 8 * i, 5);  // the S MMA's commit and each softmax warp's header read
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(fullv0 + 8 * i, 1);
      mbar_init(emptyv0 + 8 * i, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full + 8 * b, 1);
      mbar_init(q_empty + 8 * b, 1);
      mbar_init(s_full + 8 * b, 1);
      mbar_init(p_full + 8 * b, 4);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    mbar_init(grp, 4);
    flags[0] = 0;
    fence_mbar_init();
  }
  // query rows past an item's rows are never copied: zeros, once
  for (int e = threadIdx.x; e < 2 * kKeysTile / 16; e += blockDim.x)
    reinterpret_cast<uint4 *>(qbuf)[e] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  // Launched with programmatic dependent launch: wait for the previous kernel
  // in the stream before the tensor memory is taken and before any global
  // access.
  pdl_wait_primary();
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kKeysTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 32;

  if (warp == 4) {
    // ======================= producer warp =======================
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
      prefetch_tmap(&tmap_q);
    }
    const int U = p.unit_rows;
    const int TQ = decode ? 1 : p.chunk_tokens;  // query tokens of an item
    const bool v2 = p.write_partials != 0;
    // the running count of items per sequence, 32 sequences at a time; items
    // are (KV head, partition) in decode, (KV head, partition, row group)
    // for query chunks; V1 decode gives an empty sequence its items too (they
    // write zeros)
    int cs = 0, cbase = 0, c_cnt = 0, c_incl = 0, c_L = 0, c_total = 0, c_qs = 0, c_n = 0,
        c_nrg = 0;
    bool c_loaded = false;
    auto per_head_of = [&](int L, int nrg) -> int {
      const int np = (L + p.range_tokens - 1) / p.range_tokens;
      if (!decode) return np * nrg;
      return v2 ? max(0, min(np, p.part_end) - p.part_begin) : 1;
    };
    auto load_chunk = [&]() {
      const int sl = cs + lane;
      c_L = 0;
      c_qs = 0;
      c_n = 0;
      if (sl < p.num_seqs) {
        c_L = __ldg(p.seq_lens + sl);
        if (c_L < 0 || c_L > p.max_seq_len) {
          report(p.status, kStatusBadInput);
          c_L = c_L < 0 ? 0 : p.max_seq_len;
        }
        if (!decode) {
          c_qs = __ldg(p.q_start + sl);
          const int qe = __ldg(p.q_start + sl + 1);
          c_n = qe - c_qs;
          if (c_qs < 0 || c_n < 0 || c_n > c_L || qe > p.num_rows) {
            report(p.status, kStatusBadInput);  // its rows get no items
            c_n = 0;
          }
        }
      }
      c_nrg = (c_n + TQ - 1) / TQ;
      c_cnt = sl < p.num_seqs ? p.num_kv_heads * per_head_of(c_L, c_nrg) : 0;
      c_incl = c_cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, c_incl, off);
        if (lane >= off) c_incl += t;
      }
      c_total = __shfl_sync(0xffffffffu, c_incl, 31);
      c_loaded = true;
    };
    bool ok = true;
    auto grab_issue = [&]() -> int { return atomic_add_lane0(p.sched, lane); };
    const int takers = (int)gridDim.x;
    auto next_item = [&](int raw) -> int { return takers + __shfl_sync(0xffffffffu, raw, 0); };
    // An item: its sequence, KV head, partition, keys [tok_begin, tok_end),
    // output rows (row0, rows) and key limits; found = false past the last.
    struct Item {
      int s, kvh, part, tok_begin, tok_end, row0, rows, lim_base;
      bool found;
    };
    auto locate = [&](int item, Item &d) {
      d.found = false;
      if (item < 0) {  // a corrupted work counter: stop rather than guess
        if (lane == 0) report(p.status, kStatusBadInput);
        return;
      }
      int L = 0, qs = 0, n_s = 0, rg = 0;
      while (true) {
        if (!c_loaded) load_chunk();
        if (item < cbase + c_total) {
          const unsigned hit = __ballot_sync(0xffffffffu, cbase + c_incl > item);
          const int ls = __ffs(hit) - 1;
          d.s = cs + ls;
          L = __shfl_sync(0xffffffffu, c_L, ls);
          const int nrg = __shfl_sync(0xffffffffu, c_nrg, ls);
          qs = __shfl_sync(0xffffffffu, c_qs, ls);
          n_s = __shfl_sync(0xffffffffu, c_n, ls);
          const int first = cbase + __shfl_sync(0xffffffffu, c_incl - c_cnt, ls);
          const int per_head = per_head_of(L, nrg);
          d.kvh = (item - first) / per_head;
          const int rem = (item - first) % per_head;
          if (decode) {
            d.part = v2 ? p.part_begin + rem : 0;
          } else {
            d.part = rem / nrg;
            rg = rem % nrg;
          }
          d.found = d.s < p.num_seqs;
          break;
        }
        if (cs + 32 >= p.num_seqs) break;
        cs += 32;
        cbase += c_total;
        c_loaded = false;
      }
      if (!d.found) return;
      d.tok_begin = d.part * p.range_tokens;
      d.tok_end = min(d.tok_begin + p.range_tokens, L);
      d.row0 = d.s;  // decode: row s, every key of the range
      d.rows = G;
      d.lim_base = L - 1;
      if (!decode) {
        const int t_first = rg * TQ;
        const int ntok = min(TQ, n_s - t_first);
        d.rows = ntok * G;
        d.lim_base = L - n_s + t_first;  // keys below lim_base + t + 1 for token t of the group
        d.row0 = qs + t_first;
        d.tok_end = min(d.tok_end, d.lim_base + ntok);
        if (d.part == 0 && p.row_limit)
          for (int t = lane; t < ntok; t += 32) p.row_limit[d.row0 + t] = d.lim_base + t + 1;
      }
    };
    // The first item from `item` on that has keys; V1 decode writes the zeros
    // of empty sequences on the way
    auto advance = [&](int item, Item &d) {
      while (true) {
        locate(item, d);
        if (!d.found || d.tok_end > d.tok_begin) return;
        if (decode && !v2) {
          T *o = static_cast<T *>(p.out) + ((size_t)d.s * p.num_heads + (size_t)d.kvh * G) * D;
          for (int e = lane; e < G * D; e += 32) o[e] = from_float<T>(0.f);
        }
        item = next_item(grab_issue());
      }
    };
    // a window of 64 block-table entries of the item (lane j: pages
    // win0 + j and win0 + 32 + j), slid by 32 pages when a stage reaches the
    // second half; loaded ahead, while the item before streams
    auto load_window = [&](const Item &d, int w0, int &c0, int &c1) {
      const int32_t *bt = p.block_tables + (size_t)d.s * p.max_blocks_per_seq;
      const int last_page = (d.tok_end - 1) >> p.log2_block_size;
      const int a = w0 + lane, b = w0 + 32 + lane;
      c0 = (a <= last_page) ? __ldg(bt + a) : -1;
      c1 = (b <= last_page) ? __ldg(bt + b) : -1;
    };
    int i = 0;           // stages issued
    int ik = 0, iv = 0;  // stages whose K (with the end marker) and V copies are issued
    int qi = 0;          // items whose queries are issued
    Item d;
    advance((int)blockIdx.x, d);
    int cur = -1, nxt = -1;
    if (d.found) load_window(d, d.tok_begin >> p.log2_block_size, cur, nxt);
    while (d.found) {
      // the item's queries: rows (token t, head j) at n = t * G + j of the
      // buffer, one 3-D copy a panel; the buffer was read by the S MMAs of
      // the item two before
      const int qb = qi & 1;
      if (qi >= 2) {
        bool w = true;
        if (lane == 0) w = mbar_wait(q_empty + 8 * qb, ((qi >> 1) - 1) & 1, limit, flags);
        ok = __shfl_sync(0xffffffffu, w, 0);
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full + 8 * qb, (uint32_t)(NPANELS * 128 * G * TQ));
        for (int pn = 0; pn < NPANELS; ++pn)
          tma_load_3d(q_u32 + (uint32_t)(qb * kKeysTile + pn * kKeysTilePanel), &tmap_q, pn * 64,
                      d.kvh * G, d.row0, q_full + 8 * qb);
      }
      ++qi;
      const int32_t *bt = p.block_tables + (size_t)d.s * p.max_blocks_per_seq;
      const int last_page = (d.tok_end - 1) >> p.log2_block_size;
      int win0 = d.tok_begin >> p.log2_block_size;
      const int n_st = (d.tok_end - d.tok_begin + kKeysStage - 1) / kKeysStage;
      int next_raw = 0;
      Item dn;
      dn.found = false;
      int ncur = -1, nnxt = -1;
      for (int j = 0; j < n_st; ++j) {
        const int sk = i % NK, sv = i % NV;
        if (i >= NK) {  // K slot: the S MMA and every softmax warp are done with it
          bool w = true;
          if (lane == 0) w = mbar_wait(emptyk0 + 8 * sk, ((i / NK) - 1) & 1, limit, flags);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
        }
        const int stage_tok0 = d.tok_begin + j * kKeysStage;
        const int valid = min(kKeysStage, d.tok_end - stage_tok0);
        const int n_units = (valid + U - 1) / U;
        const int tok = stage_tok0 + lane * U;
        const int rel = ((lane < n_units ? tok : stage_tok0) >> p.log2_block_size) - win0;
        const int a = __shfl_sync(0xffffffffu, cur, rel & 31);
        const int b = __shfl_sync(0xffffffffu, nxt, rel & 31);
        int y = -1;
        if (lane < n_units) {
          const int blk = rel < 32 ? a : b;
          if ((unsigned)blk >= (unsigned)p.num_blocks)
            report(p.status, kStatusBadInput);
          else
            y = (blk * p.num_kv_heads + d.kvh) * p.block_size + (tok & (p.block_size - 1));
        }
        const unsigned valid_mask = __ballot_sync(0xffffffffu, y >= 0);
        const uint32_t stage_bytes = (uint32_t)__popc(valid_mask) * U * 128u * NPANELS;
        if (lane == 0) {
          KeysStage &h = info[sk];
          h.row0 = d.row0;
          h.kvh = d.kvh;
          h.part = d.part;
          h.tok0 = stage_tok0;
          h.valid = valid;
          h.flags = (j == 0 ? kStageFirst : 0) | (j == n_st - 1 ? kStageLast : 0);
          h.rows = d.rows;
          h.lim_base = d.lim_base;
          h.qb = qb;
          mbar_arrive_expect_tx(fullk0 + 8 * sk, stage_bytes);
        }
        __syncwarp();
        // rows lane * U .. of the stage: groups lane * U / 8 .., every panel
        if (y >= 0)
          tma_load_4d(kring_u32 + (uint32_t)sk * kKeysSlot + (uint32_t)(lane * U / 8) * kKeysGroup,
                      &tmap_k, 0, 0, 0, y >> 3, fullk0 + 8 * sk);
        ik = i + 1;
        if (i >= NV) {  // V slot: the PV of stage i - NV has read it
          bool w = true;
          if (lane == 0) w = mbar_wait(emptyv0 + 8 * sv, ((i / NV) - 1) & 1, limit, flags);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
        }
        if (lane == 0) mbar_arrive_expect_tx(fullv0 + 8 * sv, stage_bytes);
        __syncwarp();
        if (y >= 0)
          tma_load_4d(vring_u32 + (uint32_t)sv * kKeysSlot + (uint32_t)(lane * U / 8) * kKeysGroup,
                      &tmap_v, 0, 0, 0, y >> 3, fullv0 + 8 * sv);
        iv = i + 1;
        ++i;
        // The next item is taken from the counter once this item's first
        // copies are issued, and located, with its block-table window
        // loading, once its second are (at once for an item of one stage):
        // the producer then mostly waits for free slots, and the next item
        // starts without a round trip.
        if (j == 0) next_raw = grab_issue();
        if (j == min(1, n_st - 1)) {
          advance(next_item(next_raw), dn);
          if (dn.found) load_window(dn, dn.tok_begin >> p.log2_block_size, ncur, nnxt);
        }
        const int next_rel = ((stage_tok0 + kKeysStage) >> p.log2_block_size) - win0;
        if (next_rel >= 32) {
          cur = nxt;
          win0 += 32;
          const int e = win0 + 32 + lane;
          nxt = (e <= last_page) ? __ldg(bt + e) : -1;
        }
      }
      if (!ok) break;
      d = dn;
      cur = ncur;
      nxt = nnxt;
    }
    pdl_launch_dependents();
    if (ok) {  // no more items: a K slot's header says so
      const int sk = i % NK;
      if (i >= NK) {
        bool w = true;
        if (lane == 0) w = mbar_wait(emptyk0 + 8 * sk, ((i / NK) - 1) & 1, limit, flags);
        ok = __shfl_sync(0xffffffffu, w, 0);
      }
      if (ok && lane == 0) {
        info[sk].flags = kStageEnd;
        mbar_arrive(fullk0 + 8 * sk);
      }
      if (ok) ik = ++i;
    }
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    if (lane == 0) {  // every copy of this CTA lands before it retires
      for (int j = ik > NK ? ik - NK : 0; j < ik; ++j)
        mbar_wait(fullk0 + 8 * (j % NK), (j / NK) & 1, kDrainLimitNs, nullptr);
      for (int j = iv > NV ? iv - NV : 0; j < iv; ++j)
        mbar_wait(fullv0 + 8 * (j % NV), (j / NV) & 1, kDrainLimitNs, nullptr);
      for (int j = qi > 2 ? qi - 2 : 0; j < qi; ++j)
        mbar_wait(q_full + 8 * (j & 1), (j >> 1) & 1, kDrainLimitNs, nullptr);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================= MMA warp (one thread issues) =======================
    if (lane == 0) {
      bool ok = true;
      int km = 0;  // items whose queries the S MMAs have taken
      // S^T = K Q^T of the stage in K slot `sk` into S buffer b: D / 16
      // k-steps, each 32 bytes inside a 128-byte panel of K (8-key groups
      // kKeysGroup bytes apart, panels 1024 bytes apart) and of Q (8-row
      // atoms 1024 bytes apart, panels 2 KB apart).  Its commit also frees
      // the K slot (with the softmax warps' header reads), and after an
      // item's last stage the query buffer.
      auto issue_s = [&](int sk, int b, const KeysStage &hs) {
        const uint32_t kst = kring_u32 + (uint32_t)sk * kKeysSlot;
        const uint32_t qst = q_u32 + (uint32_t)hs.qb * kKeysTile;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (uint32_t)(ks & 3) * 32u;
          const uint64_t da = smem_desc(kst + (uint32_t)(ks >> 2) * 1024u + koff, 16, kKeysGroup);
          const uint64_t db = smem_desc(qst + (uint32_t)(ks >> 2) * kKeysTilePanel + koff, 16, 1024);
          tc_mma(tmem_s + 16u * (uint32_t)b, da, db, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full + 8u * (uint32_t)b);
        tc_commit(emptyk0 + 8u * (uint32_t)sk);
        if (hs.flags & kStageLast) tc_commit(q_empty + 8u * (uint32_t)hs.qb);
      };
      // The S of stage i + 1 is issued before the PV of stage i whenever its
      // keys (and, for a new item, its queries) are already here: its buffer
      // was read by the softmax of stage i - 1, whose P the PV of i - 1
      // waited for.
      KeysStage h{};
      ok = mbar_wait(fullk0, 0, limit, flags);
      if (ok) h = info[0];
      bool more = ok && !(h.flags & kStageEnd);
      if (more) {
        ok = mbar_wait(q_full + 8 * h.qb, (km >> 1) & 1, limit, flags);
        ++km;
        if (ok) {
          tc_fence_after();
          issue_s(0, 0, h);
        }
        more = ok;
      }
      for (int i = 0; more; ++i) {
        const int sv = i % NV, sk1 = (i + 1) % NK;
        const uint32_t par1 = ((i + 1) / NK) & 1;
        bool s1 = false;
        KeysStage h1{};
        if (mbar_test(fullk0 + 8 * sk1, par1)) {
          h1 = info[sk1];
          if (!(h1.flags & kStageEnd)) {
            const bool fresh = (h1.flags & kStageFirst) != 0;
            if (!fresh || mbar_test(q_full + 8 * h1.qb, (km >> 1) & 1)) {
              if (fresh) ++km;
              tc_fence_after();
              issue_s(sk1, (i + 1) & 1, h1);
              s1 = true;
            }
          }
        }
        ok = mbar_wait(p_full + 8 * (i & 1), (i >> 1) & 1, limit, flags);
        if (!ok) break;
        ok = mbar_wait(fullv0 + 8 * sv, (i / NV) & 1, limit, flags);  // the stage's V is in
        if (!ok) break;
        tc_fence_after();
        // O^T += V^T P^T: 8 k-steps of 16 keys; V^T MN-major (64 columns of D
        // a panel, panels 1024 bytes apart (LBO); 8 keys a group, groups
        // kKeysGroup apart (SBO)); P^T K-major like Q
        const uint32_t vst = vring_u32 + (uint32_t)sv * kKeysSlot;
        const uint32_t pst = p_u32 + (uint32_t)(i & 1) * kKeysPTile;
#pragma unroll
        for (int kk = 0; kk < kKeysStage / 16; ++kk) {
          const uint64_t da = smem_desc(vst + (uint32_t)kk * 2u * kKeysGroup, 1024, kKeysGroup);
          const uint64_t db =
              smem_desc(pst + (uint32_t)(kk >> 2) * kKeysTilePanel + (uint32_t)(kk & 3) * 32u, 16, 1024);
          tc_mma(tmem_o, da, db, kIdescPV, ((h.flags & kStageFirst) && kk == 0) ? 0u : 1u);
        }
        tc_commit(emptyv0 + 8 * sv);  // the V slot and the P^T buffer are read
        if (h.flags & kStageLast) tc_commit(o_done);
        if (!s1) {
          ok = mbar_wait(fullk0 + 8 * sk1, par1, limit, flags);
          if (!ok) break;
          h1 = info[sk1];
          if (h1.flags & kStageEnd) break;
          if (h1.flags & kStageFirst) {
            ok = mbar_wait(q_full + 8 * h1.qb, (km >> 1) & 1, limit, flags);
            if (!ok) break;
            ++km;
          }
          tc_fence_after();
          issue_s(sk1, (i + 1) & 1, h1);
        }
        h = h1;
      }
      // nothing of this thread's may still run when the memory is freed
      tc_commit(drain);
      mbar_wait(drain, 0, kDrainLimitNs, nullptr);
      if (!ok) {
        report(p.status, kStatusTimeout);
        flags[0] = 1;
      }
    }
    __syncwarp();
  } else {
    // =============== softmax warps: thread = key of the stage ===============
    // thread t: key t of each stage (tensor-memory lane t of S^T), and row
    // d = t of O^T (its lane there) in the rescale and the epilogue
    const int t = threadIdx.x;
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    float m_run[kKeysN], l[kKeysN], mt[kKeysN];
    int tokn[kKeysN];  // row n's token within the item
#pragma unroll
    for (int n = 0; n < kKeysN; ++n) {
      tokn[n] = n / G;
      m_run[n] = -CUDART_INF_F;
      l[n] = 0.f;
      mt[n] = -CUDART_INF_F;
    }
    bool ok = true;
    int items = 0, gx = 0;
    // One exchange among the four softmax warps: a lane's value into place
    // `idx` of its warp's row (when `put`), then all four warps' rows, after a
    // bounded wait; two areas in turn, so a warp that runs ahead never
    // overwrites what a slower one has still to read.
    auto exchange = [&](bool put, int idx, float v) -> const float * {
      float *area = xbuf + (gx & 1) * 128;
      if (put) area[warp * 32 + idx] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(grp);
      const bool w = mbar_wait(grp, (uint32_t)(gx & 1), limit, flags);
      ok = __all_sync(0xffffffffu, w);
      ++gx;
      return area;
    };
    if (p.debug_flags & kDebugStallConsumers) {
      // Wait on a barrier that nothing releases: the bound must end it.
      ok = mbar_wait(never, 0, limit, flags);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; ok; ++i) {
      const int sk = i % NK, sv = i % NV;
      {
        const bool w = mbar_wait(fullk0 + 8 * sk, (i / NK) & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
      }
      const KeysStage h = info[sk];
      __syncwarp();
      if (h.flags & kStageEnd) break;
      if (lane == 0) mbar_arrive(emptyk0 + 8 * sk);  // this warp is done with the header
      if (h.flags & kStageFirst) {
#pragma unroll
        for (int n = 0; n < kKeysN; ++n) {
          m_run[n] = -CUDART_INF_F;
          l[n] = 0.f;
          mt[n] = -CUDART_INF_F;
        }
      }
      {
        const bool w = mbar_wait(s_full + 8 * (i & 1), (i >> 1) & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
      }
      tc_fence_after();
      uint32_t sr[kKeysN];
      tmem_ld16(tmem_s + 16u * (uint32_t)(i & 1) + lane_off, sr);
      tmem_ld_wait16(sr);
      // scores in log2 units; key t is seen by row n if it lies in the
      // item's range and below the row's limit, else -inf
      const bool in_range = t < h.valid;
      const int klim = h.lim_base + 1 - h.tok0 - t;  // key t visible to row n iff klim + tokn[n] > 0
      float x[kKeysN];
      bool up = false;
#pragma unroll
      for (int n = 0; n < kKeysN; ++n) {
        x[n] = (in_range && klim + tokn[n] > 0) ? __uint_as_float(sr[n]) * p.scale_log2
                                                : -CUDART_INF_F;
        mt[n] = fmaxf(mt[n], x[n]);
        up |= x[n] > m_run[n] + kKeysMargin;  // also m_run = -inf and x finite
      }
      // does any score of the stage pass its row's maximum in use by the
      // margin?  (And this warp's bulk copies of the last item's outputs
      // have read the output tile, which any warp may write again once all
      // are past this vote.)
      if (lane == 0) bulk_wait_read();
      const float *vote = exchange(lane == 0, 0, __any_sync(0xffffffffu, up) ? 1.f : 0.f);
      if (!ok) break;
      if ((vote[0] + vote[32]) + (vote[64] + vote[96]) > 0.f) {
        // every row's maximum over the stage, from all four warps
        const float wm = warp_rows_reduce<true>(x, lane);
        const float *sm = exchange((lane & 1) == 0, lane >> 1, wm);
        if (!ok) break;
        float alpha[kKeysN];
#pragma unroll
        for (int n = 0; n < kKeysN; ++n) {
          const float mn = fmaxf(m_run[n], fmaxf(fmaxf(sm[n], sm[32 + n]), fmaxf(sm[64 + n], sm[96 + n])));
          alpha[n] = mn == -CUDART_INF_F ? 1.f : exp2f(m_run[n] - mn);  // 0 when m_run = -inf
          m_run[n] = mn;
          l[n] *= alpha[n];
        }
        if (!(h.flags & kStageFirst)) {
          // O^T's row t, once the PV of the stage before has completed (its
          // commit released that stage's V slot)
          const int ip = i - 1;
          const bool w = mbar_wait(emptyv0 + 8 * (ip % NV), (ip / NV) & 1, limit, flags);
          ok = __all_sync(0xffffffffu, w);
          if (!ok) break;
          tc_fence_after();
          uint32_t o[kKeysN];
          tmem_ld16(tmem_o + lane_off, o);
          tmem_ld_wait16(o);
#pragma unroll
          for (int n = 0; n < kKeysN; ++n) o[n] = __float_as_uint(__uint_as_float(o[n]) * alpha[n]);
          tmem_st16(tmem_o + lane_off, o);
          tmem_st_wait();
        }
      }
      // P^T rounded to the input type into buffer i & 1, which the PV of
      // stage i - 2 read; the row sums add the fp32 exponentials.  Key t is
      // column t of P^T: panel t / 64, 2 bytes at (t % 64) * 2 of each
      // row's 128 bytes, 128-byte swizzle.
      if (i >= 2) {
        const int ip = i - 2;
        const bool w = mbar_wait(emptyv0 + 8 * (ip % NV), (ip / NV) & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
      }
      {
        uint8_t *pt = pbuf + (i & 1) * kKeysPTile + (t >> 6) * kKeysTilePanel + (t & 7) * 2;
        const int pc = (t & 63) >> 3;
#pragma unroll
        for (int n = 0; n < kKeysN; ++n) {
          const float mb = m_run[n] == -CUDART_INF_F ? 0.f : m_run[n];
          const float pr = ex2(x[n] - mb);
          l[n] += pr;
          *reinterpret_cast<unsigned short *>(pt + (n >> 3) * 1024 + (n & 7) * 128 +
                                              ((pc ^ (n & 7)) << 4)) = to_bits16<T>(pr);
        }
      }
      // V rows past the range may hold stale or foreign bytes (0 x NaN would
      // reach O^T): zero them
      if (h.valid < kKeysStage) {
        const bool w = mbar_wait(fullv0 + 8 * sv, (i / NV) & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        uint8_t *vst = vring + (size_t)sv * kKeysSlot;
        constexpr int kChunks = D * (int)sizeof(T) / 16;  // 16-byte pieces of a key's row
        const int n = (kKeysStage - h.valid) * kChunks;
        for (int idx = t; idx < n; idx += 128) {
          const int row = h.valid + idx / kChunks;
          const int c = idx % kChunks;
          *reinterpret_cast<uint4 *>(vst + (row >> 3) * kKeysGroup + (c >> 3) * 1024 + (row & 7) * 128 +
                                     (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + 8 * (i & 1));
      if (h.flags & kStageLast) {
        {
          const bool w = mbar_wait(o_done, items & 1, limit, flags);
          ok = __all_sync(0xffffffffu, w);
          if (!ok) break;
        }
        ++items;
        tc_fence_after();
        uint32_t o[kKeysN];
        tmem_ld16(tmem_o + lane_off, o);
        tmem_ld_wait16(o);
        tc_fence_before();
        // O^T's row t into the output tile as [row n][d] fp32 (free: every
        // warp waited for its bulk copies to read it before the last vote)
        float *ob = obuf;
#pragma unroll
        for (int n = 0; n < kKeysN; ++n) ob[n * D + t] = __uint_as_float(o[n]);
        // each row's sum (lanes 2c: row c) and true maximum (lanes 2c + 1)
        // over the 128 keys' threads; the exchange also completes the tile
        const float ws = warp_rows_reduce<false>(l, lane);
        const float wx = warp_rows_reduce<true>(mt, lane);
        const float *rs = exchange(true, (lane & 1) ? kKeysN + (lane >> 1) : (lane >> 1),
                                   (lane & 1) ? wx : ws);
        if (!ok) break;
        // warp w normalises rows w, w + 4, ... in place (lane l: columns
        // 4l .. 4l + 3; as the input type in the first half of the row for
        // the final output) and copies them out
        void *dst[kKeysN / 4];  // the rows' destinations, null past the item's rows
#pragma unroll
        for (int k = 0; k < kKeysN / 4; ++k) dst[k] = nullptr;
#pragma unroll
        for (int k = 0; k < kKeysN / 4; ++k) {
          const int n = warp + 4 * k;
          if (n >= h.rows) break;
          const float lsum = (rs[n] + rs[32 + n]) + (rs[64 + n] + rs[96 + n]);
          const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
          const int tk = n / G;
          const size_t orow =
              (size_t)(h.row0 + tk) * p.num_heads + (size_t)(h.kvh * G + n - tk * G);
          float4 *row = reinterpret_cast<float4 *>(ob + n * D);
          float4 v = row[lane];
          v.x *= inv;
          v.y *= inv;
          v.z *= inv;
          v.w *= inv;
          __syncwarp();
          if (p.write_partials) {
            row[lane] = v;
            dst[k] = p.tmp_out + (orow * p.max_parts + h.part) * D;
            if (lane == 0) {  // the row's record: relative to its true maximum
              float mr = 0.f;
#pragma unroll
              for (int q = 0; q < kKeysN; ++q) mr = q == n ? m_run[q] : mr;
              const float mx = fmaxf(fmaxf(rs[kKeysN + n], rs[32 + kKeysN + n]),
                                     fmaxf(rs[64 + kKeysN + n], rs[96 + kKeysN + n]));
              const size_t prow = orow * p.max_parts + h.part;
              p.max_logits[prow] = mx * 0.69314718055994530942f;  // natural-log units
              p.exp_sums[prow] = mx == -CUDART_INF_F ? 0.f : lsum * exp2f(mr - mx);
            }
          } else {
            uint2 w;
            w.x = MmaOp<T>::pack(v.x, v.y);
            w.y = MmaOp<T>::pack(v.z, v.w);
            reinterpret_cast<uint2 *>(row)[lane] = w;
            dst[k] = static_cast<T *>(p.out) + orow * D;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const uint32_t rbytes = p.write_partials ? D * 4u : D * (uint32_t)sizeof(T);
#pragma unroll
          for (int k = 0; k < kKeysN / 4; ++k)
            if (dst[k]) bulk_store(dst[k], smem_u32(ob + (warp + 4 * k) * D), rbytes);
          bulk_commit();
        }
      }
    }
    // the outputs are written before the CTA retires
    if (lane == 0) bulk_wait_all();
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    pdl_launch_dependents();
  }

  // every role is done with the tensor memory: free it
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kKeysTmemCols);
  }
  if (!p.sched_reset_later) {
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(p.sched, 0);
        atomicExch(p.sched + 1, 0);
      }
    }
  }
}

size_t umma_keys_smem_bytes() {
  return (size_t)(kKeysKSlots + kKeysVSlots) * kKeysSlot + 2 * (size_t)kKeysTile +
         2 * (size_t)kKeysPTile + kKeysOTile + kKeysKSlots * sizeof(KeysStage) +
         2 * 4 * 32 * sizeof(float) + (2 * kKeysKSlots + 2 * kKeysVSlots + 12) * 8 +
         8 * 4;  // flags, tensor-memory address
}

AttnKernelInfo attn_kernel_umma_keys(int dtype_bf16) {
  AttnKernelInfo k{};
  k.fn = dtype_bf16 ? reinterpret_cast<const void *>(&pa_umma_keys_kernel<__nv_bfloat16>)
                    : reinterpret_cast<const void *>(&pa_umma_keys_kernel<__half>);
  k.consumer_warps = 5;  // 4 softmax warps and the MMA warp; the producer is the sixth
  k.stage_tokens = kKeysStage;
  k.max_group = kKeysN;
  k.umma = 2;
  return k;
}

}  // namespace pa
