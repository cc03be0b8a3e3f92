// Query chunks on the 5th-generation tensor cores (tcgen05, sm_103a): items
// of 128 (token, head) rows, D = 128, 16-bit inputs.
//
// S = Q.K^T and O += P.V are each a few tcgen05.mma instructions issued by one
// thread, operands in shared memory (128-byte swizzle, as TMA lands them), the
// fp32 accumulators in tensor memory:
//   S[128 rows][64 keys]  = Q[128][D] . K^T          (K-major A and B)
//   O[128 rows][D]       += P[128][64 keys] . V[64][D] (P K-major, V MN-major)
// Four softmax warps own one row each per thread (tensor-memory lane = row):
// a row's maximum and sum need no shuffles.  P is written, rounded to the
// input type, over the stage's K bytes (dead once S is computed), so a stage
// is only its K and V.  The running maximum is raised lazily: O is rescaled
// only when a stage's maximum exceeds the one in use by more than 2^8 in the
// exponent's units, which is exact (the final normaliser uses the same
// reference) and leaves the rescale out of almost every stage.
//
// Warps: 0-3 softmax and output, 4 producer (TMA of K/V pages, work items),
// 5 MMA issuer (and the tensor-memory allocation).  Every wait is bounded.
#include <type_traits>

#include "pa_attn.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kUmmaRows = 128;        // rows of an item: the MMA's M
constexpr int kUmmaKeys = 64;         // keys of a stage: the S MMA's N
constexpr int kUmmaD = 128;           // head size
constexpr int kUmmaTmemCols = 256;    // S at columns 0 and 64 (two buffers), O at 128
// K and V of a stage live in separate rings: three K slots (a stage's P is
// written over its K, so a K slot is busy until the stage's PV), two V slots.
// K of stage i + 1 then loads while stage i - 1's PV runs.
constexpr int kUmmaKSlots = 3;
constexpr int kUmmaVSlots = 2;
// A K (or V) slot holds 64 keys as [8-key group][panel][8 keys][128 B]: each
// 8-row piece of a panel is one 1024-byte swizzle atom, a group is kUmmaGroup
// bytes (every panel), and a page's rows arrive in one 4-D copy.
constexpr int kUmmaGroup = (kUmmaD * 2 / 128) * 1024;
constexpr int kUmmaHalf = (kUmmaKeys / 8) * kUmmaGroup;  // K (or V) bytes of a stage
constexpr int kUmmaQPanel = kUmmaRows * 128;
constexpr int kUmmaQBytes = (kUmmaD * 2 / 128) * kUmmaQPanel;
constexpr float kLazyMargin = 8.f;    // log2 units
constexpr int kMailSlots = 8;         // cluster: items the leader may run ahead of the others

struct UmmaStage {
  int row0, kvh, part;  // the item: first query row, KV head, partition
  int tok0;             // key of the stage's first row
  int valid;            // keys of the stage in the item's range
  int flags;            // kStage*
  int rows;             // (token, head) rows of the item
  int lim_base;         // the item's first token sees keys below lim_base + 1
};

// ---- thread-block clusters: the CTAs of a cluster take the row groups of
// the same keys, each issuing a share of every stage's copies into all of them
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// the same shared-memory offset in the CTA of the given rank
__device__ __forceinline__ uint32_t cluster_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// every thread of every CTA of the cluster
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// one arrival, with release at cluster scope, on an mbarrier of another CTA
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// a bounded wait that also acquires what other CTAs of the cluster released
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int *abort) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_cluster(bar, parity)) return true;
    if (abort && *abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
// a 4-D copy landing at the same offset in every CTA of `mask`, each CTA's
// mbarrier (same offset) counting the bytes it receives
__device__ __forceinline__ void tma_load_4d_multicast(uint32_t dst, const CUtensorMap *map, int x,
                                                      int y, int z, int w, uint32_t bar,
                                                      uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "h"(mask)
      : "memory");
}
// one arrival on the mbarrier at this offset in every CTA of `mask` once
// this thread's earlier tcgen05 operations have completed
__device__ __forceinline__ void tc_commit_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

}  // namespace

// CLUSTERED: launched in thread-block clusters of p.cluster CTAs (else the
// cluster code compiles away).  Two CTAs an SM: at most 168 registers a thread.
template <typename T, bool CLUSTERED>
__global__ void __launch_bounds__(192, 2)
    pa_umma_chunk_kernel(const __grid_constant__ AttnParams p,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int D = kUmmaD;
  constexpr int NK = kUmmaKSlots, NV = kUmmaVSlots;
  constexpr int NPANELS = D * (int)sizeof(T) / 128;
  constexpr uint32_t kIdescS = instr_desc<T>(kUmmaRows, kUmmaKeys, false);
  constexpr uint32_t kIdescPV = instr_desc<T>(kUmmaRows, D, true);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The 128-byte swizzle needs every tile 1024-byte aligned.  Two CTAs of
  // this kernel fit on an SM only without alignment slack, so the kernel
  // relies on the dynamic shared memory starting 1024-byte aligned (it
  // starts right after the 1 KB the system reserves) and checks it.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const bool misaligned = (smem_u32(smem_raw) & 1023u) != 0;
  // CL CTAs a cluster (p.cluster, 1 = none): rank r takes row group
  // g * CL + r of each cluster item g, the leader (rank 0) takes the items
  // from the work counter and hands them on
  const int CL = CLUSTERED && p.cluster > 1 ? p.cluster : 1;
  const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
  const uint16_t all_ctas = (uint16_t)((1u << CL) - 1u);
  if (misaligned) {
    if (threadIdx.x == 0) report(p.status, kStatusBadInput);
    if (CL > 1) {  // every CTA of the cluster meets both cluster barriers
      cluster_sync();
      cluster_sync();
    }
    return;
  }
  uint8_t *kring = smem_raw;                             // NK x K: [panel][64 keys][128 B]
  uint8_t *vring = kring + NK * kUmmaHalf;               // NV x V, the same layout
  uint8_t *qbuf = vring + NV * kUmmaHalf;                // [panel][128 rows][128 B]
  UmmaStage *info = reinterpret_cast<UmmaStage *>(qbuf + kUmmaQBytes);  // per K slot
  uint64_t *bars = reinterpret_cast<uint64_t *>(info + NK);
  // fullK[NK], emptyK[NK], fullV[NV], emptyV[NV], q_full, s_full[2], p_full[2],
  // o_done, drain, never.  S and P barriers come in pairs (stage parity): the
  // softmax may run one stage ahead of the MMA thread's wait for its P (the
  // next S is issued before this PV), and one barrier for every stage would
  // then complete twice before that wait and never show the awaited phase.
  // then mail[kMailSlots]: the leader's hand-over of each next item
  constexpr int NBARS = 2 * NK + 2 * NV + 8 + kMailSlots;
  volatile int *flags = reinterpret_cast<volatile int *>(bars + NBARS);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBARS) + 4;
  volatile int *mailbox = reinterpret_cast<volatile int *>(bars + NBARS) + 8;  // kMailSlots items
  const uint32_t kring_u32 = smem_u32(kring), vring_u32 = smem_u32(vring), q_u32 = smem_u32(qbuf);
  const uint32_t fullk0 = smem_u32(bars), emptyk0 = fullk0 + 8 * NK;
  const uint32_t fullv0 = emptyk0 + 8 * NK, emptyv0 = fullv0 + 8 * NV;
  const uint32_t q_full = emptyv0 + 8 * NV, s_full = q_full + 8, p_full = s_full + 16,
                 o_done = p_full + 16, drain = o_done + 8, never = drain + 8, mail0 = never + 8;
  const uint64_t limit = p.wait_limit_ns;

  if (threadIdx.x == 0) {
    // a slot is free once the PV of every CTA of the cluster has read it
    for (int i = 0; i < NK; ++i) {
      mbar_init(fullk0 + 8 * i, 1);
      mbar_init(emptyk0 + 8 * i, CL);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(fullv0 + 8 * i, 1);
      mbar_init(emptyv0 + 8 * i, CL);
    }
    for (int i = 0; i < kMailSlots; ++i) mbar_init(mail0 + 8 * i, 1);
    mbar_init(q_full, 4);
    mbar_init(s_full, 1);
    mbar_init(s_full + 8, 1);
    mbar_init(p_full, 4);
    mbar_init(p_full + 8, 4);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    flags[0] = 0;
    fence_mbar_init();
  }
  // every CTA's barriers are initialised before any CTA of the cluster
  // touches another's
  if (CL > 1) cluster_sync();
  // Launched with programmatic dependent launch: wait for the previous kernel
  // in the stream before the tensor memory is taken, so that a CTA started
  // early never holds columns that a still-running CTA of an earlier launch
  // of this kernel on the same SM is waiting for.
  pdl_wait_primary();
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kUmmaTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem, tmem_o = tmem + 128;

  if (warp == 4) {
    // ======================= producer warp =======================
    if (lane == 0) {
      prefetch_tmap(&tmap_k);
      prefetch_tmap(&tmap_v);
    }
    const int U = p.unit_rows;
    const int G = p.group;
    int cs = 0, cbase = 0, c_cnt = 0, c_incl = 0, c_L = 0, c_total = 0, c_qs = 0, c_n = 0,
        c_nrg = 0;
    bool c_loaded = false;
    // the running count of items per sequence, 32 sequences at a time:
    // items are (KV head, partition, group of CL row groups) of each sequence
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
        c_qs = __ldg(p.q_start + sl);
        const int qe = __ldg(p.q_start + sl + 1);
        c_n = qe - c_qs;
        if (c_qs < 0 || c_n < 0 || c_n > c_L || qe > p.num_rows) {
          report(p.status, kStatusBadInput);  // its rows get no items
          c_n = 0;
        }
      }
      const int c_np = (c_L + p.range_tokens - 1) / p.range_tokens;
      c_nrg = (c_n + p.chunk_tokens - 1) / p.chunk_tokens;  // row groups
      c_cnt = sl < p.num_seqs ? p.num_kv_heads * c_np * ((c_nrg + CL - 1) / CL) : 0;
      c_incl = c_cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, c_incl, off);
        if (lane >= off) c_incl += t;
      }
      c_total = __shfl_sync(0xffffffffu, c_incl, 31);
      c_loaded = true;
    };
    // The leader of a cluster takes the next item from the counter and mails
    // it to the others (a store into their mailbox slot, then a release
    // arrival on the slot's mbarrier); they wait for it, bounded.  The leader
    // runs at most a few items ahead (the stage slots are freed only by every
    // CTA), well within kMailSlots.
    bool ok = true;
    auto grab_issue = [&]() -> int { return rank == 0 ? atomic_add_lane0(p.sched, lane) : 0; };
    const int takers = (int)gridDim.x / CL;
    int ordinal = 0;  // items handed over so far
    auto next_item = [&](int raw) -> int {
      if (CL == 1) return takers + __shfl_sync(0xffffffffu, raw, 0);
      // hand-over k (from 0) uses slot k % kMailSlots, the (k / kMailSlots)-th
      // time: its phase parity
      const int e = ordinal % kMailSlots;
      const uint32_t par = (uint32_t)(ordinal / kMailSlots) & 1u;
      ++ordinal;
      int nx = 0;
      if (rank == 0) {
        nx = takers + __shfl_sync(0xffffffffu, raw, 0);
        if (lane > 0 && lane < CL) {
          st_cluster(cluster_addr(smem_u32(const_cast<int *>(mailbox) + e), (uint32_t)lane), nx);
          mbar_arrive_remote(cluster_addr(mail0 + 8 * e, (uint32_t)lane));
        }
        __syncwarp();
      } else {
        bool w = true;
        if (lane == 0) w = mbar_wait_cluster(mail0 + 8 * e, par, limit, flags);
        ok = __shfl_sync(0xffffffffu, w, 0);
        nx = ok ? mailbox[e] : -1;
        nx = __shfl_sync(0xffffffffu, nx, 0);
      }
      return nx;
    };
    int item = (int)blockIdx.x / CL;  // a cluster's first item: its index
    int i = 0;           // stages issued
    int ik = 0, iv = 0;  // stages whose K (with the end marker) and V copies are issued
    while (true) {
      int s = 0, kvh = 0, part = 0, L = 0, nrg = 0, qs = 0, n_s = 0, rg = 0, gr = 0;
      bool found = false;
      if (item < 0) {
        if (lane == 0 && ok) report(p.status, kStatusBadInput);
      } else {
        while (true) {
          if (!c_loaded) load_chunk();
          if (item < cbase + c_total) {
            const unsigned hit = __ballot_sync(0xffffffffu, cbase + c_incl > item);
            const int ls = __ffs(hit) - 1;
            s = cs + ls;
            L = __shfl_sync(0xffffffffu, c_L, ls);
            nrg = __shfl_sync(0xffffffffu, c_nrg, ls);
            qs = __shfl_sync(0xffffffffu, c_qs, ls);
            n_s = __shfl_sync(0xffffffffu, c_n, ls);
            const int first = cbase + __shfl_sync(0xffffffffu, c_incl - c_cnt, ls);
            const int np_s = (L + p.range_tokens - 1) / p.range_tokens;
            const int ngr = (nrg + CL - 1) / CL;  // groups of CL row groups
            const int per_head = np_s * ngr;
            kvh = (item - first) / per_head;
            const int rem = (item - first) % per_head;
            part = rem / ngr;
            gr = rem % ngr;
            rg = gr * CL + (int)rank;  // this CTA's row group (maybe past the chunk)
            found = s < p.num_seqs;
            break;
          }
          if (cs + 32 >= p.num_seqs) break;
          cs += 32;
          cbase += c_total;
          c_loaded = false;
        }
      }
      if (!found) break;
      int next_raw = 0;
      const int t_first = rg * p.chunk_tokens;
      const int ntok = max(0, min(p.chunk_tokens, n_s - t_first));  // 0: no rows here
      const int lim_base = L - n_s + t_first;
      const int row0 = qs + t_first;
      const int tok_begin = part * p.range_tokens;
      // the cluster's keys: up to the limit of its last row group's last token
      const int lim_cluster = L - n_s + min(n_s, (gr * CL + CL) * p.chunk_tokens);
      const int tok_end = min(min(tok_begin + p.range_tokens, L), lim_cluster);
      if (part == 0 && p.row_limit)
        for (int t = lane; t < ntok; t += 32) p.row_limit[row0 + t] = lim_base + t + 1;
      if (tok_end <= tok_begin) {  // the partition lies past every token of the group
        item = next_item(grab_issue());
        if (!ok) break;
        continue;
      }
      // a window of 64 block-table entries (lane j: pages win0 + j and
      // win0 + 32 + j), slid by 32 pages when a stage reaches the second half
      const int32_t *bt = p.block_tables + (size_t)s * p.max_blocks_per_seq;
      const int last_page = (tok_end - 1) >> p.log2_block_size;
      auto load_entry = [&](int page) -> int {
        return (page >= 0 && page <= last_page) ? __ldg(bt + page) : -1;
      };
      int win0 = tok_begin >> p.log2_block_size;
      int cur = load_entry(win0 + lane);
      int nxt = load_entry(win0 + 32 + lane);
      const int n_st = (tok_end - tok_begin + kUmmaKeys - 1) / kUmmaKeys;
      for (int j = 0; j < n_st; ++j) {
        const int sk = i % NK, sv = i % NV;
        if (i >= NK) {  // K slot: the PV of stage i - NK has read its K and P
          bool w = true;
          if (lane == 0) w = mbar_wait(emptyk0 + 8 * sk, ((i / NK) - 1) & 1, limit, flags);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
        }
        const int stage_tok0 = tok_begin + j * kUmmaKeys;
        const int valid = min(kUmmaKeys, tok_end - stage_tok0);
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
            y = (blk * p.num_kv_heads + kvh) * p.block_size + (tok & (p.block_size - 1));
        }
        const unsigned valid_mask = __ballot_sync(0xffffffffu, y >= 0);
        if (lane == 0) {
          UmmaStage &h = info[sk];
          h.row0 = row0;
          h.kvh = kvh;
          h.part = part;
          h.tok0 = stage_tok0;
          h.valid = valid;
          h.flags = (j == 0 ? kStageFirst : 0) | (j == n_st - 1 ? kStageLast : 0);
          h.rows = ntok * G;
          h.lim_base = lim_base;
          mbar_arrive_expect_tx(fullk0 + 8 * sk, (uint32_t)__popc(valid_mask) * U * 128u * NPANELS);
        }
        __syncwarp();
        // rows lane*U .. : groups lane*U/8 .. of the slot, every panel, one
        // copy; in a cluster each CTA issues the units lane = rank (mod CL),
        // multicast to every CTA (each counts all the stage's bytes)
        const bool mine = y >= 0 && (lane % CL) == (int)rank;
        if (mine) {
          const uint32_t kdst = kring_u32 + (uint32_t)sk * kUmmaHalf + (uint32_t)(lane * U / 8) * kUmmaGroup;
          if (CL > 1)
            tma_load_4d_multicast(kdst, &tmap_k, 0, 0, 0, y >> 3, fullk0 + 8 * sk, all_ctas);
          else
            tma_load_4d(kdst, &tmap_k, 0, 0, 0, y >> 3, fullk0 + 8 * sk);
        }
        ik = i + 1;
        if (i >= NV) {  // V slot: the PV of stage i - NV has read it
          bool w = true;
          if (lane == 0) w = mbar_wait(emptyv0 + 8 * sv, ((i / NV) - 1) & 1, limit, flags);
          ok = __shfl_sync(0xffffffffu, w, 0);
          if (!ok) break;
        }
        if (lane == 0)
          mbar_arrive_expect_tx(fullv0 + 8 * sv, (uint32_t)__popc(valid_mask) * U * 128u * NPANELS);
        __syncwarp();
        if (mine) {
          const uint32_t vdst = vring_u32 + (uint32_t)sv * kUmmaHalf + (uint32_t)(lane * U / 8) * kUmmaGroup;
          if (CL > 1)
            tma_load_4d_multicast(vdst, &tmap_v, 0, 0, 0, y >> 3, fullv0 + 8 * sv, all_ctas);
          else
            tma_load_4d(vdst, &tmap_v, 0, 0, 0, y >> 3, fullv0 + 8 * sv);
        }
        iv = i + 1;
        if (j == 0) next_raw = grab_issue();
        ++i;
        const int next_rel = ((stage_tok0 + kUmmaKeys) >> p.log2_block_size) - win0;
        if (next_rel >= 32) {
          cur = nxt;
          win0 += 32;
          nxt = load_entry(win0 + 32 + lane);
        }
      }
      if (!ok) break;
      item = next_item(next_raw);
      if (!ok) break;
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
    }
    __syncwarp();
  } else if (warp == 5) {
    // ======================= MMA warp (one thread issues) =======================
    if (lane == 0) {
      bool ok = true;
      int items = 0;
      // S = Q K^T of the stage in K slot `sk` into S buffer b: D / 16
      // k-steps; a k-step is 32 bytes inside a 128-byte panel of Q (128 rows,
      // 8-row atoms 1024 bytes apart, panels 16 KB apart) and of K (8-key
      // groups kUmmaGroup bytes apart, panels 1024 bytes apart)
      auto issue_s = [&](int sk, int b) {
        const uint32_t kst = kring_u32 + (uint32_t)sk * kUmmaHalf;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t koff = (uint32_t)(ks & 3) * 32u;
          const uint64_t da = smem_desc(q_u32 + (uint32_t)(ks >> 2) * kUmmaQPanel + koff, 16, 1024);
          const uint64_t db = smem_desc(kst + (uint32_t)(ks >> 2) * 1024u + koff, 16, kUmmaGroup);
          tc_mma(tmem_s + 64u * (uint32_t)b, da, db, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc_commit(s_full + 8u * (uint32_t)b);
      };
      // The S of stage i + 1 is issued before the PV of stage i (its buffer
      // was read by the softmax of stage i - 1, whose P the PV of i - 1
      // waited for), so the tensor cores compute it while the softmax warps
      // work on stage i; within an item only, since a new item's S needs its
      // queries, which the softmax warps store after the item before ends.
      UmmaStage h{};
      ok = mbar_wait(fullk0, 0, limit, flags);
      if (ok) h = info[0];
      bool more = ok && !(h.flags & kStageEnd);
      if (more) {
        ok = mbar_wait(q_full, 0, limit, flags);
        items = 1;
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
        }
        more = ok;
      }
      for (int i = 0; more; ++i) {
        const int sk = i % NK, sv = i % NV, sk1 = (i + 1) % NK;
        const uint32_t par1 = ((i + 1) / NK) & 1;
        // the next stage's S goes first only if its bytes are already here:
        // the PV of this stage never waits for the next stage's copies
        bool s1 = false;
        UmmaStage h1{};
        if (mbar_test(fullk0 + 8 * sk1, par1)) {
          h1 = info[sk1];
          if (!(h1.flags & (kStageEnd | kStageFirst))) {
            tc_fence_after();
            issue_s(sk1, (i + 1) & 1);
            s1 = true;
          }
        }
        ok = mbar_wait(p_full + 8 * (i & 1), (i >> 1) & 1, limit, flags);
        if (!ok) break;
        ok = mbar_wait(fullv0 + 8 * sv, (i / NV) & 1, limit, flags);  // the stage's V is in
        if (!ok) break;
        tc_fence_after();
        // O += P V: 4 k-steps of 16 keys; P [128 rows][64 keys] over the K
        // bytes (8 rows a 1024-byte atom), V MN-major: 64 columns a panel
        // 1024 bytes apart (LBO), 8 keys a group kUmmaGroup bytes apart (SBO)
        const uint32_t kst = kring_u32 + (uint32_t)sk * kUmmaHalf;
        const uint32_t vst = vring_u32 + (uint32_t)sv * kUmmaHalf;
#pragma unroll
        for (int kk = 0; kk < kUmmaKeys / 16; ++kk) {
          const uint64_t da = smem_desc(kst + (uint32_t)kk * 32u, 16, 1024);
          const uint64_t db = smem_desc(vst + (uint32_t)kk * 2u * kUmmaGroup, 1024, kUmmaGroup);
          tc_mma(tmem_o, da, db, kIdescPV, ((h.flags & kStageFirst) && kk == 0) ? 0u : 1u);
        }
        if (CL > 1) {  // every CTA's slot counts this CTA's release
          tc_commit_multicast(emptyk0 + 8 * sk, all_ctas);  // the stage's K and P are read
          tc_commit_multicast(emptyv0 + 8 * sv, all_ctas);  // and its V
        } else {
          tc_commit(emptyk0 + 8 * sk);
          tc_commit(emptyv0 + 8 * sv);
        }
        if (h.flags & kStageLast) tc_commit(o_done);
        if (!s1) {
          ok = mbar_wait(fullk0 + 8 * sk1, par1, limit, flags);
          if (!ok) break;
          h1 = info[sk1];
          if (h1.flags & kStageEnd) break;
          if (h1.flags & kStageFirst) {
            ok = mbar_wait(q_full, items & 1, limit, flags);
            if (!ok) break;
            ++items;
          }
          tc_fence_after();
          issue_s(sk1, (i + 1) & 1);
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
    // ======================= softmax warps: thread = row =======================
    const int r = threadIdx.x;  // 0..127: the row, and its tensor-memory lane
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int G = p.group;
    float m_run = -CUDART_INF_F, m_true = -CUDART_INF_F, l = 0.f;
    int lim = 0;
    bool ok = true;
    int items = 0;
    if (p.debug_flags & kDebugStallConsumers) {
      // Wait on a barrier that nothing releases: the bound must end it.
      ok = mbar_wait(never, 0, limit, flags);
      ok = __all_sync(0xffffffffu, ok);
    }
    for (int i = 0; ok; ++i) {
      const int sk = i % NK, sv = i % NV;
      const bool w = mbar_wait(fullk0 + 8 * sk, (i / NK) & 1, limit, flags);
      ok = __all_sync(0xffffffffu, w);
      if (!ok) break;
      const UmmaStage h = info[sk];
      if (h.flags & kStageEnd) break;
      uint8_t *kst = kring + (size_t)sk * kUmmaHalf;
      uint8_t *vst = vring + (size_t)sv * kUmmaHalf;
      const int orow_tok = r / G, orow_head = h.kvh * G + r % G;
      if (h.flags & kStageFirst) {
        // this row's query into the swizzled Q tile (zeros past the item's rows)
        const bool live = r < h.rows;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const T *>(p.query) +
            ((size_t)(h.row0 + (live ? orow_tok : 0)) * p.num_heads + orow_head) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = live ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
          const int pn = c >> 3, cc = c & 7;
          *reinterpret_cast<uint4 *>(qbuf + pn * kUmmaQPanel + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
        }
        lim = live ? h.lim_base + orow_tok + 1 : 0;
        m_run = -CUDART_INF_F;
        m_true = -CUDART_INF_F;
        l = 0.f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      // Every warp waits for the stage's S: S(i) is issued only after the P of
      // stage i - 2 was taken, so no warp's P-ready arrival can land in the
      // phase of another stage.
      {
        const bool w2 = mbar_wait(s_full + 8 * (i & 1), (i >> 1) & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w2);
        if (!ok) break;
      }
      // A warp whose 32 rows are all past the item's rows skips its scores,
      // softmax and P: its rows of P hold stale bytes, which reach only
      // those rows of O (each row of O depends on its own row of P alone),
      // and they are never written out.
      const bool warp_live = 32 * warp < h.rows;
      if (!warp_live) {
        // only its share of zeroing the V rows past the range (below), and
        // the P-ready arrival
        if (h.valid < kUmmaKeys) {
          {  // the stage's V must have landed
            const bool w5 = mbar_wait(fullv0 + 8 * sv, (i / NV) & 1, limit, flags);
            ok = __all_sync(0xffffffffu, w5);
            if (!ok) break;
          }
          const int n = (kUmmaKeys - h.valid) * (D * (int)sizeof(T) / 16);
          for (int idx = r; idx < n; idx += 128) {
            const int row = h.valid + idx / (D * (int)sizeof(T) / 16);
            const int c = idx % (D * (int)sizeof(T) / 16);
            *reinterpret_cast<uint4 *>(vst + (row >> 3) * kUmmaGroup + (c >> 3) * 1024 + (row & 7) * 128 +
                                       (((c & 7) ^ (row & 7)) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full + 8 * (i & 1));
        if (h.flags & kStageLast) ++items;  // this warp has no rows to write
        continue;
      }
      tc_fence_after();
      uint32_t sa[32], sb[32];
      const uint32_t sbuf = tmem_s + 64u * (uint32_t)(i & 1) + lane_off;
      tmem_ld32(sbuf, sa);
      tmem_ld32(sbuf + 32, sb);
      tmem_ld_wait(sa);
      tmem_ld_wait(sb);
      // scores in log2 units; keys past the range or this row's limit
      // (key index kvis and up) get -inf, a step every row of the warp skips
      // when all of them see the whole stage
      float x[64];
  #pragma unroll
      for (int k = 0; k < 64; ++k) x[k] = __uint_as_float(k < 32 ? sa[k] : sb[k - 32]) * p.scale_log2;
      const int kvis = min(h.valid, lim - h.tok0);
      if (!__all_sync(0xffffffffu, kvis >= kUmmaKeys)) {
  #pragma unroll
        for (int k = 0; k < 64; ++k)
          if (k >= kvis) x[k] = -CUDART_INF_F;
      }
      // the row maximum: 8 chains of three-input maxima over 8 keys each
      float m8[8];
  #pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float *v = x + 8 * j;
        m8[j] = fmax3(fmax3(v[0], v[1], v[2]), fmax3(v[3], v[4], v[5]), fmaxf(v[6], v[7]));
      }
      const float mt = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]),
                             fmaxf(m8[6], m8[7]));
      m_true = fmaxf(m_true, mt);
      const bool raise = mt > m_run + kLazyMargin;  // also m_run = -inf and mt finite
      const float alpha = raise ? exp2f(m_run - mt) : 1.f;  // 0 when m_run = -inf
      if (raise) m_run = mt;
      if (!(h.flags & kStageFirst) && __any_sync(0xffffffffu, raise)) {
        // rescale this row's O (every lane takes part in the warp's loads),
        // once the PV of the stage before has completed: its commit
        // released that stage's slot
        {
          const int ip = i - 1;
          const bool w4 = mbar_wait(emptyv0 + 8 * (ip % NV), (ip / NV) & 1, limit, flags);
          ok = __all_sync(0xffffffffu, w4);
          if (!ok) break;
        }
        tc_fence_after();
  #pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem_o + lane_off + 32 * c, o);
          tmem_ld_wait(o);
  #pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(tmem_o + lane_off + 32 * c, o);
        }
        tmem_st_wait();
      }
      l *= alpha;
      const float mb = m_run == -CUDART_INF_F ? 0.f : m_run;
      // P rounded to the input type for the PV product; the row sum adds the
      // fp32 exponentials (four partial sums), so that no rounded pair needs
      // unpacking: the two differ by the rounding of P, about 2^-9 relative
      // and unbiased.  Row r of P [128][64 keys] over the stage's K bytes,
      // 128-byte swizzle.
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w4[4];
  #pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(x[8 * c + 2 * e] - mb), p1 = ex2(x[8 * c + 2 * e + 1] - mb);
          l4[e] += p0 + p1;
          w4[e] = MmaOp<T>::pack(p0, p1);
        }
        *reinterpret_cast<uint4 *>(kst + r * 128 + ((c ^ (r & 7)) << 4)) =
            make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      // V rows past the range may hold stale or foreign bytes (0 x NaN would
      // reach O): zero them
      if (h.valid < kUmmaKeys) {
        {  // the stage's V must have landed
          const bool w5 = mbar_wait(fullv0 + 8 * sv, (i / NV) & 1, limit, flags);
          ok = __all_sync(0xffffffffu, w5);
          if (!ok) break;
        }
        const int n = (kUmmaKeys - h.valid) * (D * (int)sizeof(T) / 16);
        for (int idx = r; idx < n; idx += 128) {
          const int row = h.valid + idx / (D * (int)sizeof(T) / 16);
          const int c = idx % (D * (int)sizeof(T) / 16);
          *reinterpret_cast<uint4 *>(vst + (row >> 3) * kUmmaGroup + (c >> 3) * 1024 + (row & 7) * 128 +
                                     (((c & 7) ^ (row & 7)) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full + 8 * (i & 1));
      if (h.flags & kStageLast) {
        const bool w3 = mbar_wait(o_done, items & 1, limit, flags);
        ok = __all_sync(0xffffffffu, w3);
        if (!ok) break;
        ++items;
        tc_fence_after();
        // O is relative to m_run; the record takes the true maximum
        const float lt = m_true == -CUDART_INF_F ? 0.f : l * exp2f(m_run - m_true);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool live = r < h.rows;
        const size_t orow = ((size_t)h.row0 + orow_tok) * p.num_heads + orow_head;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem_o + lane_off + 32 * c, o);
          tmem_ld_wait(o);
          if (!live) continue;
          if (p.write_partials) {
            float *dst = p.tmp_out + (orow * p.max_parts + h.part) * D + 32 * c;
#pragma unroll
            for (int k = 0; k < 32; k += 4)
              *reinterpret_cast<float4 *>(dst + k) =
                  make_float4(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv,
                              __uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
          } else {
            T *dst = static_cast<T *>(p.out) + orow * D + 32 * c;
#pragma unroll
            for (int k = 0; k < 32; k += 8) {
              uint4 v;
              v.x = MmaOp<T>::pack(__uint_as_float(o[k]) * inv, __uint_as_float(o[k + 1]) * inv);
              v.y = MmaOp<T>::pack(__uint_as_float(o[k + 2]) * inv, __uint_as_float(o[k + 3]) * inv);
              v.z = MmaOp<T>::pack(__uint_as_float(o[k + 4]) * inv, __uint_as_float(o[k + 5]) * inv);
              v.w = MmaOp<T>::pack(__uint_as_float(o[k + 6]) * inv, __uint_as_float(o[k + 7]) * inv);
              *reinterpret_cast<uint4 *>(dst + k) = v;
            }
          }
        }
        if (live && p.write_partials) {
          const size_t prow = orow * p.max_parts + h.part;
          p.max_logits[prow] = m_true * 0.69314718055994530942f;  // natural-log units
          p.exp_sums[prow] = lt;
        }
        tc_fence_before();
      }
    }
    if (!ok && lane == 0) {
      report(p.status, kStatusTimeout);
      flags[0] = 1;
    }
    pdl_launch_dependents();
  }

  // every role is done with the tensor memory: free it.  In a cluster, no CTA
  // leaves while another may still copy into its shared memory or arrive on
  // its barriers.
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kUmmaTmemCols);
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

size_t umma_chunk_smem_bytes() {
  return (size_t)(kUmmaKSlots + kUmmaVSlots) * kUmmaHalf + kUmmaQBytes +
         kUmmaKSlots * sizeof(UmmaStage) +
         (2 * kUmmaKSlots + 2 * kUmmaVSlots + 8 + kMailSlots) * 8 +
         (8 + kMailSlots) * 4;  // flags, tensor-memory address, mailbox
}

AttnKernelInfo attn_kernel_umma_chunk(int dtype_bf16, bool clustered) {
  AttnKernelInfo k{};
  if (clustered)
    k.fn = dtype_bf16 ? reinterpret_cast<const void *>(&pa_umma_chunk_kernel<__nv_bfloat16, true>)
                      : reinterpret_cast<const void *>(&pa_umma_chunk_kernel<__half, true>);
  else
    k.fn = dtype_bf16 ? reinterpret_cast<const void *>(&pa_umma_chunk_kernel<__nv_bfloat16, false>)
                      : reinterpret_cast<const void *>(&pa_umma_chunk_kernel<__half, false>);
  k.consumer_warps = 5;  // 4 softmax warps and the MMA warp; the producer is the sixth
  k.stage_tokens = kUmmaKeys;
  k.max_group = kUmmaRows;
  k.umma = 1;
  return k;
}

}  // namespace pa
