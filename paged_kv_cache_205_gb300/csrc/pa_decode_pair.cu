// pa_decode_pair.cu -- the two cluster kernels of the decode step of
// PagedAttention: one thread-block cluster per (sequence, kv head)
// (decode_pair_kernel, small batches) and one per sequence
// (decode_seq_kernel, batches of similar context lengths).  Both combine the
// pieces of a context inside the cluster, through distributed shared memory,
// instead of through partials in global memory and a merge kernel.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "What is in
// the box": one query token's attention over K/V stored in 16-token pages
// found through block_table, online softmax, GQA_Q_TO_K_RATIO = 4.
//
// decode_pair_kernel (GB300-first):
//  * One thread-block cluster of c CTAs (c = 1, 2, 4 or 8) per (sequence, kv
//    head).  The c CTAs cut the head's 16-token tiles into c equal ranges, so
//    a small batch still puts every SM to work, and they combine their
//    results through distributed shared memory: no split partials in global
//    memory, no merge kernel, no prefix over the batch, no work counter.
//  * A producer warp streams the range's tiles with TMA tensor copies, one
//    4 KiB copy (K and V of the head, 16 tokens) per tile, 8 tiles per 32 KiB
//    stage, 3 stages.  Eight consumer warps take one tile of each stage each
//    and keep their own online-softmax state (the 4 q heads of the group are
//    the M rows of m16n8k16 bf16 MMAs, as in the split-context kernel); at the
//    end the 8 warp states are combined in shared memory, then the c CTA
//    states in the cluster leader's shared memory (asynchronous stores that
//    complete the leader's barrier by their byte count).
//  * Before the dependency wait the CTA reads its sequence's context length
//    and first page ids as they are then and prefetches those tiles into L2.
//    Right after the wait the first stages are fetched from those ids while
//    the length and ids are read again; if either changed, the consumers drop
//    what they accumulated (a reset stage) and the range is streamed again
//    from the current values.  Nothing is written before that check.
//  * Packed plan (batches with two CTAs per pair on average, the c = 2
//    case): rather than 2 CTAs for every pair, a sequence gets 1, 2 or 4 CTAs
//    per kv head by its length (the longest the most, within the same total),
//    in clusters of 4, so that the longest heads' CTAs stream fewer tiles
//    (llama1b's contexts, 256 to 2048 tokens: 54 tiles at most instead of 64).
//    Every CTA's producer warp works the plan out from all the context lengths
//    before the dependency wait and again after it; if the plan moved, the
//    first stage streamed after the check carries the final role to the
//    consumers (who started on q of the planned one).
#include <cfloat>
#include <climits>
#include <cuda.h>

#include "pa_decode_tile.cuh"
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kPairWarps = 8;                              // consumer warps
constexpr int kPairThreads = (kPairWarps + 1) * 32;        // + producer warp
constexpr int kPairStages = 3;
constexpr int kPairCtasPerSm = 2;
constexpr int kSlotBytes = 2 * kBs * kHeadRowBytes;        // one tile of one head, K and V: 4 KiB
constexpr int kPairStageBytes = kPairWarps * kSlotBytes;   // 32 KiB
constexpr int kMaxCluster = 8;
constexpr int kIdBatch = 32;                               // page ids read at a time (4 stages)
constexpr int kPrefetchTiles = 24;                         // tiles prefetched before the wait
static_assert(kPrefetchTiles <= kIdBatch, "prefetched tiles come from the first id batch");
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kReset = 1;   // consumers drop their state before this stage
constexpr int kEnd = 2;     // no more tiles; the stage carries no data
constexpr int kMoved = 4;   // packed plan: the CTA's role changed after the wait (see role[])
constexpr int kIdle = 8;    // packed plan: the CTA has no part of it

struct PairStage {
  int j0;      // tile of slot 0
  int n;       // slots holding a tile (slot w: tile j0 + w)
  int last;    // the sequence's last tile
  int tail;    // tokens in it (1..16)
  int bad;     // bit w: slot w's page id was out of range (tile skipped); with 8-token
               // pages instead bit w / 8 + w: slot w's first / second page was loaded
  int flags;
};

struct __align__(1024) PairSmem {
  unsigned char kv[kPairStages][kPairStageBytes];
  float part_o[kMaxCluster][kGqa][kD];   // cluster leader: each CTA's unnormalised result
  float2 part_ml[kMaxCluster][kGqa];     // and its (m, l), m in the log2 domain
  // (part_o rows are 16-byte aligned: the stages before them are 1 KiB multiples)
  PairStage desc[kPairStages];
  int role[4];                           // packed plan: sequence (-1: idle), kv head, parts, part
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t parts_full;                   // cluster leader: every CTA's result has landed
};

struct PairParams {
  const unsigned char *kv;   // the pool (L2 prefetches; copies go through the tensor map)
  __nv_bfloat16 *out;
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *context_lens;
  int32_t *err;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int layer;
  int cap_tokens;
  float qscale;
  int num_seqs;
  int packed;                // clusters of 4 CTAs shared out by the packed plan
  int test_plan;             // test hook: plan first from the first length (pa_decode_set_test_plan)
};

// ------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}

__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t i;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(i));
  return i;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y)
               : "memory");
}

// Arrival on an mbarrier in another CTA of the cluster; orders this thread's
// earlier writes before it at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (as mbar_wait) with cluster-scope acquire: the writes other
// CTAs released with their arrivals are visible afterwards.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Asynchronous stores into the shared memory of a CTA of the cluster,
// counted as transaction bytes on that CTA's mbarrier: the receiver sees the
// data once the barrier's phase completes; the sender needs no fence and no
// arrival of its own.  Addresses from map_to_rank.
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(addr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float2 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::
                   "r"(addr),
               "f"(v.x), "f"(v.y), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void fma4(float4 &acc, const float4 &o, float sc) {
  acc.x = fmaf(o.x, sc, acc.x);
  acc.y = fmaf(o.y, sc, acc.y);
  acc.z = fmaf(o.z, sc, acc.z);
  acc.w = fmaf(o.w, sc, acc.w);
}

__device__ __forceinline__ uint2 bf16x4_scaled(const float4 &o, float s) {
  return make_uint2(float2_to_bf16x2(o.x * s, o.y * s), float2_to_bf16x2(o.z * s, o.w * s));
}

// L2 prefetch of the box of the tensor map at (head h, K|V kv, page blk):
// with 8-token pages one page's K or V rows of the head.
__device__ __forceinline__ void prefetch_rows_l2(const void *tmap, int h, int kv, int blk) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(0), "r"(h), "r"(0), "r"(kv), "r"(blk)
      : "memory");
}

// L2 prefetch of one tile: the box of the tensor map at (head h, first
// token tok0 of page blk).
__device__ __forceinline__ void prefetch_tile_l2(const void *tmap, int h, int tok0, int blk) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(0), "r"(h), "r"(tok0), "r"(0), "r"(blk)
      : "memory");
}

// Pages of BT tokens hold BT / 16 tiles: tile j is tokens 16 (j mod that)
// .. of page j / that.  With 8-token pages a tile is two pages, 2j and 2j+1
// (page() is the first, tok0() 0).
template <int BT>
struct TileOfPage {
  static constexpr int kTiles = BT >= kBs ? BT / kBs : 1;
  __device__ static int page(int j) { return BT >= kBs ? j / kTiles : 2 * j; }
  __device__ static int tok0(int j) { return BT >= kBs ? (j % kTiles) * kBs : 0; }
};

// Page ids of tile j of a table row: blk (the tile's page, or with 8-token
// pages its first) and, with 8-token pages, blk2 = the second page when the
// context reaches into it (else -1).  -1 for both when j >= t1.
template <int BT>
__device__ __forceinline__ void tile_ids(const int32_t *row, int j, int t1, int ctx, int &blk,
                                         int &blk2) {
  blk = -1;
  blk2 = -1;
  if (j < t1) {
    blk = row[TileOfPage<BT>::page(j)];
    if (BT < kBs && j * kBs + BT < ctx) blk2 = row[2 * j + 1];
  }
}

// Tiles [t0, t1) of a head with nb tiles, for CTA `rank` of c.
__device__ __forceinline__ void tile_range(int nb, int rank, int c, int &t0, int &t1) {
  t0 = static_cast<int>(static_cast<long long>(nb) * rank / c);
  t1 = static_cast<int>(static_cast<long long>(nb) * (rank + 1) / c);
}

// Barrier `id` over `count` threads that also returns whether v held for all.
__device__ __forceinline__ bool bar_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int warp_sum(int v) { return __reduce_add_sync(0xffffffffu, v); }

// The packed plan (one warp; n <= 32 sequences, lane s holding sequence s's
// 16-token tiles).  Sequence s gets k_s in {1, 2, 4} CTAs per kv head: for the
// smallest M (binary search) with every k_s = 1 if T_s <= M, 2 if T_s <= 2M,
// else 4 (T_s <= 4M), and sum k_s <= 2n, so that no CTA takes more than M
// tiles where a uniform 2 CTAs per pair would give the longest head's CTAs
// T_max / 2.  Sequence s's 8 k_s CTAs follow sequence s-1's in the grid
// (clusters of 4: a part never straddles one), kv head e / k_s taking part
// e mod k_s of them.  Writes the role of grid CTA g: the sequence (-1 past
// the plan's CTAs: nothing to do), kv head, parts and part.
__device__ __forceinline__ void packed_role(int tiles, int n, int g, int lane, int (&role)[4]) {
  const bool live = lane < n;
  const int tmax = __reduce_max_sync(0xffffffffu, live ? tiles : 0);
  auto parts_for = [&](int m) { return !live ? 0 : (tiles <= m ? 1 : (tiles <= 2 * m ? 2 : 4)); };
  int lo = (tmax + 3) / 4, hi = max(tmax, 1);
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    if (warp_sum(parts_for(mid)) <= 2 * n) hi = mid;
    else lo = mid + 1;
  }
  const int k = parts_for(max(lo, 1));
  int incl = 8 * k;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - 8 * k;
  const unsigned hit = __ballot_sync(0xffffffffu, live && g >= excl && g < incl);
  const int sl = hit ? __ffs(hit) - 1 : 0;
  const int ks = __shfl_sync(0xffffffffu, k, sl);
  const int e = g - __shfl_sync(0xffffffffu, excl, sl);
  role[0] = hit ? sl : -1;
  role[1] = hit ? e / ks : 0;
  role[2] = hit ? ks : 1;
  role[3] = hit ? e % ks : 0;
}

// One stage: wait until it is free, write its descriptor, issue the copies
// of tiles j0 .. j0+n-1 (lane w < n holds the page ids of tile j0 + w, see
// tile_ids).  Returns the slots with a page id out of range, or -1 if the
// wait timed out.
template <int BT>
__device__ __forceinline__ int publish_stage(PairSmem &sm, const CUtensorMap *map, int stage,
                                             uint32_t phase, int h, int j0, int n, int blk,
                                             int blk2, int last, int tail, int flags,
                                             int num_blocks, int lane) {
  int good = 1;
  if (lane == 0) good = mbar_wait(&sm.empty[stage], phase ^ 1) ? 1 : 0;
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good) return -1;
  const bool mine = lane < n;
  const bool valid = mine && blk >= 0 && blk < num_blocks;
  unsigned char *slot = sm.kv[stage] + lane * kSlotBytes;
  if constexpr (BT < kBs) {
    // the tile's second page, where its tokens reach into it
    const int n_tok = (j0 + lane == last) ? tail : kBs;
    const bool need2 = mine && n_tok > BT;
    const bool valid2 = need2 && blk2 >= 0 && blk2 < num_blocks;
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned vmask2 = __ballot_sync(0xffffffffu, valid2);
    const unsigned bad = __ballot_sync(0xffffffffu, (mine && !valid) || (need2 && !valid2));
    if (lane == 0) {
      PairStage d;
      d.j0 = j0;
      d.n = n;
      d.last = last;
      d.tail = tail;
      d.bad = static_cast<int>(vmask | (vmask2 << kPairWarps));   // pages loaded
      d.flags = flags;
      sm.desc[stage] = d;
      const uint32_t bytes = static_cast<uint32_t>(__popc(vmask) + __popc(vmask2)) * (kSlotBytes / 2);
      if (bytes) mbar_arrive_expect_tx(&sm.full[stage], bytes);
      else mbar_arrive(&sm.full[stage]);
    }
    __syncwarp();
    // K and V rows of each 8-token page, 1 KiB each: the first page's to
    // token rows 0..7 of the slot's K and V halves, the second's to 8..15
    if (valid) {
      tma_load_5d(slot, map, 0, h, 0, 0, blk, &sm.full[stage]);
      tma_load_5d(slot + kSlotBytes / 2, map, 0, h, 0, 1, blk, &sm.full[stage]);
    }
    if (valid2) {
      tma_load_5d(slot + kSlotBytes / 4, map, 0, h, 0, 0, blk2, &sm.full[stage]);
      tma_load_5d(slot + 3 * kSlotBytes / 4, map, 0, h, 0, 1, blk2, &sm.full[stage]);
    }
    return static_cast<int>(bad);
  } else {
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    const unsigned bad = __ballot_sync(0xffffffffu, mine && !valid);
    if (lane == 0) {
      PairStage d;
      d.j0 = j0;
      d.n = n;
      d.last = last;
      d.tail = tail;
      d.bad = static_cast<int>(bad);
      d.flags = flags;
      sm.desc[stage] = d;
      const uint32_t bytes = static_cast<uint32_t>(__popc(vmask)) * kSlotBytes;
      if (bytes) mbar_arrive_expect_tx(&sm.full[stage], bytes);
      else mbar_arrive(&sm.full[stage]);
    }
    __syncwarp();
    if (valid)
      tma_load_5d(slot, map, 0, h, TileOfPage<BT>::tok0(j0 + lane), 0, blk, &sm.full[stage]);
    return static_cast<int>(bad);
  }
}

template <int BT>
__global__ void __launch_bounds__(kPairThreads, kPairCtasPerSm)
    decode_pair_kernel(const __grid_constant__ CUtensorMap kv_map, PairParams p) {
  using TP = TileOfPage<BT>;
  extern __shared__ unsigned char smem_raw[];
  PairSmem &sm = *reinterpret_cast<PairSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const bool packed = p.packed != 0;
  // this CTA's (sequence, kv head), and its part of the kparts CTAs that
  // share that pair's tiles; with the packed plan the producer warp works
  // them out (below) and hands them to the consumers through role[]
  int s = -1, h = 0, kparts = c, part = rank;
  if (!packed) {
    const int pair = static_cast<int>(cluster_id());
    s = pair / kHkv;
    h = pair % kHkv;
  }
  const int32_t *row = nullptr;
  // the next kernel on the stream may be scheduled at once: it waits for
  // this one to finish before it reads anything this one writes
  pdl_launch_dependents();

  // ---- before the previous kernel on the stream has finished
  if (tid == 0) {
    prefetch_tensormap(&kv_map);
    for (int st = 0; st < kPairStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kPairWarps);
    }
    // the leader expects every CTA's state (O and (m, l) of 4 q heads) as
    // bytes (with the packed plan, once it knows how many parts it has)
    mbar_init(&sm.parts_full, 1);
    if (!packed && rank == 0 && c > 1)
      mbar_arrive_expect_tx(&sm.parts_full, static_cast<uint32_t>(c * kGqa * (kD * 4 + 8)));
    fence_mbar_init();
  }
  // the speculative plan: this CTA's range under the context length as it
  // reads now, and its first page ids; their tiles are prefetched into L2
  int spec_ctx = 0, spec_t0 = 0, spec_t1 = 0, spec_blk = -1, spec_blk2 = -1;
  int spec_len = 0;   // packed plan: lane s's sequence length as read before the wait
  if (warp == kPairWarps) {
    if (packed) {
      spec_len = lane < p.num_seqs ? min(max(p.context_lens[lane], 0), p.cap_tokens) : 0;
      if (p.test_plan) {   // (every lane takes part in the shuffle)
        const int first = __shfl_sync(0xffffffffu, spec_len, 0);
        spec_len = lane < p.num_seqs ? first : 0;
      }
      int role[4];
      packed_role((spec_len + kBs - 1) / kBs, p.num_seqs,
                  static_cast<int>(cluster_id()) * c + rank, lane, role);
      s = role[0];
      h = role[1];
      kparts = role[2];
      part = role[3];
      if (lane == 0) {   // for the consumers' first q load (the barrier below publishes it)
        sm.role[0] = s;
        sm.role[1] = h;
        sm.role[2] = kparts;
        sm.role[3] = part;
      }
    }
    if (s >= 0) {
      row = p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
      // (the packed plan has every length already: one dependent read less
      // before the first copies, whose chain of reads is on the critical
      // path of the CTAs that start late)
      spec_ctx = packed ? __shfl_sync(0xffffffffu, spec_len, s)
                        : min(max(p.context_lens[s], 0), p.cap_tokens);
      tile_range((spec_ctx + kBs - 1) / kBs, part, kparts, spec_t0, spec_t1);
      // (the first 32 ids are kept for the first stages; the prefetches share
      // the SM's TMA unit with the copies, so only the first 3 stages' worth)
      const int j = spec_t0 + lane;
      tile_ids<BT>(row, j, spec_t1, spec_ctx, spec_blk, spec_blk2);
      if (spec_blk >= 0 && spec_blk < p.num_blocks) {
        if (BT < kBs) {
          // (the first page's K and V of a third as many tiles: the same count of requests)
          if (lane < kPrefetchTiles / 3) {
            prefetch_rows_l2(&kv_map, h, 0, spec_blk);
            prefetch_rows_l2(&kv_map, h, 1, spec_blk);
          }
        } else if (lane < kPrefetchTiles) {
          prefetch_tile_l2(&kv_map, h, TP::tok0(j), spec_blk);
        }
      }
    }
  }
  if (c > 1) cluster_sync_all();   // every CTA's barriers exist before any remote arrival
  else __syncthreads();
  // everything read below may come from the previous kernel on the stream
  pdl_wait_primary();

  if (warp == kPairWarps) {
    // ===================================================== producer warp ==
    // current values, read now and checked against the speculative ones
    // once the first stages are on their way (with the packed plan, every
    // sequence's length: the plan itself may have moved)
    const int now_raw = packed ? (lane < p.num_seqs ? p.context_lens[lane] : 0)
                               : (s >= 0 ? p.context_lens[s] : 0);
    int blk_now, blk_now2;
    tile_ids<BT>(row, spec_t0 + lane, spec_t1, spec_ctx, blk_now, blk_now2);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;   // per stage: used / parity of its last phase
    bool ok = true;
    int bad_seen = 0;
    const int spec_nb = (spec_ctx + kBs - 1) / kBs;
    const int spec_stages = min(kPairStages, (spec_t1 - spec_t0 + kPairWarps - 1) / kPairWarps);
    for (int e = 0; e < spec_stages && ok; ++e) {
      const int j0 = spec_t0 + e * kPairWarps;
      const int blk = __shfl_sync(0xffffffffu, spec_blk, (e * kPairWarps + lane) & 31);
      const int blk2 = BT < kBs ? __shfl_sync(0xffffffffu, spec_blk2, (e * kPairWarps + lane) & 31)
                                : -1;
      const int bad = publish_stage<BT>(sm, &kv_map, stage, phase, h, j0,
                                        min(kPairWarps, spec_t1 - j0), blk, blk2, spec_nb - 1,
                                        spec_ctx - (spec_nb - 1) * kBs, 0, p.num_blocks, lane);
      if (bad < 0) {
        ok = false;
        break;
      }
      bad_seen |= bad;
      if (lane == 0) {
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      }
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    // the next layer's table row of this sequence into L2 (one CTA per
    // sequence): the next call's CTAs read it before their dependency wait,
    // while this call streams, and a miss to DRAM there is on their path
    if (s >= 0 && part == 0 && h == 0 && p.layer + 1 < p.n_layers) {
      const int32_t *next =
          p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer + 1) * p.max_blocks;
      for (int i = lane * 32; i < p.max_blocks; i += 32 * 32) prefetch_l2(next + i);
    }
    int ctx_raw = now_raw;
    bool moved = false;   // the packed plan gave this CTA another role
    if (packed) {
      const int now_len = min(max(now_raw, 0), p.cap_tokens);
      if (!__all_sync(0xffffffffu, now_len == spec_len)) {
        int role[4];
        packed_role((now_len + kBs - 1) / kBs, p.num_seqs,
                    static_cast<int>(cluster_id()) * c + rank, lane, role);
        moved = role[0] != s || role[1] != h || role[2] != kparts || role[3] != part;
        s = role[0];
        h = role[1];
        kparts = role[2];
        part = role[3];
        row = s >= 0 ? p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks
                     : nullptr;
      }
      ctx_raw = __shfl_sync(0xffffffffu, now_raw, s >= 0 ? s : 0);
      // the final role, for the consumers: written before any later stage
      // is published, so a consumer that sees kMoved or the end reads it
      if (moved && lane == 0) {
        sm.role[0] = s;
        sm.role[1] = h;
        sm.role[2] = kparts;
        sm.role[3] = part;
      }
    }
    const bool idle = s < 0;   // no part of the plan: only the end stage follows
    const int ctx = idle ? 0 : min(max(ctx_raw, 0), p.cap_tokens);
    if (!idle && lane == 0 && part == 0 && h == 0 && (ctx_raw < 0 || ctx_raw > p.cap_tokens))
      report(p.err, PA_DEV_CTX_RANGE);
    const bool same =
        !moved && ctx == spec_ctx &&
        __all_sync(0xffffffffu, blk_now == spec_blk && (BT >= kBs || blk_now2 == spec_blk2));
    const int nb = (ctx + kBs - 1) / kBs;
    const int last = nb - 1, tail = ctx - (nb - 1) * kBs;
    int t0 = spec_t0, t1 = spec_t1, j = spec_t0 + spec_stages * kPairWarps, base = spec_t0;
    int ids = blk_now, ids2 = blk_now2, flags = 0;
    if (!same) {
      // the plan moved: stream the current range from its start; the
      // consumers drop what they accumulated from the speculative stages
      tile_range(nb, part, kparts, t0, t1);
      j = base = t0;
      tile_ids<BT>(row, t0 + lane, t1, ctx, ids, ids2);
      flags = kReset | (moved ? kMoved : 0);
    } else if (bad_seen && lane == 0) {
      report(p.err, PA_DEV_BAD_BLOCK);
    }
    int ids_next, ids_next2;
    tile_ids<BT>(row, base + kIdBatch + lane, t1, ctx, ids_next, ids_next2);
    while (ok && j < t1) {
      if (j >= base + kIdBatch) {
        base += kIdBatch;
        ids = ids_next;
        ids2 = ids_next2;
        tile_ids<BT>(row, base + kIdBatch + lane, t1, ctx, ids_next, ids_next2);
      }
      const int blk = __shfl_sync(0xffffffffu, ids, (j - base + lane) & 31);
      const int blk2 = BT < kBs ? __shfl_sync(0xffffffffu, ids2, (j - base + lane) & 31) : -1;
      const int bad = publish_stage<BT>(sm, &kv_map, stage, phase, h, j, min(kPairWarps, t1 - j),
                                        blk, blk2, last, tail, flags, p.num_blocks, lane);
      if (bad < 0) {
        ok = false;
        break;
      }
      if (bad && lane == 0) report(p.err, PA_DEV_BAD_BLOCK);
      flags = 0;
      if (lane == 0) {
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      }
      j += kPairWarps;
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (lane == 0) {
      if (ok && mbar_wait(&sm.empty[stage], phase ^ 1)) {
        PairStage d;
        d.j0 = 0;
        d.n = 0;
        d.last = -1;
        d.tail = 0;
        d.bad = 0;
        d.flags = kEnd | flags | (idle ? kIdle : 0);
        sm.desc[stage] = d;
        mbar_arrive(&sm.full[stage]);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      } else {
        report(p.err, PA_DEV_TIMEOUT);
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (int st = 0; st < kPairStages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.full[st], (issued_parity >> st) & 1u)) report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
    return;
  }

  // ======================================================= consumer warps ==
  const int w = warp;                    // slot of every stage this warp takes
  const int r = lane >> 2;               // fragment row = q head within the group (0..3 real)
  const int c2 = 2 * (lane & 3);         // fragment column pair
  const bool real_row = r < kGqa;
  uint32_t qa[4], qc[4];
  // with the packed plan: the role as planned before the wait (a stage
  // flagged kMoved hands over the final one; a consumer that reads role[]
  // after the producer rewrote it starts on the final role, or on a mix of
  // the two, and the kMoved stage, which comes before any stage of the new
  // range, sets it right and drops what it accumulated)
  if (packed) {
    s = sm.role[0];
    h = sm.role[1];
  }
  if (s >= 0) load_q_fragments(p.q + static_cast<size_t>(s) * kHq * kD, h, lane, qa, qc);
  TileState ts;
  ts.reset();
  int stage = 0;
  uint32_t phase = 0;
  bool timed_out = false;
  while (true) {
    if (!mbar_wait(&sm.full[stage], phase)) {
      report(p.err, PA_DEV_TIMEOUT);
      timed_out = true;
      break;
    }
    const PairStage d = sm.desc[stage];
    if (d.flags & kMoved) {
      s = sm.role[0];
      h = sm.role[1];
      if (s >= 0) load_q_fragments(p.q + static_cast<size_t>(s) * kHq * kD, h, lane, qa, qc);
    }
    if (d.flags & kReset) ts.reset();
    if (d.flags & kEnd) break;
    if constexpr (BT < kBs) {
      // 8-token pages: the rows of the pages that were loaded
      const unsigned ld = ((d.bad >> w) & 1u ? 0x00ffu : 0u) |
                          ((d.bad >> (kPairWarps + w)) & 1u ? 0xff00u : 0u);
      if (s >= 0 && w < d.n && ld) {
        const int n_valid = (d.j0 + w == d.last) ? d.tail : kBs;
        const uint32_t ktile = smem_u32(sm.kv[stage] + w * kSlotBytes);
        attend_tile<true>(ktile, ktile + kBs * kHeadRowBytes, n_valid,
                          ld & ((1u << n_valid) - 1u), qa, qc, p.qscale, lane, ts);
      }
    } else if (s >= 0 && w < d.n && !((d.bad >> w) & 1)) {
      const int n_valid = (d.j0 + w == d.last) ? d.tail : kBs;
      const uint32_t ktile = smem_u32(sm.kv[stage] + w * kSlotBytes);
      attend_tile<false>(ktile, ktile + kBs * kHeadRowBytes, n_valid, 0u, qa, qc, p.qscale, lane,
                         ts);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
    if (++stage == kPairStages) {
      stage = 0;
      phase ^= 1;
    }
  }

  if (packed) {
    // the consumer warps agree: all of them saw the end (then the final role
    // is in role[]), or the CTA writes nothing (the wait that ran out is
    // reported; the pair's leader, missing this part, reports its own)
    if (!bar_and(1, kPairWarps * 32, !timed_out)) return;
    s = sm.role[0];
    h = sm.role[1];
    kparts = sm.role[2];
    part = sm.role[3];
    if (s < 0) return;
  }

  // ---- the 8 warp states -> one CTA state.  Each warp parks its state in
  // its own slot of stage 0: every copy has landed (the warp has waited on
  // every stage up to the end), and no other warp reads that slot any more.
  const float lt = row_sum(ts);
  {
    float *my_o = reinterpret_cast<float *>(sm.kv[0] + w * kSlotBytes);   // [4 rows][64]
    float2 *my_ml = reinterpret_cast<float2 *>(my_o + kGqa * kD);
    if (real_row) {
#pragma unroll
      for (int t = 0; t < 8; ++t)
        *reinterpret_cast<float2 *>(my_o + r * kD + 8 * t + c2) = make_float2(ts.out(t, 0), ts.out(t, 1));
      if ((lane & 3) == 0) my_ml[r] = make_float2(timed_out ? neg_inf() : ts.m, timed_out ? 0.f : lt);
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kPairWarps * 32) : "memory");
  // threads 0..63: q head row qrow, dims d0 .. d0+3
  if (tid >= kGqa * 16) return;
  const int qrow = tid >> 4, d0 = 4 * (tid & 15);
  float M = neg_inf();
#pragma unroll
  for (int k = 0; k < kPairWarps; ++k) {
    const float2 ml = reinterpret_cast<const float2 *>(
        reinterpret_cast<const float *>(sm.kv[0] + k * kSlotBytes) + kGqa * kD)[qrow];
    M = fmaxf(M, ml.x);
  }
  float L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != neg_inf()) {
#pragma unroll
    for (int k = 0; k < kPairWarps; ++k) {
      const float *ko = reinterpret_cast<const float *>(sm.kv[0] + k * kSlotBytes);
      const float2 ml = reinterpret_cast<const float2 *>(ko + kGqa * kD)[qrow];
      const float sc = fast_exp2(ml.x - M);   // empty warp states carry m = -inf: weight 0
      L = fmaf(ml.y, sc, L);
      fma4(O, *reinterpret_cast<const float4 *>(ko + qrow * kD + d0), sc);
    }
  }
  uint2 *dst = reinterpret_cast<uint2 *>(
      p.out + (static_cast<size_t>(s) * kHq + h * kGqa + qrow) * kD + d0);
  if (kparts == 1) {
    *dst = bf16x4_scaled(O, L > 0.f ? 1.f / L : 0.f);
    return;
  }

  // ---- the kparts CTA states -> the output, in the shared memory of the
  // pair's first CTA (the leader): 64 asynchronous 16-byte stores and 4 of
  // 8 bytes per CTA, which complete the leader's barrier by their byte count
  const uint32_t lead = static_cast<uint32_t>(rank - part);
  const uint32_t bar = map_to_rank(&sm.parts_full, lead);
  st_async_f32x4(map_to_rank(&sm.part_o[part][qrow][d0], lead), O, bar);
  if ((tid & 15) == 0)
    st_async_f32x2(map_to_rank(&sm.part_ml[part][qrow], lead), make_float2(M, L), bar);
  if (part != 0) return;
  // (with the packed plan the leader learns its part count only now; bytes
  // that land before it says how many to expect are counted all the same)
  if (packed && tid == 0)
    mbar_arrive_expect_tx(&sm.parts_full, static_cast<uint32_t>(kparts * kGqa * (kD * 4 + 8)));
  if (!mbar_wait_cluster(&sm.parts_full, 0)) {
    report(p.err, PA_DEV_TIMEOUT);
    return;
  }
  float Mc = neg_inf();
  for (int k = 0; k < kparts; ++k) Mc = fmaxf(Mc, sm.part_ml[k][qrow].x);
  float Lc = 0.f;
  float4 Oc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (Mc != neg_inf()) {
    for (int k = 0; k < kparts; ++k) {
      const float sc = fast_exp2(sm.part_ml[k][qrow].x - Mc);
      Lc = fmaf(sm.part_ml[k][qrow].y, sc, Lc);
      fma4(Oc, *reinterpret_cast<const float4 *>(&sm.part_o[k][qrow][d0]), sc);
    }
  }
  *dst = bf16x4_scaled(Oc, Lc > 0.f ? 1.f / Lc : 0.f);
}

// ===========================================================================
// One cluster of c CTAs (c = 1 .. 16) per sequence.  A CTA streams a range
// of the sequence's pages, one 32 KiB copy per page (all 8 kv heads, through
// the page tensor map: [K|V][head][token][64] in shared memory, each head's
// token rows 128-byte swizzled), and warp h computes kv head h.  CTA r owns
// q heads [r * 32/c, (r + 1) * 32/c): every CTA sends its state for those
// heads to their owner's shared memory, and the owner combines and writes.
constexpr int kSeqPrefetchPages = 4;
constexpr int kBadPage = 4;   // the stage's page id was out of range (no data)

struct SeqStage {
  int j;       // tile (page) of the sequence
  int last;    // the sequence's last tile
  int tail;    // tokens in it (1..16)
  int flags;   // kReset, kEnd, kBadPage
};

struct __align__(1024) SeqSmem {
  unsigned char kv[kPairStages][kPairStageBytes];
  float part_o[kHq][kD];     // owner: row (sender rank * 32/c + owned head) -> unnormalised state
  float2 part_ml[kHq];       // and its (m, l)
  SeqStage desc[kPairStages];
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t parts_full;       // owner: every sender's states have landed
};

// One page into a stage (lane 0 of the producer warp).  False if the wait
// for the stage timed out.
__device__ __forceinline__ bool publish_page(SeqSmem &sm, const CUtensorMap *map, int stage,
                                             uint32_t phase, int j, int blk, int last, int tail,
                                             int flags, int num_blocks) {
  if (!mbar_wait(&sm.empty[stage], phase ^ 1)) return false;
  const bool valid = blk >= 0 && blk < num_blocks;
  SeqStage d;
  d.j = j;
  d.last = last;
  d.tail = tail;
  d.flags = flags | (valid ? 0 : kBadPage);
  sm.desc[stage] = d;
  if (valid) {
    mbar_arrive_expect_tx(&sm.full[stage], kPairStageBytes);
    tma_load_5d(sm.kv[stage], map, 0, 0, 0, 0, blk, &sm.full[stage]);
  } else {
    mbar_arrive(&sm.full[stage]);
  }
  return true;
}

__global__ void __launch_bounds__(kPairThreads, kPairCtasPerSm)
    decode_seq_kernel(const __grid_constant__ CUtensorMap page_map, PairParams p) {
  extern __shared__ unsigned char smem_raw[];
  SeqSmem &sm = *reinterpret_cast<SeqSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_rank());
  const int s = static_cast<int>(cluster_id());
  const int qpo = kHq / c;   // q heads each CTA owns
  const int32_t *row = p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
  pdl_launch_dependents();   // the next kernel waits for this one before reading its output

  // ---- before the previous kernel on the stream has finished
  if (tid == 0) {
    prefetch_tensormap(&page_map);
    for (int st = 0; st < kPairStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kPairWarps);
    }
    mbar_init(&sm.parts_full, c * qpo * 4);   // per sender and owned head: one lane quad
    fence_mbar_init();
  }
  int spec_ctx = 0, spec_t0 = 0, spec_t1 = 0, spec_blk = -1;
  if (warp == kPairWarps) {
    spec_ctx = min(max(p.context_lens[s], 0), p.cap_tokens);
    tile_range((spec_ctx + kBs - 1) / kBs, rank, c, spec_t0, spec_t1);
    const int j = spec_t0 + lane;
    if (j < spec_t1) {
      spec_blk = row[j];
      if (lane < kSeqPrefetchPages && spec_blk >= 0 && spec_blk < p.num_blocks)
        prefetch_bulk_l2(p.kv + static_cast<size_t>(spec_blk) * kBlockBytes, kBlockBytes);
    }
  }
  if (c > 1) cluster_sync_all();   // every CTA's barriers exist before any remote arrival
  else __syncthreads();
  // everything read below may come from the previous kernel on the stream
  pdl_wait_primary();

  if (warp == kPairWarps) {
    // ===================================================== producer warp ==
    const int ctx_raw = p.context_lens[s];
    const int blk_now = spec_t0 + lane < spec_t1 ? row[spec_t0 + lane] : -1;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    const int spec_nb = (spec_ctx + kBs - 1) / kBs;
    const int spec_pages = min(kPairStages, spec_t1 - spec_t0);
    bool spec_bad_page = false;
    for (int e = 0; e < spec_pages; ++e) {
      const int blk = __shfl_sync(0xffffffffu, spec_blk, e);
      spec_bad_page |= !(blk >= 0 && blk < p.num_blocks);
      int good = 1;
      if (lane == 0)
        good = publish_page(sm, &page_map, stage, phase, spec_t0 + e, blk, spec_nb - 1,
                            spec_ctx - (spec_nb - 1) * kBs, 0, p.num_blocks);
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      }
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    const int ctx = min(max(ctx_raw, 0), p.cap_tokens);
    if (lane == 0 && rank == 0 && (ctx_raw < 0 || ctx_raw > p.cap_tokens))
      report(p.err, PA_DEV_CTX_RANGE);
    const bool same = ctx == spec_ctx && __all_sync(0xffffffffu, blk_now == spec_blk);
    const int nb = (ctx + kBs - 1) / kBs;
    const int last = nb - 1, tail = ctx - (nb - 1) * kBs;
    int t0 = spec_t0, t1 = spec_t1, j = spec_t0 + spec_pages, base = spec_t0;
    int ids = blk_now, flags = 0;
    if (!same) {
      tile_range(nb, rank, c, t0, t1);
      j = base = t0;
      ids = t0 + lane < t1 ? row[t0 + lane] : -1;
      flags = kReset;
    } else if (spec_bad_page && lane == 0) {
      report(p.err, PA_DEV_BAD_BLOCK);
    }
    int ids_next = base + kIdBatch + lane < t1 ? row[base + kIdBatch + lane] : -1;
    while (ok && j < t1) {
      if (j >= base + kIdBatch) {
        base += kIdBatch;
        ids = ids_next;
        ids_next = base + kIdBatch + lane < t1 ? row[base + kIdBatch + lane] : -1;
      }
      const int blk = __shfl_sync(0xffffffffu, ids, (j - base) & 31);
      int good = 1;
      if (lane == 0) {
        good = publish_page(sm, &page_map, stage, phase, j, blk, last, tail, flags, p.num_blocks);
        if (good && !(blk >= 0 && blk < p.num_blocks)) report(p.err, PA_DEV_BAD_BLOCK);
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) {
        ok = false;
        break;
      }
      flags = 0;
      if (lane == 0) {
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      }
      ++j;
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1;
      }
    }
    if (lane == 0) {
      if (ok && mbar_wait(&sm.empty[stage], phase ^ 1)) {
        SeqStage d;
        d.j = 0;
        d.last = -1;
        d.tail = 0;
        d.flags = kEnd | flags;
        sm.desc[stage] = d;
        mbar_arrive(&sm.full[stage]);
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      } else {
        report(p.err, PA_DEV_TIMEOUT);
      }
      for (int st = 0; st < kPairStages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.full[st], (issued_parity >> st) & 1u)) report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
    return;
  }

  // ======================================================= consumer warps ==
  const int h = warp;                    // kv head
  const int r = lane >> 2;               // fragment row = q head within the group (0..3 real)
  const int c2 = 2 * (lane & 3);
  const bool real_row = r < kGqa;
  uint32_t qa[4], qc[4];
  load_q_fragments(p.q + static_cast<size_t>(s) * kHq * kD, h, lane, qa, qc);
  TileState ts;
  ts.reset();
  int stage = 0;
  uint32_t phase = 0;
  bool timed_out = false;
  while (true) {
    if (!mbar_wait(&sm.full[stage], phase)) {
      report(p.err, PA_DEV_TIMEOUT);
      timed_out = true;
      break;
    }
    const SeqStage d = sm.desc[stage];
    if (d.flags & kReset) ts.reset();
    if (d.flags & kEnd) break;
    if (!(d.flags & kBadPage)) {
      const int n_valid = (d.j == d.last) ? d.tail : kBs;
      // [K|V][head][token][64]: head h's K rows, then (16 KiB on) its V rows
      const uint32_t ktile = smem_u32(sm.kv[stage] + h * (kBs * kHeadRowBytes));
      attend_tile<false>(ktile, ktile + kPairStageBytes / 2, n_valid, 0u, qa, qc, p.qscale, lane,
                         ts);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
    if (++stage == kPairStages) {
      stage = 0;
      phase ^= 1;
    }
  }

  // ---- each q head's state to the CTA that owns it
  const float lt = row_sum(ts);
  if (real_row) {
    const int qh = h * kGqa + r;
    const int owner = qh / qpo, slot = rank * qpo + qh % qpo;
#pragma unroll
    for (int t = 0; t < 8; ++t)
      st_cluster_f32x2(map_to_rank(&sm.part_o[slot][8 * t + c2], owner),
                       make_float2(ts.out(t, 0), ts.out(t, 1)));
    if ((lane & 3) == 0)
      st_cluster_f32x2(map_to_rank(&sm.part_ml[slot], owner),
                       make_float2(timed_out ? neg_inf() : ts.m, timed_out ? 0.f : lt));
    mbar_arrive_cluster(map_to_rank(&sm.parts_full, owner));
  }
  if (!mbar_wait_cluster(&sm.parts_full, 0)) {
    report(p.err, PA_DEV_TIMEOUT);
    return;
  }
  for (int e = tid; e < qpo * kD; e += kPairWarps * 32) {
    const int oh = e / kD, dd = e % kD;   // owned head, dim
    float M = neg_inf();
    for (int k = 0; k < c; ++k) M = fmaxf(M, sm.part_ml[k * qpo + oh].x);
    float L = 0.f, O = 0.f;
    if (M != neg_inf()) {
      for (int k = 0; k < c; ++k) {
        const float2 ml = sm.part_ml[k * qpo + oh];
        const float sc = fast_exp2(ml.x - M);
        L = fmaf(ml.y, sc, L);
        O = fmaf(sm.part_o[k * qpo + oh][dd], sc, O);
      }
    }
    p.out[(static_cast<size_t>(s) * kHq + rank * qpo + oh) * kD + dd] =
        __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
  }
}

}  // namespace

size_t decode_pair_smem_bytes() { return sizeof(PairSmem) + 1024; }

int decode_seq_cluster(int num_seqs, int sm_count, int max_ctas) {
  long long cap = static_cast<long long>(sm_count) * kPairCtasPerSm;
  if (max_ctas > 0) cap = min(cap, static_cast<long long>(max_ctas));
  if (num_seqs <= 0 || num_seqs > cap) return 0;
  int c = 1;
  while (c < 16 && static_cast<long long>(num_seqs) * (2 * c) <= cap) c *= 2;
  return c;
}

int launch_decode_seq(const CUtensorMap &page_map, uint16_t *out, const uint16_t *q,
                      const void *kv_cache, int num_blocks, const int32_t *block_table,
                      int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                      int num_seqs, int layer, float scale, int32_t *err, int cluster,
                      cudaStream_t stream) {
  if (cluster != 1 && cluster != 2 && cluster != 4 && cluster != 8 && cluster != 16)
    return PA_ERR_ARG;
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  static bool attr_done[64] = {};
  static int c16_fits[64] = {};   // 0 not asked yet, 1 clusters of 16 schedule, 2 they do not
  const size_t smem = sizeof(SeqSmem) + 1024;
  if (!attr_done[di.device]) {
    if (cudaFuncSetAttribute(decode_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess ||
        cudaFuncSetAttribute(decode_seq_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[di.device] = true;
  }
  if (cluster == 16) {
    // 16 CTAs is beyond the portable cluster size: use it only where the
    // device reports that such clusters of this kernel can be resident
    if (c16_fits[di.device] == 0) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(16);
      qc.blockDim = dim3(kPairThreads);
      qc.dynamicSmemBytes = smem;
      cudaLaunchAttribute qa;
      qa.id = cudaLaunchAttributeClusterDimension;
      qa.val.clusterDim.x = 16;
      qa.val.clusterDim.y = 1;
      qa.val.clusterDim.z = 1;
      qc.attrs = &qa;
      qc.numAttrs = 1;
      int n = 0;
      const bool ok = cudaOccupancyMaxActiveClusters(&n, decode_seq_kernel, &qc) == cudaSuccess;
      cudaGetLastError();
      c16_fits[di.device] = ok && n > 0 ? 1 : 2;
    }
    if (c16_fits[di.device] == 2) cluster = 8;
  }
  PairParams prm;
  prm.kv = static_cast<const unsigned char *>(kv_cache);
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.q = q;
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.layer = layer;
  prm.cap_tokens = max_blocks_per_seq * kBs;
  prm.qscale = scale * kLog2e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_seqs) * cluster);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, decode_seq_kernel, page_map, prm) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

int decode_pair_cluster(int num_seqs, int sm_count, int max_ctas) {
  const long long pairs = static_cast<long long>(num_seqs) * kHkv;
  long long cap = static_cast<long long>(sm_count) * kPairCtasPerSm;
  if (max_ctas > 0) cap = min(cap, static_cast<long long>(max_ctas));
  // at least two CTAs per pair: with one, a batch of uneven contexts leaves
  // its longest heads on single CTAs and the split-context kernel is faster
  if (pairs * 2 > cap) return 0;
  int c = 2;
  while (c < kMaxCluster && pairs * (2 * c) <= cap) c *= 2;
  return c;
}

int g_test_plan = 0;   // pa_decode_set_test_plan

int launch_decode_pair(const CUtensorMap &map, uint16_t *out, const uint16_t *q,
                       int num_blocks, int block_tokens, const int32_t *block_table, int n_layers,
                       int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                       int layer, float scale, int32_t *err, int cluster, cudaStream_t stream) {
  if (cluster != 1 && cluster != 2 && cluster != 4 && cluster != 8) return PA_ERR_ARG;
  if (block_tokens != kBs / 2 && block_tokens != kBs && block_tokens != 2 * kBs) return PA_ERR_ARG;
  const int bi = block_tokens == kBs ? 0 : (block_tokens == 2 * kBs ? 1 : 2);
  void (*kern)(const CUtensorMap, PairParams) =
      bi == 0 ? decode_pair_kernel<kBs>
              : (bi == 1 ? decode_pair_kernel<2 * kBs> : decode_pair_kernel<kBs / 2>);
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  static bool attr_done[3][64] = {};
  const size_t smem = decode_pair_smem_bytes();
  if (!attr_done[bi][di.device]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[bi][di.device] = true;
  }
  PairParams prm;
  prm.kv = nullptr;
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.q = q;
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.layer = layer;
  prm.cap_tokens = max_blocks_per_seq * block_tokens;
  prm.qscale = scale * kLog2e;
  prm.num_seqs = num_seqs;
  // two CTAs per pair on average: the packed plan shares them out by length
  // (1, 2 or 4 per kv head of a sequence) in clusters of 4
  const bool packed = cluster == 2 && num_seqs <= 32;
  prm.packed = packed ? 1 : 0;
  prm.test_plan = g_test_plan;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_seqs) * kHkv * cluster);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(packed ? 4 : cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kern, map, prm) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace pa

extern "C" int pa_decode_set_test_plan(int mode) {
  if (mode != 0 && mode != 1) return PA_ERR_ARG;
  pa::g_test_plan = mode;
  return PA_OK;
}
