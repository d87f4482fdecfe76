// pa_prefill.cu -- causal attention of a prompt chunk over its sequence's
// paged cache (the prefill side of the paged path) on the sm_103a tensor
// cores: tcgen05 MMAs from shared memory into TMEM accumulators.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of
// one inference": prefill pushes the whole prompt through at once (matrix x
// matrix), decode one token per step; "What is in the box": 16-token pages
// plus block_table, GQA_Q_TO_K_RATIO = 4, online softmax.
//
// Token i of sequence s (row cu_tokens[s] + i) sits at position
// context_lens[s] + i and attends over positions 0..context_lens[s] + i of its
// sequence, whose K/V (the chunk's own included) are already in the cache.
//
// Persistent CTAs (one per SM) work through (64-token query tile, kv head)
// items, each tile in two halves of 32 tokens:
// each half's 128 MMA rows are its 32 tokens x the 4 q heads of the GQA group
// (row = 4 * token + head), so every K/V byte brought into shared memory
// serves 256 query rows.  Keys go in chunks of 128 (8 pages).  Warp roles
// (384 threads):
//   warp 8      producer: the two Q tiles (TMA), then per chunk 16 TMA copies
//               (K rows and V rows of 8 pages) into a 5-stage ring;
//   warps 9, 10 MMA warps, one per half: one thread issues the half's
//               S_{j+1} = Q K_{j+1}^T (M 128, N 128, 4 k-steps) into its TMEM
//               S columns as soon as the half's softmax has read S_j, and,
//               once the softmax has written P_j, O += P_j V_j (M 128, N 64,
//               8 k-steps, P from TMEM, V read from shared memory as an
//               MN-major operand) into its O columns.  S_{j+1} is thus
//               computed while the softmax works on S_j.  A tcgen05.mma issue
//               blocks while the tensor core's queue is full, so each half
//               has its own issuing warp; an elected lane of the converged
//               warp issues (from a branch on the lane index, each MMA takes
//               two to three times as long).  The warp of the half that sees
//               every chunk also zeroes the V rows that lie past the tile's
//               last key or in a page that was not loaded;
//   warps 0-3, 4-7   softmax of half 0 / half 1, one thread per row (TMEM
//               lane): S_j from TMEM in one round trip, causal mask, row
//               maximum and sum in fp32 (log2 domain), P_j rounded to bf16
//               into the half's own 64 TMEM columns (two keys per column),
//               from which the PV MMA reads its A operand, once PV_{j-1} has
//               completed; O accumulates in TMEM and is rescaled only when
//               the row maximum grows by more than 2^8; the output row at
//               the end.
// The tensor core alternates between the halves: one half's MMAs run while
// the other half's softmax works.
#include <climits>
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kQTok = 32;                     // query tokens per half
constexpr int kHalves = 2;
constexpr int kCtaTok = kQTok * kHalves;      // query tokens per CTA
constexpr int kRows = kQTok * kGqa;           // 128 MMA rows per half
constexpr int kChunk = 128;                   // keys per chunk (8 pages of 16 tokens)
constexpr int kStagesP = 4;
constexpr int kQBufs = 2;                     // Q tiles in flight: the next item's loads early
constexpr int kSortTiles = 4096;              // tiles ordered by weight; beyond, by index
constexpr int kWeightBins = 256;              // weight classes (see tile_bin)
constexpr int kSoftThreads = kRows;           // one softmax warpgroup per half
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPThreads = 12 * 32;            // 3 warpgroups; warp 11 only rebalances registers
// Register budget: 384 threads x 168 at launch = 64,512.  The producer/MMA
// warpgroup gives up to 80 and each softmax warpgroup takes 200:
// 2 x 128 x 200 + 128 x 80 = 61,440 (every SM sub-partition: 2 x 200 + 80
// registers per lane, within its 512).
constexpr int kRegsLaunch = 168;
constexpr int kRegsSoft = 200;
constexpr int kRegsOther = 80;
static_assert(2 * 128 * kRegsSoft + 128 * kRegsOther <= kPThreads * kRegsLaunch,
              "register split above the launch budget");
constexpr int kTileRowBytes = kHeadRowBytes;             // 128-byte rows
constexpr int kOperandBytes = kChunk * kTileRowBytes;    // 16 KiB: 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;                      // S x2 (256) + O x2 (128) + P x2 (128)
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;                         // P of half h: 64 columns of bf16 pairs
constexpr int kMaxSeqsP = 2048;
constexpr float kLog2eP = 1.4426950408889634f;

struct PrefillParams {
  __nv_bfloat16 *out;
  const int32_t *cu_tokens;
  const int32_t *block_table;
  const int32_t *context_lens;
  int32_t *err;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int num_seqs;
  int layer;
  int total_tokens;        // rows of q and out
  float qscale;
  // test hook (pa_prefill_set_test_fault): the chunk of CTA 0 whose copies
  // are left out (-1: none), and the limit of every wait
  int fault_chunk;
  unsigned long long wait_ns;
};

struct __align__(1024) PSmem {
  unsigned char q[kQBufs][kHalves][kOperandBytes]; // per half [32 tok][4 heads][64], swizzled
  unsigned char k[kStagesP][kOperandBytes];        // [128 keys][64]
  unsigned char v[kStagesP][kOperandBytes];        // [128 keys][64]
  int tile_prefix[kMaxSeqsP + 1];
  int bin_start[kWeightBins];                      // counting sort of the tiles by weight
  uint16_t order[kSortTiles];                      // tiles, heaviest first
  uint8_t tile_bins[kSortTiles];                   // each tile's bin
  uint64_t q_full[kQBufs];
  uint64_t q_empty[kQBufs];
  uint64_t kv_full[kStagesP];
  uint64_t kv_empty[kStagesP];
  uint64_t s_full[kHalves];
  uint64_t s_free[kHalves];                        // the softmax has read S: the next S may land
  uint64_t p_full[kHalves];
  uint64_t o_full[kHalves];
  uint64_t o_free[kHalves];
  uint64_t v_zeroed[kStagesP];                     // zeroing warp -> the other half's MMA warp
  uint64_t staged[kHalves];                        // the half's output rows are in shared memory
  uint64_t mma_done[kHalves];                      // every MMA of the half's warp has completed
  uint32_t tmem_base;
  int pmask[kStagesP];                             // pages of the stage that were loaded
  int warp_sum[kPThreads / 32];
};

static_assert(sizeof(PSmem) + 1024 <= 227 * 1024, "shared memory above the per-CTA limit");

__device__ __forceinline__ float p_neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ float p_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Packed two-lane fp32 add.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Shared -> global 3-D tiled tensor copy (TMA store) in the thread's bulk
// async-group.
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *smem_src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(smem_src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The thread's bulk stores have read their shared-memory source.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// ... and have completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// A work item is (64-token query tile, kv head).  The tiles are ordered by
// weight class (the weight: the 128-key chunks its two halves go through),
// heaviest first, ties in tile order (a stable counting sort every CTA
// computes alike); with more than kSortTiles tiles, by tile index from the
// last (the last tiles of a sequence see the most keys).  The items of that order are dealt out in
// rounds of G, every other round backwards (CTA b takes positions b,
// 2G - 1 - b, 2G + b, ...), so that each CTA's sum of weights comes close to
// the mean; a CTA keeps its pipeline running from one item into the next.
struct Item {
  int g;                    // kv head
  int ctx, row0, t0;        // the tile's sequence: cached tokens, first row; tile start
  int rows0, rows1;         // query tokens of half 0 / half 1 (<= 0: no work)
  int halves;
  int n_keys0, n_keys;      // keys half 0 / the whole tile sees
  int n_chunks, nc0, nc1;   // 128-key chunks: the tile's, half 0's, half 1's
  int s;
};

// The sequence s whose tiles hold tile t: prefix[s] <= t < prefix[s+1].
__device__ __forceinline__ int tile_seq(const PSmem &sm, int num_seqs, int t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sm.tile_prefix[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Sort bin of tile t: kWeightBins - 1 - the class of its weight w, so that
// bins in ascending order hold the tiles heaviest first.  The class is w
// itself below 16 and w's leading four bits with its exponent above (classes
// at most 1/8 wide): a class then holds several tiles of one long sequence,
// which stay in tile order, so the CTAs of one round share more K/V in L2.
__device__ __forceinline__ int tile_bin(const PSmem &sm, const PrefillParams &p, int t) {
  const int s = tile_seq(sm, p.num_seqs, t);
  const long long t0 = static_cast<long long>(t - sm.tile_prefix[s]) * kCtaTok;
  const long long ctx = __ldg(p.context_lens + s);
  const long long n = __ldg(p.cu_tokens + s + 1) - __ldg(p.cu_tokens + s);
  const long long r0 = min(static_cast<long long>(kQTok), n - t0);
  const long long r1 = min(static_cast<long long>(kQTok), n - t0 - kQTok);
  long long w = (ctx + t0 + r0 + kChunk - 1) / kChunk;
  if (r1 > 0) w += (ctx + t0 + kQTok + r1 + kChunk - 1) / kChunk;
  w = max(w, 1LL);
  const int e = 63 - __clzll(w);                        // w < 2^62: e <= 61
  const int cls = e < 3 ? static_cast<int>(w) : 8 * (e - 3) + static_cast<int>(w >> (e - 3));
  return kWeightBins - 1 - min(cls, kWeightBins - 1);
}

// Position in the work order of this CTA's k-th item, or -1 past the end.
__device__ __forceinline__ int item_position(int k, int n_items) {
  // the walks stop at the first position past the end, so pos <= n_items +
  // 2 G, which the launch keeps below INT_MAX
  const int G = gridDim.x, b = blockIdx.x;
  const int pos = k * G + ((k & 1) ? G - 1 - b : b);
  return pos < n_items ? pos : -1;
}

// The item at position k of this CTA's walk: its place in the work order,
// tile and sequence, and the sequence's three values in global memory.  The
// roles that are on the pipeline's path fetch the next item while the
// current one runs, so that the loads' latency is not paid between items.
struct ItemRef {
  int i;                      // position in the work order; -1 past the end
  int t, s;                   // tile, sequence
  int ctx, row0, row_end;     // cached tokens; the sequence's rows [row0, row_end)
};

// A load that stays where it is written (the compiler may move a read-only
// __ldg down to its first use, which would put its latency back between
// the items).
__device__ __forceinline__ int load_early(const int32_t *ptr) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

__device__ __forceinline__ ItemRef fetch_item(const PSmem &sm, const PrefillParams &p,
                                              int total_tiles, bool sorted, int k, int n_items) {
  ItemRef r;
  r.i = item_position(k, n_items);
  r.t = r.s = r.ctx = r.row0 = r.row_end = 0;
  if (r.i < 0) return r;
  const int rank = r.i / kHkv;
  r.t = sorted ? static_cast<int>(sm.order[rank]) : total_tiles - 1 - rank;
  r.s = tile_seq(sm, p.num_seqs, r.t);
  // (read-only for the kernel's lifetime: through the non-coherent path)
  r.ctx = load_early(p.context_lens + r.s);
  r.row0 = load_early(p.cu_tokens + r.s);
  r.row_end = load_early(p.cu_tokens + r.s + 1);
  return r;
}

__device__ __forceinline__ Item decode_item(const PSmem &sm, const ItemRef &r) {
  Item it;
  it.g = r.i % kHkv;
  it.s = r.s;
  it.t0 = (r.t - sm.tile_prefix[r.s]) * kCtaTok;
  it.ctx = r.ctx;
  it.row0 = r.row0;
  const int n = r.row_end - r.row0;
  it.rows0 = min(kQTok, n - it.t0);
  it.rows1 = min(kQTok, n - it.t0 - kQTok);
  it.halves = it.rows1 > 0 ? 2 : 1;
  it.n_keys0 = it.ctx + it.t0 + it.rows0;
  it.n_keys = it.halves == 2 ? it.ctx + it.t0 + kQTok + it.rows1 : it.n_keys0;
  it.n_chunks = (it.n_keys + kChunk - 1) / kChunk;
  it.nc0 = (it.n_keys0 + kChunk - 1) / kChunk;
  it.nc1 = it.halves == 2 ? it.n_chunks : 0;
  return it;
}

// Pages of BT tokens: a chunk spans kChunk / BT pages; bit l of a stage's
// pmask says whether its page l was loaded.
template <int BT>
struct PageGeom {
  static constexpr int kPages = kChunk / BT;
  static constexpr int kAll = (1 << kPages) - 1;
};

// Chunk gc (counted over the CTA's items; kbase: its first key within its
// item) has V rows that must be zeroed: rows past the tile's last key or in
// a page that was not loaded meet P = 0 but may hold anything (NaN
// included).
template <int BT>
__device__ __forceinline__ bool chunk_needs_zero(const PSmem &sm, int gc, int kbase, int n_keys) {
  return sm.pmask[gc % kStagesP] != PageGeom<BT>::kAll || kbase + kChunk > n_keys;
}

// MMA warp: waits until chunk gc has landed (every MMA warp does, for every
// chunk of the item, before it releases the stage: so neither warp's release
// can run ahead of the stage's fill).  The zeroing warp clears the rows above
// before any MMA reads the stage and, with `handover`, signals the other
// half's MMA warp through v_zeroed.
template <int BT>
__device__ __forceinline__ bool mma_prepare_chunk(PSmem &sm, int gc, int kbase, int n_keys,
                                                  bool zeroer, bool handover, int lane,
                                                  unsigned long long wait_ns) {
  const int st = gc % kStagesP;
  int good = 1;
  if (lane == 0) good = mbar_wait_short(&sm.kv_full[st], (gc / kStagesP) & 1, wait_ns) ? 1 : 0;
  good = __shfl_sync(0xffffffffu, good, 0);
  if (!good) return false;
  __syncwarp();
  if (zeroer && chunk_needs_zero<BT>(sm, gc, kbase, n_keys)) {
    const int pm = sm.pmask[st];
    for (int e = lane; e < kChunk * (kTileRowBytes / 16); e += 32) {
      const int key = e >> 3;
      if (kbase + key >= n_keys || !((pm >> (key / BT)) & 1))
        reinterpret_cast<uint4 *>(sm.v[st])[e] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (handover && lane == 0) mbar_arrive(&sm.v_zeroed[st]);
  }
  __syncwarp();
  return true;
}

// S of half h = Q_h K^T for chunk gc into the half's S columns (one thread).
__device__ __forceinline__ void mma_issue_s(PSmem &sm, uint32_t tmem, int qb, int h, int gc,
                                            uint32_t id_s) {
  const uint32_t k_addr = smem_u32(sm.k[gc % kStagesP]);
  const uint32_t q_addr = smem_u32(sm.q[qb][h]);
#pragma unroll
  for (int ks = 0; ks < kD / 16; ++ks)
    tc::mma_bf16(tmem + h * kChunk, tc::sdesc_sw128(q_addr + 32 * ks, 16, 1024),
                 tc::sdesc_sw128(k_addr + 32 * ks, 16, 1024), id_s, ks > 0);
  tc::mma_commit(&sm.s_full[h]);
}

// O of half h += P_h V for chunk gc in the half's O columns (one thread),
// P read from the half's P columns of tensor memory (16 keys = 8 columns per
// k-step); the item's first chunk starts the sum.
__device__ __forceinline__ void mma_issue_pv(PSmem &sm, uint32_t tmem, int h, int gc, bool first,
                                             uint32_t id_o) {
  const uint32_t v_addr = smem_u32(sm.v[gc % kStagesP]);
#pragma unroll
  for (int ks = 0; ks < kChunk / 16; ++ks)
    tc::mma_bf16_ts(tmem + kTmemO + h * kD, tmem + kTmemP + h * (kChunk / 2) + 8 * ks,
                    tc::sdesc_sw128(v_addr + 2048 * ks, 16, 1024), id_o,
                    (!first || ks > 0) ? 1u : 0u);
  tc::mma_commit(&sm.o_full[h]);
}

template <int BT>
__global__ void __launch_bounds__(kPThreads, 1) prefill_attention_kernel(
    const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
    const __grid_constant__ CUtensorMap out_map, PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  PSmem &sm = *reinterpret_cast<PSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    prefetch_tensormap(&kv_map);
    prefetch_tensormap(&q_map);
    prefetch_tensormap(&out_map);
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(&sm.q_full[b], 1);
      // the MMA warps' commits and each softmax half once its output left
      // the buffer (it stages the half's output tile there)
      mbar_init(&sm.q_empty[b], 2 * kHalves);
    }
    for (int st = 0; st < kStagesP; ++st) {
      mbar_init(&sm.kv_full[st], 1);
      mbar_init(&sm.kv_empty[st], kHalves);     // one release per MMA warp
      mbar_init(&sm.v_zeroed[st], 1);
    }
    for (int h = 0; h < kHalves; ++h) {
      mbar_init(&sm.s_full[h], 1);
      mbar_init(&sm.s_free[h], kSoftThreads);
      mbar_init(&sm.p_full[h], kSoftThreads);
      mbar_init(&sm.o_full[h], 1);
      mbar_init(&sm.o_free[h], kSoftThreads);
    }
    for (int h = 0; h < kHalves; ++h) {
      mbar_init(&sm.staged[h], kSoftThreads);
      mbar_init(&sm.mma_done[h], 1);
    }
    fence_mbar_init();
  }
  pdl_launch_dependents();
  pdl_wait_primary();   // q and the cache come from the kernels before

  // ---- query tiles per sequence, laid end to end
  constexpr int kPagesPerChunk = PageGeom<BT>::kPages;
  constexpr unsigned kAllPages = PageGeom<BT>::kAll;
  const long long cap = static_cast<long long>(p.max_blocks) * BT;
  int carry = 0;
  for (int base = 0; base < p.num_seqs; base += kPThreads) {
    const int i = base + tid;
    int tiles = 0;
    if (i < p.num_seqs) {
      const int ctx = p.context_lens[i];
      const int c0 = p.cu_tokens[i], c1 = p.cu_tokens[i + 1];
      const int n = c1 - c0;
      // a chunk that does not fit its table, or rows outside [0, total_tokens), is refused
      if (ctx >= 0 && n >= 0 && c0 >= 0 && c1 <= p.total_tokens &&
          static_cast<long long>(ctx) + n <= cap)
        tiles = (n + kCtaTok - 1) / kCtaTok;
      else if (blockIdx.x == 0)
        report(p.err, PA_DEV_CTX_RANGE);
    }
    int incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    int before = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < kPThreads / 32; ++w) {
      const int v = sm.warp_sum[w];
      if (w < warp) before += v;
      chunk += v;
    }
    if (i < p.num_seqs) sm.tile_prefix[i + 1] = carry + before + incl;
    carry += chunk;
    __syncthreads();
  }
  if (tid == 0) sm.tile_prefix[0] = 0;
  const int total_tiles = carry;
  const int n_items = total_tiles * kHkv;
  __syncthreads();
  if (static_cast<int>(blockIdx.x) >= n_items) return;

  // ---- the tiles heaviest first: a stable counting sort by weight
  const bool sorted = total_tiles <= kSortTiles;
  if (sorted) {
    for (int b = tid; b < kWeightBins; b += kPThreads) sm.bin_start[b] = 0;
    __syncthreads();
    for (int t = tid; t < total_tiles; t += kPThreads) {
      const int bn = tile_bin(sm, p, t);
      sm.tile_bins[t] = static_cast<uint8_t>(bn);
      atomicAdd(&sm.bin_start[bn], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // exclusive prefix sum over the bins (16 consecutive bins per lane)
      constexpr int kPer = kWeightBins / 32;
      int cnt[kPer];
      int sum = 0;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        cnt[e] = sm.bin_start[lane * kPer + e];
        sum += cnt[e];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - sum;
#pragma unroll
      for (int e = 0; e < kPer; ++e) {
        sm.bin_start[lane * kPer + e] = run;
        run += cnt[e];
      }
      __syncwarp();
      // 32 tiles at a time in tile order: a tile's place is its bin's next
      // free place plus the number of lower lanes with the same bin
      for (int base = 0; base < total_tiles; base += 32) {
        const int t = base + lane;
        const int bn = t < total_tiles ? static_cast<int>(sm.tile_bins[t]) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, bn);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        const int at = t < total_tiles ? sm.bin_start[bn] + rank : 0;
        __syncwarp();
        if (t < total_tiles) {
          sm.order[at] = static_cast<uint16_t>(t);
          if (rank == 0) sm.bin_start[bn] += __popc(peers);
        }
        __syncwarp();
      }
    }
    __syncthreads();
  }

  if (warp == kMmaWarp) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;
  if (warp >= 8) {
    // the producer/MMA warpgroup gives registers to the softmax warpgroups
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp == kProducerWarp) {
      // ===================================================== producer warp ==
      bool ok = true;
      int gc = 0, k = 0;
      uint32_t issued = 0, issued_parity = 0;   // per stage: used / parity of its last fill
      // Lane l < kPagesPerChunk holds the block id of page l of a chunk.  The ids of the
      // next chunk (of this item or the next) are read while this chunk's
      // copies are issued, so the table read is off the producer's path.
      auto chunk_ids = [&](const Item &x, int j) -> int {
        const int32_t *row =
            p.block_table + (static_cast<size_t>(x.s) * p.n_layers + p.layer) * p.max_blocks;
        const int pg = j * kPagesPerChunk + (lane & (kPagesPerChunk - 1));
        return (lane < kPagesPerChunk && pg * BT < x.n_keys) ? row[pg] : -1;
      };
      int blk_next = -1;
      bool next_read = false;
      for (; ok; ++k) {
        const ItemRef ref = fetch_item(sm, p, total_tiles, sorted, k, n_items);
        if (ref.i < 0) break;
        const Item it = decode_item(sm, ref);
        if (!next_read && it.n_chunks > 0) blk_next = chunk_ids(it, 0);
        next_read = false;
        int good = 1;
        if (lane == 0) {
          // Q buffer k % 2: the MMAs of the item before last have read it
          const int qb = k % kQBufs;
          if (k >= kQBufs && !mbar_wait(&sm.q_empty[qb], (k / kQBufs - 1) & 1, p.wait_ns)) {
            good = 0;
          } else {
            mbar_arrive_expect_tx(&sm.q_full[qb], it.halves * kOperandBytes);
            for (int h = 0; h < it.halves; ++h)
              tma_load_3d(sm.q[qb][h], &q_map, 0, it.g * kGqa, it.row0 + it.t0 + h * kQTok,
                          &sm.q_full[qb]);
          }
        }
        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        for (int j = 0; j < it.n_chunks && ok; ++j, ++gc) {
          const int st = gc % kStagesP;
          const uint32_t ph = (gc / kStagesP) & 1;
          const int pg = j * kPagesPerChunk + (lane & (kPagesPerChunk - 1));
          const bool needed = lane < kPagesPerChunk && pg * BT < it.n_keys;
          const int blk = blk_next;
          if (j + 1 < it.n_chunks) {
            blk_next = chunk_ids(it, j + 1);
          } else {
            const ItemRef nr = fetch_item(sm, p, total_tiles, sorted, k + 1, n_items);
            if (nr.i >= 0) {
              const Item nx = decode_item(sm, nr);
              if (nx.n_chunks > 0) blk_next = chunk_ids(nx, 0);
              next_read = true;
            }
          }
          const bool valid = needed && blk >= 0 && blk < p.num_blocks;
          const unsigned vm = __ballot_sync(0xffffffffu, valid) & kAllPages;
          const unsigned nm = __ballot_sync(0xffffffffu, needed) & kAllPages;
          good = 1;
          if (lane == 0) {
            if (!mbar_wait(&sm.kv_empty[st], ph ^ 1, p.wait_ns)) {
              good = 0;
            } else {
              if (vm != nm) report(p.err, PA_DEV_BAD_BLOCK);
              sm.pmask[st] = static_cast<int>(vm);
              mbar_arrive_expect_tx(&sm.kv_full[st], __popc(vm) * 2 * BT * kTileRowBytes);
              issued |= 1u << st;
              issued_parity = (issued_parity & ~(1u << st)) | (ph << st);
            }
          }
          ok = __shfl_sync(0xffffffffu, good, 0) != 0;
          if (!ok) break;
          __syncwarp();
          // lane l < 2 kPagesPerChunk: the K rows (l < kPagesPerChunk) or the
          // V rows of page l mod kPagesPerChunk
          const int pl = lane & (kPagesPerChunk - 1), kv = (lane / kPagesPerChunk) & 1;
          const int pblk = __shfl_sync(0xffffffffu, blk, pl);
          // (test hook: CTA 0 leaves this chunk's copies out, so that the
          // waits on it run out)
          const bool fault = p.fault_chunk == gc && blockIdx.x == 0;
          if (!fault && lane < 2 * kPagesPerChunk && ((vm >> pl) & 1u)) {
            unsigned char *dst = (kv ? sm.v[st] : sm.k[st]) + pl * BT * kTileRowBytes;
            tma_load_5d(dst, &kv_map, 0, it.g, 0, kv, pblk, &sm.kv_full[st]);
          }
        }
      }
      if (lane == 0) {
        if (!ok) report(p.err, PA_DEV_TIMEOUT);
        // no copy may still be landing in shared memory when the CTA exits
        for (int kk = max(0, k - kQBufs); kk < k; ++kk)
          if (!mbar_wait(&sm.q_full[kk % kQBufs], (kk / kQBufs) & 1, p.wait_ns)) report(p.err, PA_DEV_TIMEOUT);
        for (int st = 0; st < kStagesP; ++st)
          if ((issued >> st) & 1u)
            if (!mbar_wait(&sm.kv_full[st], (issued_parity >> st) & 1u, p.wait_ns))
              report(p.err, PA_DEV_TIMEOUT);
      }
      __syncwarp();
    } else if (warp < kMmaWarp + kHalves) {
      // ======================================================== MMA warps ==
      const int h = warp - kMmaWarp;     // the half whose MMAs this warp issues
      const uint32_t id_s = tc::idesc_bf16(kRows, kChunk, false);
      const uint32_t id_o = tc::idesc_bf16(kRows, kD, true);
      int ok = 1;
      int gc = 0, k = 0;
      int n_p = 0;             // P chunks of this half consumed
      int n_active = 0;        // items in which the half had work
      uint32_t vz_parity = 0;  // per stage: parity of the next zeroing hand-over
      int n_s = 0;             // S chunks issued
      // Lane 0 waits on the mbarriers and the warp takes its result; the
      // MMAs and commits are issued by one elected lane of the converged
      // warp, which keeps the tensor core fed at its own rate.
      int qb = 0;              // the item's Q buffer
      // S of chunk gcs once the softmax has read the previous S (whole warp)
      auto issue_s = [&](int gcs) -> bool {
        int good = 1;
        if (lane == 0 && n_s > 0 && !mbar_wait_short(&sm.s_free[h], (n_s - 1) & 1, p.wait_ns)) good = 0;
        if (!__shfl_sync(0xffffffffu, good, 0)) return false;
        tc::fence_after_sync();
        if (tc::elect_one()) mma_issue_s(sm, tmem, qb, h, gcs, id_s);
        __syncwarp();
        ++n_s;
        return true;
      };
      ItemRef ref = fetch_item(sm, p, total_tiles, sorted, 0, n_items);
      for (; ok; ++k) {
        if (ref.i < 0) break;
        const Item it = decode_item(sm, ref);
        qb = k % kQBufs;
        const int nch = h == 0 ? it.nc0 : it.nc1;
        // half 1 sees every chunk of a two-half tile, half 0 every chunk of
        // a one-half tile: that half's warp zeroes, and with two halves hands
        // the chunks half 0 also reads over to it
        const bool zeroer = h == (it.halves == 2 ? 1 : 0);
        if (lane == 0) ok = mbar_wait_short(&sm.q_full[qb], (k / kQBufs) & 1, p.wait_ns) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) ok = mma_prepare_chunk<BT>(sm, gc, 0, it.n_keys, zeroer, it.halves == 2 && it.nc0 > 0, lane,
                                           p.wait_ns);
        if (ok && nch > 0) ok = issue_s(gc) ? 1 : 0;
        // the next item's loads are in flight while this item's chunks run
        ref = fetch_item(sm, p, total_tiles, sorted, k + 1, n_items);
        for (int j = 0; j < it.n_chunks && ok; ++j, ++gc) {
          if (j + 1 < it.n_chunks &&
              !mma_prepare_chunk<BT>(sm, gc + 1, (j + 1) * kChunk, it.n_keys, zeroer,
                                 it.halves == 2 && j + 1 < it.nc0, lane, p.wait_ns)) {
            ok = 0;
            break;
          }
          if (j < nch) {
            int good = 1;
            if (j + 1 < nch && !issue_s(gc + 1)) good = 0;
            if (lane == 0) {
              const int st = gc % kStagesP;
              // the half's previous item has read its O (the first PV clears it)
              if (good && j == 0 && n_active > 0 &&
                  !mbar_wait_short(&sm.o_free[h], (n_active - 1) & 1, p.wait_ns))
                good = 0;
              // the half's softmax has written P
              if (good && !mbar_wait_short(&sm.p_full[h], n_p & 1, p.wait_ns)) good = 0;
              // V rows zeroed by the other half's warp
              if (good && !zeroer && chunk_needs_zero<BT>(sm, gc, j * kChunk, it.n_keys)) {
                if (!mbar_wait_short(&sm.v_zeroed[st], (vz_parity >> st) & 1u, p.wait_ns)) good = 0;
                vz_parity ^= 1u << st;
              }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (good) {
              tc::fence_after_sync();
              if (tc::elect_one()) mma_issue_pv(sm, tmem, h, gc, j == 0, id_o);
              __syncwarp();
            }
            ++n_p;
            ok = good;
          }
          if (ok && tc::elect_one()) tc::mma_commit(&sm.kv_empty[gc % kStagesP]);
          __syncwarp();
        }
        if (ok && tc::elect_one()) tc::mma_commit(&sm.q_empty[qb]);   // every MMA that reads Q is issued
        __syncwarp();
        if (nch > 0) ++n_active;
      }
      if (!ok && lane == 0) report(p.err, PA_DEV_TIMEOUT);
      // the tensor core has finished every MMA this warp issued before the
      // TMEM columns go back (after a time-out too)
      if (tc::elect_one()) tc::mma_commit(&sm.mma_done[h]);
      __syncwarp();
      if (lane == 0 && !mbar_wait(&sm.mma_done[h], 0, p.wait_ns)) report(p.err, PA_DEV_TIMEOUT);
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoft));
    // ==================================================== softmax warps ==
    // O accumulates in TMEM.  Each row keeps the reference maximum m its
    // P values are taken against; it moves (and O, l are rescaled) only
    // when a chunk's maximum exceeds it by more than kRescale (log2 units),
    // so P stays below 2^kRescale and most chunks touch O not at all.
    // S_{j+1} is issued before PV_j, so O (for a rescale) and the P
    // columns are touched only once PV_{j-1}'s commit is there.
    constexpr float kRescale = 8.f;
    const int h = tid >> 7;                   // half
    const int r = tid & (kRows - 1);          // MMA row = TMEM lane
    const int tok = r >> 2, hh = r & 3;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_addr + h * kChunk, o_addr = lane_addr + kTmemO + h * kD;
    const uint32_t p_addr = lane_addr + kTmemP + h * (kChunk / 2);
    bool ok = true;
    int gc = 0, n_s = 0, n_o = 0;   // S chunks read; PV commits waited for
    int n_staged = 0;               // output tiles staged
    // Thread r == 0: the Q buffer its last output store reads from, released
    // to the producer only after the next item's first P (the store has read
    // it long before), so that the wait for the read is off the warp's path.
    int pend_qb = -1;
    auto release_stored = [&]() {
      if (pend_qb >= 0) {
        bulk_wait_group_read0();
        mbar_arrive(&sm.q_empty[pend_qb]);
        pend_qb = -1;
      }
    };
    ItemRef ref = fetch_item(sm, p, total_tiles, sorted, 0, n_items);
    for (int k = 0; ok; ++k) {
      if (ref.i < 0) break;
      const Item it = decode_item(sm, ref);
      // the next item's loads are in flight while this item's chunks run
      ref = fetch_item(sm, p, total_tiles, sorted, k + 1, n_items);
      const int rows = h == 0 ? it.rows0 : it.rows1;
      const int nch = h == 0 ? it.nc0 : it.nc1;
      const int qb = k % kQBufs;
      if (nch == 0) {
        // nothing staged: release the Q buffer, once it holds this item's Q
        // (an earlier arrival would count for the item before last)
        if (r == 0) {
          release_stored();
          ok = mbar_wait_short(&sm.q_full[qb], (k / kQBufs) & 1, p.wait_ns);
          if (ok) mbar_arrive(&sm.q_empty[qb]);
        }
        gc += it.n_chunks;
        continue;
      }
      const int first_pos = it.ctx + it.t0 + h * kQTok;   // the half's first query position
      const int last_pos = first_pos + rows - 1;
      const int qpos = min(first_pos + tok, last_pos);
      float m = p_neg_inf(), l = 0.f;
      for (int j = 0; j < nch; ++j) {
        const int st = (gc + j) % kStagesP;
        if (!mbar_wait_short(&sm.s_full[h], n_s & 1, p.wait_ns) ||
            !mbar_wait_short(&sm.kv_full[st], ((gc + j) / kStagesP) & 1, p.wait_ns)) {
          ok = false;
          break;
        }
        ++n_s;
        tc::fence_after_sync();
        const int pm = sm.pmask[st];
        const int kbase = j * kChunk;
        // every key of the chunk is visible to every row of the half and was loaded
        const bool full = pm == static_cast<int>(kAllPages) && kbase + kChunk - 1 <= first_pos;
        const int lim = qpos - kbase;           // keys c <= lim are at or before the row
        uint32_t v[kChunk];
#pragma unroll
        for (int c0 = 0; c0 < kChunk; c0 += 32)
          tc::tmem_ld32(s_addr + c0, *reinterpret_cast<uint32_t(*)[32]>(&v[c0]));
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        mbar_arrive(&sm.s_free[h]);             // S_{j+1} may land in the S columns
        if (!full) {
          // masked keys: -inf (loaded K rows past the tile or in a missing page may be anything)
#pragma unroll
          for (int c = 0; c < kChunk; ++c)
            if (!((c <= lim) && ((pm >> (c / BT)) & 1))) v[c] = 0xff800000u;
        }
        // row maximum: 8 chains of three-input maxima over keys q, q+8, ..
        float mx8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mx8[q] = p_neg_inf();
#pragma unroll
        for (int c = 0; c < kChunk; c += 16)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            mx8[q] = fmax3(mx8[q], __uint_as_float(v[c + q]), __uint_as_float(v[c + 8 + q]));
        const float mc = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * p.qscale;
        const bool move = mc > m + kRescale || (m == p_neg_inf() && mc != p_neg_inf());
        bool pv_done = j == 0;                  // PV_{j-1} complete: O stable, P columns read
        if (__any_sync(0xffffffffu, move) && j > 0) {
          if (!mbar_wait_short(&sm.o_full[h], n_o & 1, p.wait_ns)) {
            ok = false;
            break;
          }
          ++n_o;
          pv_done = true;
          tc::fence_after_sync();
          // rescale O (the whole warp takes part in the TMEM round trip)
          const float alpha = move ? p_exp2(m - mc) : 1.f;
#pragma unroll 1
          for (int c0 = 0; c0 < kD; c0 += 32) {
            uint32_t ov[32];
            tc::tmem_ld32(o_addr + c0, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tc::tmem_st32(o_addr + c0, ov);
          }
          tc::tmem_st_wait();
          l *= alpha;
        }
        if (move) m = mc;
        const float base = (m == p_neg_inf()) ? 0.f : m;
        const float2 qs2 = make_float2(p.qscale, p.qscale), nb2 = make_float2(-base, -base);
        // P = exp2(s * qscale - m) in bf16 pairs (key 2c in the low half of
        // column c) into the half's P columns of tensor memory; 4 partial sums
        float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        uint32_t pw[kChunk / 2];
#pragma unroll
        for (int ch = 0; ch < kChunk / 8; ++ch) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = 8 * ch + 2 * q;
            const float2 x = fma2(make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                  qs2, nb2);
            const float e0 = p_exp2(x.x), e1 = p_exp2(x.y);
            ls[q] = add2(ls[q], make_float2(e0, e1));
            pw[c >> 1] = float2_to_bf16x2(e0, e1);
          }
        }
        if (!pv_done) {
          if (!mbar_wait_short(&sm.o_full[h], n_o & 1, p.wait_ns)) {
            ok = false;
            break;
          }
          ++n_o;
          tc::fence_after_sync();
        }
        tc::tmem_st32(p_addr, *reinterpret_cast<uint32_t(*)[32]>(&pw[0]));
        tc::tmem_st32(p_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pw[32]));
        l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
        tc::tmem_st_wait();
        tc::fence_before_sync();    // P, for the tensor core
        mbar_arrive(&sm.p_full[h]);
        if (j == 0) release_stored();
      }
      if (!ok) break;
      // O is complete once the item's last PV is
      if (!mbar_wait_short(&sm.o_full[h], n_o & 1, p.wait_ns)) {
        ok = false;
        break;
      }
      ++n_o;
      tc::fence_after_sync();
      uint32_t ov[kD];
      tc::tmem_ld32(o_addr, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
      tc::tmem_ld32(o_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&sm.o_free[h]);   // the next item's first PV may clear O
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      auto row_chunk = [&](int e) {
        const float *f = reinterpret_cast<const float *>(&ov[8 * e]);
        return make_uint4(float2_to_bf16x2(f[0] * inv, f[1] * inv),
                          float2_to_bf16x2(f[2] * inv, f[3] * inv),
                          float2_to_bf16x2(f[4] * inv, f[5] * inv),
                          float2_to_bf16x2(f[6] * inv, f[7] * inv));
      };
      if (rows == kQTok) {
        // a whole half tile: the rows go into the half's part of this item's
        // Q buffer (no MMA reads it any more), in the layout of the output's
        // tensor map (row r, 16-byte chunk e at e ^ (r mod 8)), and leave in
        // one TMA store, whose writes are whole 128-byte lines
        unsigned char *stg = sm.q[qb][h] + r * kTileRowBytes;
#pragma unroll
        for (int e = 0; e < kD / 8; ++e)
          *reinterpret_cast<uint4 *>(stg + ((e ^ (r & 7)) << 4)) = row_chunk(e);
        fence_proxy_async_smem();
        mbar_arrive(&sm.staged[h]);
        if (r == 0) {
          ok = mbar_wait_short(&sm.staged[h], n_staged & 1, p.wait_ns);
          if (ok) {
            release_stored();
            tma_store_3d(&out_map, sm.q[qb][h], 0, it.g * kGqa, it.row0 + it.t0 + h * kQTok);
            bulk_commit_group();
            pend_qb = qb;
          }
        }
        ++n_staged;
      } else {
        if (tok < rows) {
          uint4 *dst = reinterpret_cast<uint4 *>(
              p.out + ((static_cast<size_t>(it.row0) + it.t0 + h * kQTok + tok) * kHq +
                       it.g * kGqa + hh) * kD);
#pragma unroll
          for (int e = 0; e < kD / 8; ++e) dst[e] = row_chunk(e);
        }
        if (r == 0) {
          release_stored();
          mbar_arrive(&sm.q_empty[qb]);
        }
      }
      gc += it.n_chunks;
    }
    if (!ok) report(p.err, PA_DEV_TIMEOUT);
    release_stored();
    if (r == 0) bulk_wait_group0();   // the output stores are complete
  }
  // every TMEM read and MMA is done (or given up on) before the columns go back
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Tensor map over q [total_tokens][32][64] bf16: box (64, 4 heads, 32 tokens)
// = one GQA group's rows of a half tile, 128-byte swizzle; rows past the
// end read as zeros.
int make_q_map(CUtensorMap *map, const void *q, int total_tokens) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return PA_ERR_CUDA;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  const cuuint64_t dims[3] = {kD, kHq, static_cast<cuuint64_t>(total_tokens)};
  const cuuint64_t strides[2] = {kHeadRowBytes, static_cast<cuuint64_t>(kHq) * kHeadRowBytes};
  const cuuint32_t box[3] = {kD, kGqa, kQTok};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult rr = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rr == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

namespace {

int g_pf_fault_chunk = -1;                     // test hook, see pa_prefill_set_test_fault
unsigned long long g_pf_fault_wait_ns = kWaitLimitNs;

template <int BT>
int prefill_attention_impl(uint16_t *out, const uint16_t *q, int total_tokens,
                           const int32_t *cu_tokens, const uint16_t *kv_cache, int num_blocks,
                           const int32_t *block_table, int n_layers, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs, int layer, float scale,
                           int32_t *err, void *stream) {
  if (num_seqs < 0 || num_seqs > kMaxSeqsP || total_tokens < 0 || num_blocks <= 0 ||
      n_layers <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * BT > INT_MAX) return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0 || total_tokens == 0) return PA_OK;
  if (!out || !q || !cu_tokens || !kv_cache || !block_table || !context_lens || !err)
    return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache)) return PA_ERR_ALIGN;
  if (!(scale > 0.f) || scale > 3.0e38f) return PA_ERR_ARG;   // the row maximum is taken before scaling
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;

  static bool attr_done[64] = {};
  const size_t smem = sizeof(PSmem) + 1024;
  if (!attr_done[di.device]) {
    if (cudaFuncSetAttribute(prefill_attention_kernel<BT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[di.device] = true;
  }
  // the pool's map (one page's K or V rows per copy) changes with the pool,
  // q's with q and the token count
  static thread_local const void *map_pool = nullptr;
  static thread_local int map_blocks = 0;
  alignas(64) static thread_local CUtensorMap kv_map;
  if (map_pool != kv_cache || map_blocks != num_blocks) {
    rc = make_kv_rows_map_bt(&kv_map, kv_cache, num_blocks, BT);
    if (rc != PA_OK) return rc;
    map_pool = kv_cache;
    map_blocks = num_blocks;
  }
  static thread_local const void *map_out = nullptr;
  static thread_local int map_out_tokens = 0;
  alignas(64) static thread_local CUtensorMap out_map;
  if (map_out != out || map_out_tokens != total_tokens) {
    rc = make_q_map(&out_map, out, total_tokens);   // out has q's layout
    if (rc != PA_OK) return rc;
    map_out = out;
    map_out_tokens = total_tokens;
  }
  static thread_local const void *map_q = nullptr;
  static thread_local int map_q_tokens = 0;
  alignas(64) static thread_local CUtensorMap q_map;
  if (map_q != q || map_q_tokens != total_tokens) {
    rc = make_q_map(&q_map, q, total_tokens);
    if (rc != PA_OK) return rc;
    map_q = q;
    map_q_tokens = total_tokens;
  }
  // every sequence's chunk ends in at most one partial tile; one CTA per SM
  // works through the (tile, kv head) items
  const long long tiles = (static_cast<long long>(total_tokens) + kCtaTok - 1) / kCtaTok + num_seqs;
  const int grid = static_cast<int>(min(static_cast<long long>(di.sm_count), tiles * kHkv));
  if (tiles * kHkv + 2LL * grid > INT_MAX) return PA_ERR_ARG;   // item positions stay in int
  PrefillParams prm;
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.cu_tokens = cu_tokens;
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.layer = layer;
  prm.total_tokens = total_tokens;
  prm.qscale = scale * kLog2eP;
  prm.fault_chunk = g_pf_fault_chunk;
  prm.wait_ns = g_pf_fault_chunk >= 0 ? g_pf_fault_wait_ns : kWaitLimitNs;
  if (launch_pdl(prefill_attention_kernel<BT>, dim3(static_cast<unsigned>(grid)),
                 dim3(kPThreads), smem, static_cast<cudaStream_t>(stream), kv_map, q_map, out_map,
                 prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" int pa_prefill_set_test_fault(int chunk, long long wait_limit_ns) {
  if (chunk < -1 || (chunk >= 0 && (wait_limit_ns < 1000 || wait_limit_ns > 1000000000LL)))
    return PA_ERR_ARG;
  g_pf_fault_chunk = chunk;
  g_pf_fault_wait_ns = chunk >= 0 ? static_cast<unsigned long long>(wait_limit_ns) : kWaitLimitNs;
  return PA_OK;
}

extern "C" int pa_prefill_attention(uint16_t *out, const uint16_t *q, int total_tokens,
                                    const int32_t *cu_tokens, const uint16_t *kv_cache,
                                    int num_blocks, const int32_t *block_table, int n_layers,
                                    int max_blocks_per_seq, const int32_t *context_lens,
                                    int num_seqs, int layer, float scale, int32_t *err,
                                    void *stream) {
  return prefill_attention_impl<kBs>(out, q, total_tokens, cu_tokens, kv_cache, num_blocks,
                                     block_table, n_layers, max_blocks_per_seq, context_lens,
                                     num_seqs, layer, scale, err, stream);
}

extern "C" int pa_prefill_attention_bt(uint16_t *out, const uint16_t *q, int total_tokens,
                                       const int32_t *cu_tokens, const uint16_t *kv_cache,
                                       int num_blocks, int block_tokens,
                                       const int32_t *block_table, int n_layers,
                                       int max_blocks_per_seq, const int32_t *context_lens,
                                       int num_seqs, int layer, float scale, int32_t *err,
                                       void *stream) {
  switch (block_tokens) {
    case 8:
      return prefill_attention_impl<8>(out, q, total_tokens, cu_tokens, kv_cache, num_blocks,
                                       block_table, n_layers, max_blocks_per_seq, context_lens,
                                       num_seqs, layer, scale, err, stream);
    case 16:
      return prefill_attention_impl<16>(out, q, total_tokens, cu_tokens, kv_cache, num_blocks,
                                        block_table, n_layers, max_blocks_per_seq, context_lens,
                                        num_seqs, layer, scale, err, stream);
    case 32:
      return prefill_attention_impl<32>(out, q, total_tokens, cu_tokens, kv_cache, num_blocks,
                                        block_table, n_layers, max_blocks_per_seq, context_lens,
                                        num_seqs, layer, scale, err, stream);
    default:
      return PA_ERR_ARG;
  }
}
