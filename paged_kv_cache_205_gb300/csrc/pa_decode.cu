// pa_decode.cu -- decode step of PagedAttention for one layer on sm_103a.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "What is in
// the box": pagedAttentionKernel computes one query token's attention over
// K/V stored in 16-token pages found through block_table, with an online
// softmax and warp-shuffle reductions; GQA_Q_TO_K_RATIO = 4.
//
// Design (GB300-first, not the page's kernel):
//  * Work is balanced by BLOCKS, not by sequences.  The blocks of all
//    sequences are laid end to end and cut into chunks of C blocks; CTAs take
//    chunks from an atomic counter (the first one is their own index), so a
//    slow SM simply ends up with fewer chunks.  Every (chunk, sequence) piece
//    leaves an fp32 partial (m, l, acc); a second kernel merges the partials
//    of sequences that span several chunks (split-context merge), launched
//    with programmatic dependent launch so its start-up hides under the
//    first kernel's tail.
//  * A producer warp streams whole physical blocks (16 tokens x 8 kv heads x
//    K,V = 32 KiB, one contiguous page) into a ring of shared-memory stages
//    with TMA tensor copies, one 4 KiB copy per kv head; the 128-byte swizzle
//    of the tensor map lays every head's [token][64] tile out so that the
//    warps read it without bank conflicts.  Each block crosses HBM once.
//  * Eight consumer warps, one per kv head.  The 4 query heads of a GQA group
//    are the M rows of m16n8k16 bf16 tensor-core MMAs (rows 4..15 are zero):
//    S = Q K^T and O += P V take 16 MMAs per block, fed by ldmatrix.  The
//    online softmax runs on the S fragments in fp32 (log2 domain, 2 shuffles
//    per block); P is rounded to bf16 for the PV MMA and l sums the rounded
//    weights so numerator and denominator agree.
#include <cfloat>
#include <climits>
#include <cstdio>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <atomic>
#include <mutex>

#include "pa_decode_tile.cuh"
#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kConsumerWarps = kHkv;                       // one per kv head
constexpr int kThreads = (kConsumerWarps + 1) * 32;        // + producer warp
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kScanThreads = kConsumerWarps * 32;          // 256
constexpr int kMaxSeqs = 2048;                             // block prefix kept in shared memory
constexpr int kMaxGrid = 512;
constexpr int kChunksPerCta = 4;                           // average chunks a CTA takes
constexpr int kHeadTileBytes = 2 * kBs * kHeadRowBytes;    // K and V of one kv head: 4 KiB
constexpr int kPrefetchBlocks = 4;                         // first blocks prefetched before the wait
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kSegStart = 1;   // first block of a (chunk, sequence) piece
constexpr int kSegEnd = 2;     // last block of that piece
constexpr int kEndOfWork = 4;  // no more blocks; the stage carries no data

struct StageDesc {
  int seq;
  int n_valid;   // tokens of the tile inside the context, 1..16 (negative: tile skipped)
  int flags;
  int n_parts;   // pieces the sequence is cut into
  int slot;      // partial slot of this piece
  int vmask;     // 8-token pages: rows of the tile that were loaded (bit t = token t)
};

// The unit of work is a 16-token tile of a sequence: one page of 16 tokens,
// two pages of 8, or half a page of 32.  One stage = one tile, as 8 kv-head
// tiles of [K|V][16 tokens][64], each 128-byte row swizzled (16-byte chunk c
// stored at c ^ (token & 7)).
constexpr int kTileTokens = 16;
constexpr int kStageBytes = kHkv * kHeadTileBytes;   // 32 KiB

struct __align__(1024) Smem {
  unsigned char kv[kStages][kStageBytes];
  int prefix[kMaxSeqs + 1];      // prefix[s] = blocks of sequences 0..s-1
  unsigned char tail[kMaxSeqs];  // tokens in the last block of sequence s (1..16)
  StageDesc desc[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int warp_sum[kConsumerWarps];
};

struct DecodeParams {
  __nv_bfloat16 *out;
  const uint16_t *q;
  const unsigned char *kv;   // the pool, for L2 prefetches (loads go through the tensor map)
  const int32_t *block_table;
  const int32_t *context_lens;
  int *chunk_counter;  // zero between calls; reset by the merge kernel
  int2 *meta;          // [num_seqs] (first partial slot, number of partials)
  float2 *ml;          // [slots][32] (m, l), m in the log2 domain
  float2 *acc;         // [slots][32][32] unnormalised output, 2 dims per float2
  int32_t *err;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int num_seqs;
  int layer;
  int cap_tokens;      // max_blocks * tokens per page: the largest context
  float qscale;        // scale * log2(e), applied to the fp32 scores
  long long n_slots;   // partial slots the workspace holds
  // test hook (pa_decode_set_test_fault): the stage of CTA 0 whose copies are
  // left out (-1: none), and the limit of every wait of the split kernel
  int fault_stage;
  unsigned long long wait_ns;
};

__device__ __forceinline__ int clamped_ctx(const DecodeParams &p, int s) {
  const int t = p.context_lens[s];
  return min(max(t, 0), p.cap_tokens);
}

// Chunk length in blocks: about kChunksPerCta chunks per CTA, at least 8
// blocks (or one CTA's fair share when that is smaller).
__device__ __forceinline__ int chunk_blocks(int nb_total, int g) {
  const int fair = (nb_total + g - 1) / g;
  const int min_c = min(8, fair);
  const int c = (nb_total + kChunksPerCta * g - 1) / (kChunksPerCta * g);
  return max(1, max(min_c, c));
}

// First sequence s with prefix[s+1] > b or prefix[s] >= b (a sequence that
// reaches past block b, or an empty one starting at b or later).
__device__ __forceinline__ int first_seq_at(const int *prefix, int n, int b) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid + 1] > b || prefix[mid] >= b) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// Block prefix over all sequences into sm.prefix[1..num_seqs] (prefix[0] is
// set by the caller); returns the total.  Every thread of the CTA calls it.
__device__ __forceinline__ int block_prefix(const DecodeParams &p, Smem &sm, int tid, int warp,
                                            int lane, bool report_range) {
  int carry = 0;
  for (int base = 0; base < p.num_seqs; base += kScanThreads) {
    const int i = base + tid;
    int nb = 0;
    if (tid < kScanThreads && i < p.num_seqs) {
      const int t = p.context_lens[i];
      if (report_range && (t < 0 || t > p.cap_tokens)) report(p.err, PA_DEV_CTX_RANGE);
      nb = (clamped_ctx(p, i) + kBs - 1) / kBs;
    }
    int incl = nb;
    if (tid < kScanThreads) {
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (lane == 31) sm.warp_sum[warp] = incl;
    }
    __syncthreads();
    int before = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const int v = sm.warp_sum[w];
      if (w < warp) before += v;
      chunk += v;
    }
    if (tid < kScanThreads && i < p.num_seqs) sm.prefix[i + 1] = carry + before + incl;
    carry += chunk;
    __syncthreads();
  }
  return carry;
}

// Sequence holding global block b (b < total): smallest s with prefix[s+1] > b.
__device__ __forceinline__ int seq_of_block(const int *prefix, int n, int b) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid + 1] > b) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// Page ids of tile j of a table row, for pages of BT tokens: the tile's page
// (BT = 16), the page holding it (BT = 32, the tile is half of it), or its
// two pages (BT = 8; the second only exists when the tile has more than 8
// tokens, n_pages8 = ceil(context / 8)).
template <int BT>
__device__ __forceinline__ int tile_page(const int32_t *row, int j) {
  return BT == 32 ? row[j >> 1] : (BT == 8 ? row[2 * j] : row[j]);
}

template <int BT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    decode_split_kernel(const __grid_constant__ CUtensorMap kv_map, DecodeParams p) {
  static_assert(BT == 8 || BT == 16 || BT == 32, "pages of 8, 16 or 32 tokens");
  constexpr size_t kPageBytes = static_cast<size_t>(BT) * kTokRowBytes * 2;
  extern __shared__ unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = gridDim.x;
  // ---- before the previous kernel on the stream has finished: nothing is
  // read into registers, only L2 prefetches of what the CTA needs first
  if (tid == 0) {
    prefetch_tensormap(&kv_map);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kConsumerWarps);
    }
    fence_mbar_init();
  }
  for (int i = tid * 32; i < p.num_seqs; i += kThreads * 32) prefetch_l2(p.context_lens + i);
  {
    // this layer's table rows, shared out over the CTAs
    const int row_lines = (p.max_blocks * 4 + 127) / 128;
    for (int i = blockIdx.x * kThreads + tid; i < p.num_seqs * row_lines; i += G * kThreads) {
      const int s = i / row_lines, line = i % row_lines;
      prefetch_l2(p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks +
                  line * 32);
    }
  }
  // A plan from the context lengths as they read now steers L2 prefetches of
  // this CTA's first blocks, so HBM starts streaming while the previous
  // kernel finishes.  The lengths or table may still change: the values only
  // pick which valid pool lines to prefetch; the real plan is made after the
  // wait.
  if (tid == 0) sm.prefix[0] = 0;
  const int nb_spec = block_prefix(p, sm, tid, warp, lane, false);
  {
    if (warp == kConsumerWarps && lane < kPrefetchBlocks && nb_spec > 0) {
      const int c_spec = chunk_blocks(nb_spec, G);
      const int b = blockIdx.x * c_spec + lane;
      if (blockIdx.x < (nb_spec + c_spec - 1) / c_spec && b < min(nb_spec, (blockIdx.x + 1) * c_spec)) {
        const int s = seq_of_block(sm.prefix, p.num_seqs, b);
        const int j = b - sm.prefix[s];
        const int32_t *row =
            p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
        if (j >= 0 && j * kTileTokens < p.cap_tokens) {
          const int blk = tile_page<BT>(row, j);
          if (blk >= 0 && blk < p.num_blocks)
            prefetch_bulk_l2(p.kv + static_cast<size_t>(blk) * kPageBytes, kPageBytes);
          if (BT == 8 && 2 * j + 1 < p.max_blocks) {
            const int blk2 = row[2 * j + 1];
            if (blk2 >= 0 && blk2 < p.num_blocks)
              prefetch_bulk_l2(p.kv + static_cast<size_t>(blk2) * kPageBytes, kPageBytes);
          }
        }
      }
    }
  }
  pdl_launch_dependents();   // the merge kernel may take its place in the queue
  // everything read below may come from the previous kernel on the stream
  pdl_wait_primary();

  // ---- the real plan.  The producer reads the block ids of its first chunk
  // at the places the speculative plan puts them (these reads come after the
  // wait, so they are current) while every thread checks that each
  // sequence's block count still matches the speculative prefix.  If all
  // match, that prefix is the real one and the ids are used as read;
  // otherwise the prefix is rebuilt and the ids are read again.
  int pre_blk = -1, pre_blk2 = -1;
  const int c_spec = nb_spec > 0 ? chunk_blocks(nb_spec, G) : 1;
  const int b_pre = blockIdx.x * c_spec + lane;
  if (warp == kConsumerWarps && nb_spec > 0 && b_pre < min(nb_spec, (blockIdx.x + 1) * c_spec)) {
    const int s = seq_of_block(sm.prefix, p.num_seqs, b_pre);
    const int j = b_pre - sm.prefix[s];
    const int32_t *row =
        p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
    if (j >= 0 && j * kTileTokens < p.cap_tokens) {
      pre_blk = tile_page<BT>(row, j);
      if (BT == 8 && 2 * j + 1 < p.max_blocks) pre_blk2 = row[2 * j + 1];
    }
  }
  int changed = 0;
  for (int i = tid; i < p.num_seqs; i += kThreads) {
    const int t = p.context_lens[i];
    if (blockIdx.x == 0 && (t < 0 || t > p.cap_tokens)) report(p.err, PA_DEV_CTX_RANGE);
    const int tc = min(max(t, 0), p.cap_tokens);
    const int nb = (tc + kBs - 1) / kBs;
    sm.tail[i] = static_cast<unsigned char>(tc - (nb - 1) * kBs);
    changed |= (nb != sm.prefix[i + 1] - sm.prefix[i]);
  }
  const bool plan_kept = __syncthreads_or(changed) == 0;
  const int nb_total = plan_kept ? nb_spec : block_prefix(p, sm, tid, warp, lane, false);
  const int C = chunk_blocks(nb_total, G);
  const int n_chunks = max(1, (nb_total + C - 1) / C);

  if (warp == kConsumerWarps) {
    // ===================================================== producer warp ==
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    uint32_t issued = 0, issued_parity = 0;   // per stage: used / parity of its last phase
    int published = 0;                        // stages published so far
    int k = blockIdx.x;
    while (k < n_chunks && ok) {
      // the next chunk's index is asked for once the chunk's first copy is in
      // flight (every CTA asks at about the same moment, and the answers
      // queue at one L2 address), and lands while the chunk streams
      int next = 0;
      bool asked = false;
      const int b0 = k * C;
      const int b1 = min(nb_total, b0 + C);
      const bool last_chunk = (k == n_chunks - 1);
      for (int s = first_seq_at(sm.prefix, p.num_seqs, b0); s < p.num_seqs && ok; ++s) {
        const int B = sm.prefix[s];
        if (B >= b1 && !last_chunk) break;
        const int nb = sm.prefix[s + 1] - B;
        if (nb == 0) {
          // empty context: the chunk holding its start owns it; output zero
          uint4 *o = reinterpret_cast<uint4 *>(p.out + static_cast<size_t>(s) * kHq * kD);
          for (int e = lane; e < kHq * kD * 2 / 16; e += 32) o[e] = make_uint4(0, 0, 0, 0);
          if (lane == 0) p.meta[s] = make_int2(0, 0);
          continue;
        }
        if (B >= b1) break;   // last chunk: only empty sequences may follow
        const int tail = sm.tail[s];
        const int jb = max(b0, B) - B;
        const int je = min(b1, B + nb) - B;
        const int k_first = B / C;
        const int n_parts = (B + nb - 1) / C - k_first + 1;
        const int slot = k + s;
        if (k == k_first && lane == 0) p.meta[s] = make_int2(k_first + s, n_parts);
        const int32_t *row =
            p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
        for (int j0 = jb; j0 < je && ok; j0 += 32) {
          const int cnt = min(32, je - j0);
          // the first 32 ids of this CTA's first chunk were read with the plan
          const int off0 = B + j0 - b0;
          const bool use_pre =
              plan_kept && k == static_cast<int>(blockIdx.x) && off0 + cnt <= 32;
          int my_blk = 0, my_blk2 = -1;
          if (!use_pre && j0 + lane < je) {
            my_blk = tile_page<BT>(row, j0 + lane);
            // the second 8-token page exists when the tile holds more than 8 tokens
            if (BT == 8 && (j0 + lane < nb - 1 || tail > 8)) my_blk2 = row[2 * (j0 + lane) + 1];
          }
          for (int e = 0; e < cnt; ++e) {
            const int blk = use_pre ? __shfl_sync(0xffffffffu, pre_blk, off0 + e)
                                    : __shfl_sync(0xffffffffu, my_blk, e);
            const int j = j0 + e;
            int blk2 = -1;
            if (BT == 8) {
              blk2 = use_pre ? __shfl_sync(0xffffffffu, pre_blk2, off0 + e)
                             : __shfl_sync(0xffffffffu, my_blk2, e);
            }
            int good = 1;
            if (lane == 0) good = mbar_wait(&sm.empty[stage], phase ^ 1, p.wait_ns) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
              ok = false;
              break;
            }
            const int n_tok = (j == nb - 1) ? tail : kTileTokens;
            const bool valid_a = blk >= 0 && blk < p.num_blocks;
            // 8-token pages: the second page, when the tile reaches into it
            const bool has_b = BT == 8 && n_tok > 8;
            const bool valid_b = has_b && blk2 >= 0 && blk2 < p.num_blocks;
            const bool valid = valid_a || valid_b;
            if (lane == 0) {
              StageDesc d;
              d.seq = s;
              d.n_valid = valid ? n_tok : -n_tok;   // negative: consumers skip it
              d.flags = (j == jb ? kSegStart : 0) | (j == je - 1 ? kSegEnd : 0);
              d.n_parts = n_parts;
              d.slot = slot;
              d.vmask = (valid_a ? 0x00ff : 0) | (valid_b ? 0xff00 : 0);
              sm.desc[stage] = d;
              if (!valid_a || (has_b && !valid_b)) report(p.err, PA_DEV_BAD_BLOCK);
              if (valid) {
                const uint32_t bytes =
                    BT == 8 ? (valid_a ? kStageBytes / 2 : 0) + (valid_b ? kStageBytes / 2 : 0)
                            : kStageBytes;
                mbar_arrive_expect_tx(&sm.full[stage], bytes);
              } else {
                mbar_arrive(&sm.full[stage]);
              }
              issued |= 1u << stage;
              issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
            __syncwarp();
            // test hook: this stage's copies are left out, so its barrier
            // never completes and every wait on it runs out
            const bool fault = p.fault_stage == published && blockIdx.x == 0;
            ++published;
            if (fault) {
              // (no copy)
            } else if (BT == 16) {
              if (valid && lane < kHkv)   // one 4 KiB tile per kv head, 8 lanes in parallel
                tma_load_5d(sm.kv[stage] + lane * kHeadTileBytes, &kv_map, 0, lane, 0, 0, blk,
                            &sm.full[stage]);
            } else if (BT == 32) {
              // K (lanes 0..7) and V (lanes 8..15) halves of the page, 2 KiB each
              if (valid && lane < 2 * kHkv) {
                const int h = lane & 7, kv = lane >> 3;
                tma_load_5d(sm.kv[stage] + h * kHeadTileBytes + kv * (kHeadTileBytes / 2),
                            &kv_map, 0, h, (j & 1) * kTileTokens, kv, blk, &sm.full[stage]);
              }
            } else {
              // K and V of each 8-token page, 1 KiB each: lane = head + 8 * part,
              // part 0/1 = K/V of the first page, 2/3 = K/V of the second
              const int h = lane & 7, part = lane >> 3;
              const bool second = part >= 2;
              const int kv = part & 1;
              if (second ? valid_b : valid_a)
                tma_load_5d(sm.kv[stage] + h * kHeadTileBytes + kv * (kHeadTileBytes / 2) +
                                (second ? kHeadTileBytes / 4 : 0),
                            &kv_map, 0, h, 0, kv, second ? blk2 : blk, &sm.full[stage]);
            }
            if (!asked) {
              if (lane == 0) next = G + atomicAdd(p.chunk_counter, 1);
              asked = true;
            }
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      if (!asked && lane == 0) next = G + atomicAdd(p.chunk_counter, 1);
      k = __shfl_sync(0xffffffffu, next, 0);
      if (k < G) k = n_chunks;   // a counter that was never zeroed
    }
    if (lane == 0) {
      if (ok && mbar_wait(&sm.empty[stage], phase ^ 1, p.wait_ns)) {
        sm.desc[stage].flags = kEndOfWork;
        mbar_arrive(&sm.full[stage]);
        // this arrive is now the stage's last phase; the copy before it on
        // the same stage has landed, or the consumers could not have freed it
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      } else {
        report(p.err, PA_DEV_TIMEOUT);
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (int st = 0; st < kStages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.full[st], (issued_parity >> st) & 1u, p.wait_ns))
            report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ===================================================== consumer warps ==
    const int g = warp;                    // kv head
    const int r = lane >> 2;               // fragment row = q head within the group (0..3 real)
    const int c2 = 2 * (lane & 3);         // fragment column pair
    const bool real_row = r < kGqa;
    uint32_t qa[4], qc[4];                 // Q fragments of the current sequence
    TileState ts;
    ts.reset();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) qa[ks] = qc[ks] = 0u;
    int stage = 0;
    uint32_t phase = 0;
    while (true) {
      if (!mbar_wait(&sm.full[stage], phase, p.wait_ns)) {
        report(p.err, PA_DEV_TIMEOUT);
        break;
      }
      const StageDesc d = sm.desc[stage];
      if (d.flags & kEndOfWork) break;
      if (d.flags & kSegStart) {
        load_q_fragments(p.q + static_cast<size_t>(d.seq) * kHq * kD, g, lane, qa, qc);
        ts.reset();
      }
      const int n_valid = d.n_valid;
      if (n_valid > 0) {
        const uint32_t ktile = smem_u32(sm.kv[stage] + g * kHeadTileBytes);
        const uint32_t vtile = ktile + kBs * kHeadRowBytes;
        // rows to use: the tile's tokens inside the context, less (8-token
        // pages) a page that was out of range
        const unsigned use = (BT == 8) ? (d.vmask & ((1u << n_valid) - 1u)) : 0u;
        attend_tile<BT == 8>(ktile, vtile, n_valid, use, qa, qc, p.qscale, lane, ts);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
      if (d.flags & kSegEnd) {
        // ---- finish this piece of sequence d.seq
        const float lt = row_sum(ts);
        if (real_row) {
          const int h = g * kGqa + r;
          if (d.n_parts == 1) {
            const float inv = 1.f / lt;
            uint32_t *dst = reinterpret_cast<uint32_t *>(
                p.out + (static_cast<size_t>(d.seq) * kHq + h) * kD);
#pragma unroll
            for (int t = 0; t < 8; ++t)
              dst[(8 * t + c2) / 2] = float2_to_bf16x2(ts.out(t, 0) * inv, ts.out(t, 1) * inv);
          } else {
            const size_t slot = static_cast<size_t>(d.slot);
            float2 *dst = p.acc + (slot * kHq + h) * (kD / 2);
#pragma unroll
            for (int t = 0; t < 8; ++t) dst[(8 * t + c2) / 2] = make_float2(ts.out(t, 0), ts.out(t, 1));
            if ((lane & 3) == 0) p.ml[slot * kHq + h] = make_float2(ts.m, lt);
          }
        }
      }
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
}

// Combines the partials of every sequence cut into several pieces, and
// returns the chunk counter to zero for the next call.  Grid (num_seqs, 32
// q heads), kShares warps = interleaved shares of the partials, lane = 2
// dims.  Each thread folds its share into a running (m, l, o) as it loads it
// (one round of independent loads), then the shares are combined in shared
// memory.  There are about 4 partials per CTA of the split kernel in all, so
// a few sequences have many partials each (16 shares) and a larger batch a
// few each (4 shares: small CTAs, which leave room on the SMs for the next
// split kernel's CTAs to start their prefetches).

__device__ __forceinline__ void fold(float mk, float lk, float &m, float &l, float &s_old,
                                     float &s_new) {
  const float mn = fmaxf(m, mk);
  s_old = fast_exp2(m - mn);
  s_new = fast_exp2(mk - mn);
  l = fmaf(l, s_old, lk * s_new);
  m = mn;
}

template <int kShares>
__global__ void __launch_bounds__(kShares * 32) decode_merge_kernel(DecodeParams p) {
  pdl_launch_dependents();   // the next kernel may start its own set-up
  pdl_wait_primary();
  __shared__ float sm_m[kShares], sm_l[kShares];
  __shared__ float2 sm_o[kShares][32];
  const int s = blockIdx.x, h = blockIdx.y;
  const int lane = threadIdx.x & 31, share = threadIdx.x >> 5;
  if (s == 0 && h == 0 && threadIdx.x == 0) *p.chunk_counter = 0;   // the split kernel is done
  const int2 mt = p.meta[s];
  const int np = mt.y;
  if (np <= 1) return;
  // partials left by an aborted or earlier call may name slots beyond this
  // workspace: read none of them (the call has reported its error)
  if (mt.x < 0 || static_cast<long long>(mt.x) + np > p.n_slots) return;
  const size_t slot0 = static_cast<size_t>(mt.x);
  float m = neg_inf(), l = 0.f, so, sn;
  float2 o = make_float2(0.f, 0.f);
  // loads are issued kBatch partials at a time before any of them is folded,
  // so a share costs one L2 round trip per kBatch partials
  constexpr int kBatch = 8;
  for (int k0 = share; k0 < np; k0 += kShares * kBatch) {
    float2 mk[kBatch], a[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int k = k0 + b * kShares;
      if (k < np) {
        mk[b] = p.ml[(slot0 + k) * kHq + h];
        a[b] = p.acc[((slot0 + k) * kHq + h) * (kD / 2) + lane];
      } else {
        mk[b] = make_float2(neg_inf(), 0.f);
        a[b] = make_float2(0.f, 0.f);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (mk[b].x == neg_inf()) continue;
      fold(mk[b].x, mk[b].y, m, l, so, sn);
      o.x = fmaf(o.x, so, a[b].x * sn);
      o.y = fmaf(o.y, so, a[b].y * sn);
    }
  }
  if (lane == 0) {
    sm_m[share] = m;
    sm_l[share] = l;
  }
  sm_o[share][lane] = o;
  __syncthreads();
  if (share == 0) {
    float M = neg_inf();
#pragma unroll
    for (int w = 0; w < kShares; ++w) M = fmaxf(M, sm_m[w]);
    float L = 0.f;
    float2 t = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kShares; ++w) {
      const float sc = fast_exp2(sm_m[w] - M);   // empty shares carry m = -inf: weight 0
      L = fmaf(sm_l[w], sc, L);
      t.x = fmaf(sm_o[w][lane].x, sc, t.x);
      t.y = fmaf(sm_o[w][lane].y, sc, t.y);
    }
    const float inv = 1.f / L;
    uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + (static_cast<size_t>(s) * kHq + h) * kD);
    dst[lane] = float2_to_bf16x2(t.x * inv, t.y * inv);
  }
}


int g_grid_limit = 0;
// max context / mean context (in 16-token tiles) above which a batch counts
// as heavy-tailed for pa_decode_kernel_for_lengths
constexpr double kHeavyTail = 3.0;
int g_fault_stage = -1;                        // test hook, see pa_decode_set_test_fault
unsigned long long g_fault_wait_ns = kWaitLimitNs;
int g_decode_path = 0;   // 0 automatic, 1 split-context kernel, 2 cluster kernel

struct WsLayout {
  size_t counter_off, meta_off, ml_off, acc_off, total;
};

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

long long max_slots(int num_seqs, int grid) {
  return static_cast<long long>(kChunksPerCta) * grid + 2 + num_seqs;
}

WsLayout ws_layout(int num_seqs, long long slots) {
  WsLayout w;
  w.counter_off = 0;
  w.meta_off = 256;
  w.ml_off = w.meta_off + align256(sizeof(int2) * static_cast<size_t>(num_seqs));
  w.acc_off = w.ml_off + align256(sizeof(float2) * kHq * static_cast<size_t>(slots));
  w.total = w.acc_off + align256(sizeof(float) * kHq * kD * static_cast<size_t>(slots));
  return w;
}

// max_tiles: 16-token tiles of the longest context a table row can hold
int auto_grid(const DeviceInfo &di, int num_seqs, int max_tiles) {
  long long g = static_cast<long long>(di.sm_count) * kCtasPerSm;
  if (g_grid_limit > 0) g = min(g, static_cast<long long>(g_grid_limit));
  g = min(g, static_cast<long long>(num_seqs) * max_tiles);
  g = min(g, static_cast<long long>(kMaxGrid));
  return static_cast<int>(max(g, 1LL));
}

// Tensor map over the whole pool: dims (d 64, kv head 8, token 16, K|V 2,
// block), box (64, 1, 16, 2, 1) = one kv head's K and V tiles, 128B swizzle.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

}  // namespace

int make_kv_map(CUtensorMap *map, const void *kv_cache, int num_blocks) {
  return make_kv_map_bt(map, kv_cache, num_blocks, kBs);
}

// Pages of bt tokens: dims (d 64, kv head 8, token bt, K|V 2, block); box one
// kv head's K and V of a 16-token page (64, 1, 16, 2, 1), or, for 8- and
// 32-token pages, one kv head's K or V rows of a tile's page (64, 1, 8 or
// 16, 1, 1).
int make_kv_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const cuuint64_t row = kTokRowBytes;
  const cuuint64_t dims[5] = {kD, kHkv, static_cast<cuuint64_t>(bt), 2,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {kHeadRowBytes, row, row * bt, row * bt * 2};
  const cuuint32_t box_tok = bt == 8 ? 8u : 16u;
  const cuuint32_t box_kv = bt == 16 ? 2u : 1u;
  const cuuint32_t box[5] = {kD, 1, box_tok, box_kv, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_tile_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const cuuint64_t row = kTokRowBytes;
  const cuuint64_t dims[5] = {kD, kHkv, static_cast<cuuint64_t>(bt), 2,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {kHeadRowBytes, row, row * bt, row * bt * 2};
  const cuuint32_t box[5] = {kD, 1, kBs, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_page_map(CUtensorMap *map, const void *kv_cache, int num_blocks) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  // the token dimension comes before the head dimension although its stride
  // is the larger one: the copy then writes each head's token rows together
  const cuuint64_t dims[5] = {kD, kBs, kHkv, 2, static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {kTokRowBytes, kHeadRowBytes, kHalfBlockBytes, kBlockBytes};
  const cuuint32_t box[5] = {kD, kBs, kHkv, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int make_kv_rows_map(CUtensorMap *map, const void *kv_cache, int num_blocks) {
  return make_kv_rows_map_bt(map, kv_cache, num_blocks, kBs);
}

int make_kv_rows_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt) {
  auto fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const cuuint64_t row = kTokRowBytes;
  const cuuint64_t dims[5] = {kD, kHkv, static_cast<cuuint64_t>(bt), 2,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {kHeadRowBytes, row, row * bt, row * bt * 2};
  const cuuint32_t box[5] = {kD, 1, static_cast<cuuint32_t>(bt), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int current_device(DeviceInfo *info) {
  static DeviceInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return PA_ERR_DEVICE;
  DeviceInfo &d = cache[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    if (cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    d = n;
  }
  *info = d;
  if (d.major != 10 || d.minor != 3) return PA_ERR_DEVICE;
  return PA_OK;
}

}  // namespace pa

using namespace pa;

namespace {

bool page_size_ok(int bt) { return bt == 8 || bt == 16 || bt == 32; }

long long max_tiles(int max_blocks_per_seq, int bt) {
  return (static_cast<long long>(max_blocks_per_seq) * bt + kTileTokens - 1) / kTileTokens;
}

}  // namespace

extern "C" size_t pa_decode_workspace_size_bt(int num_seqs, int max_blocks_per_seq,
                                              int block_tokens) {
  if (num_seqs <= 0 || max_blocks_per_seq <= 0 || !page_size_ok(block_tokens)) return 0;
  DeviceInfo di;
  if (current_device(&di) != PA_OK) di.sm_count = kMaxGrid;   // generous when no device answers
  const long long tiles = max_tiles(max_blocks_per_seq, block_tokens);
  const int G = auto_grid(di, num_seqs, static_cast<int>(min(tiles, static_cast<long long>(INT_MAX))));
  return ws_layout(num_seqs, max_slots(num_seqs, G)).total;
}

extern "C" size_t pa_decode_workspace_size(int num_seqs, int max_blocks_per_seq) {
  return pa_decode_workspace_size_bt(num_seqs, max_blocks_per_seq, kBs);
}

extern "C" int pa_decode_set_grid_limit(int max_ctas) {
  if (max_ctas < 0) return PA_ERR_ARG;
  g_grid_limit = max_ctas;
  return PA_OK;
}

extern "C" int pa_decode_kernel_for(int num_seqs, int block_tokens) {
  if (num_seqs < 0 || !page_size_ok(block_tokens)) return PA_ERR_ARG;
  // the per-sequence kernel takes 16-token pages, the per-head one 8, 16 or
  // 32 (with 8, four 1 KiB copies per tile make it slower than the split
  // kernel: only when forced)
  if (g_decode_path == PA_DECODE_SPLIT) return PA_DECODE_SPLIT;
  if (block_tokens == kBs / 2 && g_decode_path == PA_DECODE_AUTO) return PA_DECODE_SPLIT;
  if (g_decode_path == PA_DECODE_SEQ) return block_tokens == kBs ? PA_DECODE_SEQ : PA_DECODE_SPLIT;
  if (g_decode_path == PA_DECODE_CLUSTER) return PA_DECODE_CLUSTER;
  DeviceInfo di;
  const int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  return decode_pair_cluster(num_seqs, di.sm_count, g_grid_limit) > 0 ? PA_DECODE_CLUSTER
                                                                      : PA_DECODE_SPLIT;
}

extern "C" int pa_decode_set_test_fault(int stage, long long wait_limit_ns) {
  if (stage < -1 || (stage >= 0 && (wait_limit_ns < 1000 || wait_limit_ns > 1000000000LL)))
    return PA_ERR_ARG;
  g_fault_stage = stage;
  g_fault_wait_ns = stage >= 0 ? static_cast<unsigned long long>(wait_limit_ns) : kWaitLimitNs;
  return PA_OK;
}

extern "C" int pa_decode_kernel_for_lengths(const int32_t *context_lens, int num_seqs,
                                            int block_tokens) {
  if (num_seqs < 0 || !page_size_ok(block_tokens) || (num_seqs > 0 && !context_lens))
    return PA_ERR_ARG;
  if (num_seqs == 0 || block_tokens == kBs / 2) return PA_DECODE_SPLIT;
  DeviceInfo di;
  const int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  // how far the longest context is above the mean, in 16-token tiles
  long long sum = 0, mx = 0;
  for (int s = 0; s < num_seqs; ++s) {
    const long long t = (static_cast<long long>(max(context_lens[s], 0)) + kBs - 1) / kBs;
    sum += t;
    mx = max(mx, t);
  }
  const double rho = sum > 0 ? static_cast<double>(mx) * num_seqs / static_cast<double>(sum) : 1.0;
  // a few contexts far above the rest: only the split kernel spreads them over the GPU
  if (rho > kHeavyTail) return PA_DECODE_SPLIT;
  if (decode_pair_cluster(num_seqs, di.sm_count, g_grid_limit) > 0) return PA_DECODE_CLUSTER;
  if (block_tokens == kBs && decode_seq_cluster(num_seqs, di.sm_count, g_grid_limit) > 0)
    return PA_DECODE_SEQ;
  return PA_DECODE_SPLIT;
}

extern "C" int pa_decode_set_path(int path) {
  if (path < PA_DECODE_AUTO || path > PA_DECODE_SEQ) return PA_ERR_ARG;
  g_decode_path = path;
  return PA_OK;
}

namespace {

template <int BT>
int decode_attention_impl(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                          int num_blocks, const int32_t *block_table, int n_layers,
                          int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                          int layer, float scale, void *workspace, size_t workspace_bytes,
                          int32_t *err, void *stream, int path) {
  if (num_seqs < 0 || num_seqs > kMaxSeqs || num_blocks <= 0 || n_layers <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  const long long tiles = max_tiles(max_blocks_per_seq, BT);
  if (static_cast<long long>(max_blocks_per_seq) * BT > INT_MAX ||
      static_cast<long long>(num_seqs) * tiles > INT_MAX)
    return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !kv_cache || !block_table || !context_lens || !err) return PA_ERR_NULL;
  if (!workspace) return PA_ERR_WORKSPACE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache) || !aligned16(workspace))
    return PA_ERR_ALIGN;
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;

  int G = auto_grid(di, num_seqs, static_cast<int>(tiles));
  WsLayout w = ws_layout(num_seqs, max_slots(num_seqs, G));
  while (w.total > workspace_bytes && G > 1) {
    G = G / 2;
    w = ws_layout(num_seqs, max_slots(num_seqs, G));
  }
  if (w.total > workspace_bytes) return PA_ERR_WORKSPACE;

  static bool attr_done[64] = {};
  const size_t smem = sizeof(Smem) + 1024;   // + room to align the base to 1 KiB
  if (!attr_done[di.device]) {
    if (cudaFuncSetAttribute(decode_split_kernel<BT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[di.device] = true;
  }

  // the tensor map describes the pool; rebuilt only when the pool changes
  // (one cache per page size: each instance of this function has its own)
  static thread_local const void *map_pool = nullptr;
  static thread_local int map_blocks = 0;
  alignas(64) static thread_local CUtensorMap map;
  if (map_pool != kv_cache || map_blocks != num_blocks) {
    rc = make_kv_map_bt(&map, kv_cache, num_blocks, BT);
    if (rc != PA_OK) return rc;
    map_pool = kv_cache;
    map_blocks = num_blocks;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // a batch whose (sequence, kv head) pairs all fit on the GPU at once runs
  // one cluster per pair (16-token pages)
  if (BT == kBs && path == PA_DECODE_SEQ) {
    static thread_local const void *pmap_pool = nullptr;
    static thread_local int pmap_blocks = 0;
    alignas(64) static thread_local CUtensorMap pmap;
    if (pmap_pool != kv_cache || pmap_blocks != num_blocks) {
      rc = make_kv_page_map(&pmap, kv_cache, num_blocks);
      if (rc != PA_OK) return rc;
      pmap_pool = kv_cache;
      pmap_blocks = num_blocks;
    }
    int c = decode_seq_cluster(num_seqs, di.sm_count, g_grid_limit);
    if (c == 0) c = 1;
    return launch_decode_seq(pmap, out, q, kv_cache, num_blocks, block_table, n_layers,
                             max_blocks_per_seq, context_lens, num_seqs, layer, scale, err, c, st);
  }
  // (16-token pages; with 32-token pages a tile is half a page, with 8 two
  // pages: forced only, see pa_decode_kernel_for)
  if ((BT == kBs && path != PA_DECODE_SPLIT) ||
      (BT == 2 * kBs && (path == PA_DECODE_AUTO || path == PA_DECODE_CLUSTER)) ||
      (BT == kBs / 2 && path == PA_DECODE_CLUSTER)) {
    int c = decode_pair_cluster(num_seqs, di.sm_count, g_grid_limit);
    if (c == 0 && path == PA_DECODE_CLUSTER) c = 1;
    if (c > 0) {
      // 16-token pages: the split kernel's map is the tile map; 8-token pages:
      // its map (one page's K or V rows of a head) serves both kernels
      const CUtensorMap *tmap = &map;
      if (BT == 2 * kBs) {
        static thread_local const void *tmap_pool = nullptr;
        static thread_local int tmap_blocks = 0;
        alignas(64) static thread_local CUtensorMap tile_map;
        if (tmap_pool != kv_cache || tmap_blocks != num_blocks) {
          rc = make_kv_tile_map_bt(&tile_map, kv_cache, num_blocks, BT);
          if (rc != PA_OK) return rc;
          tmap_pool = kv_cache;
          tmap_blocks = num_blocks;
        }
        tmap = &tile_map;
      }
      return launch_decode_pair(*tmap, out, q, num_blocks, BT, block_table, n_layers,
                                max_blocks_per_seq, context_lens, num_seqs, layer, scale, err, c,
                                st);
    }
  }

  DecodeParams prm;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.q = q;
  prm.kv = reinterpret_cast<const unsigned char *>(kv_cache);
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.chunk_counter = reinterpret_cast<int *>(ws + w.counter_off);
  prm.meta = reinterpret_cast<int2 *>(ws + w.meta_off);
  prm.ml = reinterpret_cast<float2 *>(ws + w.ml_off);
  prm.acc = reinterpret_cast<float2 *>(ws + w.acc_off);
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.layer = layer;
  prm.cap_tokens = max_blocks_per_seq * BT;
  prm.qscale = scale * kLog2e;
  prm.n_slots = max_slots(num_seqs, G);
  prm.fault_stage = g_fault_stage;
  prm.wait_ns = g_fault_stage >= 0 ? g_fault_wait_ns : kWaitLimitNs;

  if (launch_pdl(decode_split_kernel<BT>, dim3(G), dim3(kThreads), smem, st, map, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  const cudaError_t e =
      num_seqs >= 8 ? launch_pdl(decode_merge_kernel<4>, dim3(num_seqs, kHq), dim3(4 * 32), 0, st, prm)
                    : launch_pdl(decode_merge_kernel<16>, dim3(num_seqs, kHq), dim3(16 * 32), 0, st, prm);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" int pa_decode_attention(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                                   int num_blocks, const int32_t *block_table, int n_layers,
                                   int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int layer, float scale, void *workspace,
                                   size_t workspace_bytes, int32_t *err, void *stream) {
  return decode_attention_impl<kBs>(out, q, kv_cache, num_blocks, block_table, n_layers,
                                    max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                    workspace, workspace_bytes, err, stream, g_decode_path);
}

namespace pa {

int decode_path_setting() { return g_decode_path; }

int decode_attention_path(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                          int num_blocks, int block_tokens, const int32_t *block_table,
                          int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                          int num_seqs, int layer, float scale, void *workspace,
                          size_t workspace_bytes, int32_t *err, void *stream, int path) {
  switch (block_tokens) {
    case 8:
      return decode_attention_impl<8>(out, q, kv_cache, num_blocks, block_table, n_layers,
                                      max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                      workspace, workspace_bytes, err, stream, path);
    case 16:
      return decode_attention_impl<16>(out, q, kv_cache, num_blocks, block_table, n_layers,
                                       max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                       workspace, workspace_bytes, err, stream, path);
    case 32:
      return decode_attention_impl<32>(out, q, kv_cache, num_blocks, block_table, n_layers,
                                       max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                       workspace, workspace_bytes, err, stream, path);
    default:
      return PA_ERR_ARG;
  }
}

}  // namespace pa

extern "C" int pa_decode_attention_bt(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                                      int num_blocks, int block_tokens,
                                      const int32_t *block_table, int n_layers,
                                      int max_blocks_per_seq, const int32_t *context_lens,
                                      int num_seqs, int layer, float scale, void *workspace,
                                      size_t workspace_bytes, int32_t *err, void *stream) {
  return decode_attention_path(out, q, kv_cache, num_blocks, block_tokens, block_table, n_layers,
                               max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                               workspace, workspace_bytes, err, stream, g_decode_path);
}

// ---------------------------------------------------------------------------
// Decode attention without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// decode step: an engine whose memory map is fixed when it starts, a caller
// that may not call cudaMalloc on its serving thread because that call can
// synchronise the whole device, or a plugin handed only the tensors it works
// on.  For them the split partials live in one file-scope device array that
// every GPU loading this library holds until the process exits.  The array
// is shared by all calls on a device, so calls whose kernels overlap on the
// GPU (two streams, two host threads) race on it and must be serialised by
// the caller.  Its work counter is cleared at the start of every call; the
// rest is rewritten before it is read.
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;   // 16 MiB per device
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of the array on the current device, looked up once per
// device (host code may not use the symbol itself: on the host it names a
// stand-in, not device memory).  Later calls read the cached address without
// taking the lock.
int static_scratch(int device, void **ptr) {
  static std::atomic<void *> addr[64] = {};
  static std::mutex mu;
  void *a = addr[device].load(std::memory_order_acquire);
  if (!a) {
    std::lock_guard<std::mutex> lock(mu);
    a = addr[device].load(std::memory_order_relaxed);
    if (!a) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return PA_ERR_CUDA;
      }
      addr[device].store(p, std::memory_order_release);
      a = p;
    }
  }
  *ptr = a;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_attention_static(uint16_t *out, const uint16_t *q,
                                          const uint16_t *kv_cache, int num_blocks,
                                          const int32_t *block_table, int n_layers,
                                          int max_blocks_per_seq, const int32_t *context_lens,
                                          int num_seqs, int layer, float scale, int32_t *err,
                                          void *stream) {
  if (num_seqs < 0 || num_seqs > PA_STATIC_MAX_SEQS) return PA_ERR_WORKSPACE;
  if (num_seqs == 0) return pa_decode_attention(out, q, kv_cache, num_blocks, block_table, n_layers,
                                                max_blocks_per_seq, context_lens, 0, layer, scale,
                                                nullptr, 0, err, stream);
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  void *scratch = nullptr;
  rc = static_scratch(di.device, &scratch);
  if (rc != PA_OK) return rc;
  // the work counter (first 256 bytes) must read zero when the kernels start
  if (cudaMemsetAsync(scratch, 0, 256, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return pa_decode_attention(out, q, kv_cache, num_blocks, block_table, n_layers,
                             max_blocks_per_seq, context_lens, num_seqs, layer, scale, scratch,
                             kStaticScratchBytes, err, stream);
}
