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
// One CTA per (32-token query tile, kv head): its 128 MMA rows are the 32
// tokens x the 4 q heads of the GQA group (row = 4 * token + head), so every
// K/V byte brought into shared memory serves 128 query rows.  Keys go in
// chunks of 128 (8 pages).  Warp roles (192 threads):
//   warp 4      producer: the Q tile (one TMA), then per chunk 16 TMA copies
//               (K rows and V rows of 8 pages) into a 3-stage ring;
//   warp 5      one thread issues the MMAs: S_j = Q K_j^T (M 128, N 128, 4
//               k-steps) into one of two TMEM buffers, and, once the
//               softmax has written P_j, O_j = P_j V_j (M 128, N 64, 8
//               k-steps, V read as an MN-major operand) into a third;
//   warps 0-3   softmax, one thread per row (TMEM lane): S_j from TMEM,
//               causal mask, running max and sum in fp32 (log2 domain), P_j
//               rounded to bf16 into shared memory (128-byte swizzle, the
//               layout the MMA reads), the previous chunk's O_j folded into
//               registers with the max correction, and the output row at the
//               end.
// S_{j+1} is computed while the softmax works on S_j.
#include <climits>
#include <cudaTypedefs.h>

#include "pa_device.cuh"
#include "pa_host.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kQTok = 32;                     // query tokens per CTA
constexpr int kRows = kQTok * kGqa;           // 128 MMA rows
constexpr int kChunk = 128;                   // keys per chunk
constexpr int kPagesPerChunk = kChunk / kBs;  // 8
constexpr int kStagesP = 3;
constexpr int kSoftWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kPThreads = 6 * 32;
constexpr int kTileRowBytes = kHeadRowBytes;             // 128-byte rows
constexpr int kOperandBytes = kChunk * kTileRowBytes;    // 16 KiB: 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;                      // S x2 (256) + O (64), rounded up
constexpr uint32_t kTmemO = 256;
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
};

struct __align__(1024) PSmem {
  unsigned char q[kOperandBytes];                  // [32 tok][4 heads][64], swizzled
  unsigned char k[kStagesP][kOperandBytes];        // [128 keys][64]
  unsigned char v[kStagesP][kOperandBytes];        // [128 keys][64]
  unsigned char p[2][kOperandBytes];               // P: keys 0-63, 64-127, [128 rows][64]
  int tile_prefix[kMaxSeqsP + 1];
  uint64_t q_full;
  uint64_t kv_full[kStagesP];
  uint64_t kv_empty[kStagesP];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_full;
  uint32_t tmem_base;
  int pmask[kStagesP];                             // pages of the stage that were loaded
  int warp_sum[kPThreads / 32];
  int seq, t0, valid;
};

__device__ __forceinline__ float p_neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ float p_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kPThreads, 1) prefill_attention_kernel(
    const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
    PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  PSmem &sm = *reinterpret_cast<PSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;   // kv head
  if (tid == 0) {
    prefetch_tensormap(&kv_map);
    prefetch_tensormap(&q_map);
    mbar_init(&sm.q_full, 1);
    for (int st = 0; st < kStagesP; ++st) {
      mbar_init(&sm.kv_full[st], 1);
      mbar_init(&sm.kv_empty[st], 1);
    }
    mbar_init(&sm.s_full[0], 1);
    mbar_init(&sm.s_full[1], 1);
    mbar_init(&sm.p_full, kSoftWarps * 32);
    mbar_init(&sm.o_full, 1);
    fence_mbar_init();
  }
  pdl_launch_dependents();
  pdl_wait_primary();   // q and the cache come from the kernels before

  // ---- query tiles per sequence, laid end to end; the last ones go first
  const long long cap = static_cast<long long>(p.max_blocks) * kBs;
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
        tiles = (n + kQTok - 1) / kQTok;
      else if (blockIdx.x == 0 && blockIdx.y == 0)
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
  const int total_tiles = carry;
  if (tid == 0) {
    sm.tile_prefix[0] = 0;
    sm.valid = 0;
    const int t = total_tiles - 1 - static_cast<int>(blockIdx.x);
    if (t >= 0) {
      int lo = 0, hi = p.num_seqs - 1;   // the sequence s with prefix[s] <= t < prefix[s+1]
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.tile_prefix[mid] <= t) lo = mid;
        else hi = mid - 1;
      }
      sm.seq = lo;
      sm.t0 = (t - sm.tile_prefix[lo]) * kQTok;
      sm.valid = 1;
    }
  }
  __syncthreads();
  if (!sm.valid) return;
  const int s = sm.seq;
  const int t0 = sm.t0;
  const int ctx = p.context_lens[s];
  const int row0 = p.cu_tokens[s];
  const int n = p.cu_tokens[s + 1] - row0;
  const int rows = min(kQTok, n - t0);                  // real query tokens of the tile
  const int last_pos = ctx + t0 + rows - 1;             // the tile's last query position
  const int n_keys = last_pos + 1;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;

  if (warp == kMmaWarp) {
    tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ===================================================== producer warp ==
    const int32_t *row =
        p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
    if (lane == 0) {
      mbar_arrive_expect_tx(&sm.q_full, kOperandBytes);
      tma_load_3d(sm.q, &q_map, 0, g * kGqa, row0 + t0, &sm.q_full);
    }
    bool ok = true;
    uint32_t issued = 0, issued_parity = 0;   // per stage: used / parity of its last fill
    for (int j = 0; j < n_chunks && ok; ++j) {
      const int st = j % kStagesP;
      const uint32_t ph = (j / kStagesP) & 1;
      // lane l < 8 looks up page j * 8 + l
      const int pg = j * kPagesPerChunk + (lane & 7);
      int blk = -1;
      const bool needed = lane < kPagesPerChunk && pg * kBs < n_keys;
      if (needed) blk = row[pg];
      const bool valid = needed && blk >= 0 && blk < p.num_blocks;
      const unsigned vm = __ballot_sync(0xffffffffu, valid) & 0xffu;
      const unsigned nm = __ballot_sync(0xffffffffu, needed) & 0xffu;
      int good = 1;
      if (lane == 0) {
        if (!mbar_wait(&sm.kv_empty[st], ph ^ 1)) {
          good = 0;
        } else {
          if (vm != nm) report(p.err, PA_DEV_BAD_BLOCK);
          sm.pmask[st] = static_cast<int>(vm);
          mbar_arrive_expect_tx(&sm.kv_full[st], __popc(vm) * 2 * kBs * kTileRowBytes);
          issued |= 1u << st;
          issued_parity = (issued_parity & ~(1u << st)) | (ph << st);
        }
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) {
        ok = false;
        break;
      }
      __syncwarp();
      // lanes 0-7: K rows of page l; lanes 8-15: V rows of page l - 8
      const int pl = lane & 7, kv = (lane >> 3) & 1;
      const int pblk = __shfl_sync(0xffffffffu, blk, pl);
      if (lane < 16 && ((vm >> pl) & 1u)) {
        unsigned char *dst = (kv ? sm.v[st] : sm.k[st]) + pl * kBs * kTileRowBytes;
        tma_load_5d(dst, &kv_map, 0, g, 0, kv, pblk, &sm.kv_full[st]);
      }
    }
    if (lane == 0) {
      if (!ok) report(p.err, PA_DEV_TIMEOUT);
      // no copy may still be landing in shared memory when the CTA exits
      if (!mbar_wait(&sm.q_full, 0)) report(p.err, PA_DEV_TIMEOUT);
      for (int st = 0; st < kStagesP; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.kv_full[st], (issued_parity >> st) & 1u)) report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ========================================================= MMA warp ==
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_bf16(kRows, kChunk, false);
      const uint32_t id_o = tc::idesc_bf16(kRows, kD, true);
      const uint32_t q_addr = smem_u32(sm.q);
      bool ok = mbar_wait(&sm.q_full, 0);
      auto issue_s = [&](int j) -> bool {
        const int st = j % kStagesP;
        if (!mbar_wait(&sm.kv_full[st], (j / kStagesP) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t k_addr = smem_u32(sm.k[st]);
        const uint32_t d = tmem + (j & 1) * kChunk;
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          tc::mma_bf16(d, tc::sdesc_sw128(q_addr + 32 * ks, 16, 1024),
                       tc::sdesc_sw128(k_addr + 32 * ks, 16, 1024), id_s, ks > 0);
        tc::mma_commit(&sm.s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n_chunks > 1) ok = issue_s(1);
      for (int j = 0; j < n_chunks && ok; ++j) {
        const int st = j % kStagesP;
        // the softmax has written P_j (and read S_j and O_{j-1})
        if (!mbar_wait(&sm.p_full, j & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t v_addr = smem_u32(sm.v[st]);
#pragma unroll
        for (int ks = 0; ks < kChunk / 16; ++ks) {
          const uint32_t pa = smem_u32(sm.p[ks >> 2]) + 32 * (ks & 3);
          tc::mma_bf16(tmem + kTmemO, tc::sdesc_sw128(pa, 16, 1024),
                       tc::sdesc_sw128(v_addr + 2048 * ks, 16, 1024), id_o, ks > 0);
        }
        tc::mma_commit(&sm.o_full);
        tc::mma_commit(&sm.kv_empty[st]);
        if (j + 2 < n_chunks) ok = issue_s(j + 2);
      }
      if (!ok) report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ==================================================== softmax warps ==
    const int r = tid;                        // MMA row = TMEM lane
    const int tok = r >> 2, hh = r & 3;
    const int qpos = min(ctx + t0 + tok, last_pos);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float o[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) o[d] = 0.f;
    float m = p_neg_inf(), l = 0.f, alpha_prev = 1.f;
    bool ok = true;
    for (int j = 0; j < n_chunks; ++j) {
      const int st = j % kStagesP;
      if (!mbar_wait(&sm.s_full[j & 1], (j >> 1) & 1) ||
          !mbar_wait(&sm.kv_full[st], (j / kStagesP) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const int pm = sm.pmask[st];
      const int kbase = j * kChunk;
      // every key of the chunk is visible to every row and was loaded
      const bool full = pm == 0xff && kbase + kChunk - 1 <= ctx + t0;
      const uint32_t s_addr = lane_addr + (j & 1) * kChunk;
      // pass 1: the chunk's row maximum
      float mx = p_neg_inf();
#pragma unroll
      for (int c0 = 0; c0 < kChunk; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(s_addr + c0, v);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int kp = kbase + c0 + c;
          const bool vis = full || (kp <= qpos && ((pm >> ((c0 + c) >> 4)) & 1));
          mx = vis ? fmaxf(mx, __uint_as_float(v[c]) * p.qscale) : mx;
        }
      }
      const float m_new = fmaxf(m, mx);
      const float alpha = (m_new == p_neg_inf()) ? 1.f : p_exp2(m - m_new);
      const float base = (m_new == p_neg_inf()) ? 0.f : m_new;
      // O_{j-1} into the registers (P_{j-1} has been consumed, P may be rewritten)
      if (j > 0) {
        if (!mbar_wait(&sm.o_full, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(lane_addr + kTmemO + c0, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c0 + c] = fmaf(o[c0 + c], alpha_prev, __uint_as_float(v[c]));
        }
      }
      // keys past the tile's last position, or in a page that was not
      // loaded, meet P = 0 but their V rows may hold anything: zero them
      {
        const int key = r;   // this thread's V row of the stage
        const int kp = kbase + key;
        if (kp >= n_keys || !((pm >> (key >> 4)) & 1)) {
          uint4 *vr = reinterpret_cast<uint4 *>(sm.v[st] + key * kTileRowBytes);
#pragma unroll
          for (int e = 0; e < kTileRowBytes / 16; ++e) vr[e] = make_uint4(0, 0, 0, 0);
        }
      }
      // pass 2: P = exp2(s * qscale - m) in bf16; l sums the rounded values
      float lsum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < kChunk; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(s_addr + c0, v);
        tc::tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int kp = kbase + c0 + c;
          const bool vis0 = full || (kp <= qpos && ((pm >> ((c0 + c) >> 4)) & 1));
          const bool vis1 = full || (kp + 1 <= qpos && ((pm >> ((c0 + c + 1) >> 4)) & 1));
          const float e0 = vis0 ? p_exp2(fmaf(__uint_as_float(v[c]), p.qscale, -base)) : 0.f;
          const float e1 = vis1 ? p_exp2(fmaf(__uint_as_float(v[c + 1]), p.qscale, -base)) : 0.f;
          const uint32_t pk = float2_to_bf16x2(e0, e1);
          const float2 back = bf16x2_to_float2(pk);
          lsum += back.x + back.y;
          packed[c >> 1] = pk;
        }
        // 32 keys = 4 chunks of 16 bytes, in region (c0 / 64), chunk c0 % 64 / 8 + i
        unsigned char *region = sm.p[c0 >> 6] + r * kTileRowBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ch = ((c0 & 63) >> 3) + i;
          *reinterpret_cast<uint4 *>(region + ((ch ^ (r & 7)) << 4)) =
              make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
      l = fmaf(l, alpha, lsum);
      m = m_new;
      alpha_prev = alpha;
      fence_proxy_async_smem();   // P and the zeroed V rows, for the tensor core
      tc::fence_before_sync();
      mbar_arrive(&sm.p_full);
    }
    if (ok && n_chunks > 0) {
      if (mbar_wait(&sm.o_full, (n_chunks - 1) & 1)) {
        tc::fence_after_sync();
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(lane_addr + kTmemO + c0, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c0 + c] = fmaf(o[c0 + c], alpha_prev, __uint_as_float(v[c]));
        }
        if (tok < rows) {
          const float inv = (l > 0.f) ? 1.f / l : 0.f;
          uint4 *dst = reinterpret_cast<uint4 *>(
              p.out + ((static_cast<size_t>(row0) + t0 + tok) * kHq + g * kGqa + hh) * kD);
#pragma unroll
          for (int e = 0; e < kD / 8; ++e)
            dst[e] = make_uint4(float2_to_bf16x2(o[8 * e] * inv, o[8 * e + 1] * inv),
                                float2_to_bf16x2(o[8 * e + 2] * inv, o[8 * e + 3] * inv),
                                float2_to_bf16x2(o[8 * e + 4] * inv, o[8 * e + 5] * inv),
                                float2_to_bf16x2(o[8 * e + 6] * inv, o[8 * e + 7] * inv));
        }
      } else {
        ok = false;
      }
    }
    if (!ok) report(p.err, PA_DEV_TIMEOUT);
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
// = one GQA group's rows of a query tile, 128-byte swizzle; rows past the
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

extern "C" int pa_prefill_attention(uint16_t *out, const uint16_t *q, int total_tokens,
                                    const int32_t *cu_tokens, const uint16_t *kv_cache,
                                    int num_blocks, const int32_t *block_table, int n_layers,
                                    int max_blocks_per_seq, const int32_t *context_lens,
                                    int num_seqs, int layer, float scale, int32_t *err,
                                    void *stream) {
  if (num_seqs < 0 || num_seqs > kMaxSeqsP || total_tokens < 0 || num_blocks <= 0 ||
      n_layers <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * kBs > INT_MAX) return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0 || total_tokens == 0) return PA_OK;
  if (!out || !q || !cu_tokens || !kv_cache || !block_table || !context_lens || !err)
    return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache)) return PA_ERR_ALIGN;
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;

  static bool attr_done[64] = {};
  const size_t smem = sizeof(PSmem) + 1024;
  if (!attr_done[di.device]) {
    if (cudaFuncSetAttribute(prefill_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    rc = make_kv_rows_map(&kv_map, kv_cache, num_blocks);
    if (rc != PA_OK) return rc;
    map_pool = kv_cache;
    map_blocks = num_blocks;
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
  // every sequence's chunk ends in at most one partial tile
  const long long tiles = (static_cast<long long>(total_tokens) + kQTok - 1) / kQTok + num_seqs;
  if (tiles > INT_MAX) return PA_ERR_ARG;
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
  if (launch_pdl(prefill_attention_kernel, dim3(static_cast<unsigned>(tiles), kHkv),
                 dim3(kPThreads), smem, static_cast<cudaStream_t>(stream), kv_map, q_map, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
