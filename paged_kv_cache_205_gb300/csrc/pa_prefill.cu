// pa_prefill.cu -- causal attention of a prompt chunk over its sequence's
// paged cache (the prefill side of the paged path) on sm_103a.
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
// One CTA per (16-token query tile, kv head).  A producer warp streams the
// kv head's [K|V][16 tokens][64] tiles of blocks 0..(last position)/16 with
// TMA tensor copies into a ring of stages; four consumer warps, one per q
// head of the GQA group, each own the tile's 16 query rows and run m16n8k16
// bf16 MMAs with every row real: S = Q K^T (8 MMAs per block), a causal mask
// on the diagonal blocks, the online softmax in fp32 (log2 domain), O += P V
// (8 MMAs).  The tiles of one sequence are read by all its query tiles and
// stay L2-resident.
#include <climits>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kQTile = 16;                         // query tokens per CTA
constexpr int kPWarps = kGqa;                      // consumer warps: one per q head of the group
constexpr int kPThreads = (kPWarps + 1) * 32;
constexpr int kPStages = 8;
constexpr int kTileBytes = 2 * kBs * kHeadRowBytes;   // K and V of one kv head: 4 KiB
constexpr int kMaxSeqsP = 2048;
constexpr float kLog2eP = 1.4426950408889634f;

struct PrefillParams {
  __nv_bfloat16 *out;
  const uint16_t *q;
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
  unsigned char kv[kPStages][kTileBytes];
  int tile_prefix[kMaxSeqsP + 1];
  int blk_of_stage[kPStages];   // < 0: the block was not loaded
  uint64_t full[kPStages];
  uint64_t empty[kPStages];
  int warp_sum[kPThreads / 32];
  int seq, t0, valid;
};

__device__ __forceinline__ float p_neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ float p_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kPThreads) prefill_attention_kernel(
    const __grid_constant__ CUtensorMap kv_map, PrefillParams p) {
  extern __shared__ unsigned char smem_raw[];
  PSmem &sm = *reinterpret_cast<PSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;   // kv head
  if (tid == 0) {
    prefetch_tensormap(&kv_map);
    for (int st = 0; st < kPStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kPWarps);
    }
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
        tiles = (n + kQTile - 1) / kQTile;
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
      sm.t0 = (t - sm.tile_prefix[lo]) * kQTile;
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
  const int rows = min(kQTile, n - t0);
  const int last_pos = ctx + t0 + rows - 1;   // the tile's last query position
  const int n_blocks = last_pos / kBs + 1;

  if (warp == kPWarps) {
    // ===================================================== producer warp ==
    const int32_t *row =
        p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
    uint32_t issued = 0, issued_parity = 0;
    bool ok = true;
    for (int j0 = 0; j0 < n_blocks && ok; j0 += 32) {
      const int my_blk = (j0 + lane < n_blocks) ? row[j0 + lane] : 0;
      const int cnt = min(32, n_blocks - j0);
      for (int e = 0; e < cnt; ++e) {
        const int j = j0 + e;
        const int stage = j % kPStages;
        const uint32_t phase = (j / kPStages) & 1;
        const int blk = __shfl_sync(0xffffffffu, my_blk, e);
        int good = 1;
        if (lane == 0) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1)) {
            good = 0;
          } else {
            const bool valid = blk >= 0 && blk < p.num_blocks;
            sm.blk_of_stage[stage] = valid ? blk : -1;
            if (valid) {
              mbar_arrive_expect_tx(&sm.full[stage], kTileBytes);
              tma_load_5d(sm.kv[stage], &kv_map, 0, g, 0, 0, blk, &sm.full[stage]);
            } else {
              report(p.err, PA_DEV_BAD_BLOCK);
              mbar_arrive(&sm.full[stage]);
            }
            issued |= 1u << stage;
            issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          }
        }
        ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        if (!ok) break;
      }
    }
    if (lane == 0) {
      if (!ok) report(p.err, PA_DEV_TIMEOUT);
      // no copy may still be landing in shared memory when the CTA exits
      for (int st = 0; st < kPStages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.full[st], (issued_parity >> st) & 1u)) report(p.err, PA_DEV_TIMEOUT);
    }
    return;
  }

  // ===================================================== consumer warps ==
  const int h = g * kGqa + warp;   // q head
  const int r = lane >> 2, c2 = 2 * (lane & 3);
  const int lm_i = lane >> 3, lm_r = lane & 7;
  // the fragment rows r and r + 8 are query tokens t0 + r and t0 + r + 8
  const bool row_a = r < rows, row_b = r + 8 < rows;
  const int qpos_a = ctx + t0 + r, qpos_b = ctx + t0 + r + 8;
  // A fragments per k-step: (row r, k c2), (row r+8, c2), (row r, c2+8), (row r+8, c2+8)
  uint32_t qa[4][4];
  {
    const uint32_t *qra = reinterpret_cast<const uint32_t *>(
        p.q + ((static_cast<size_t>(row0) + t0 + r) * kHq + h) * kD);
    const uint32_t *qrb = reinterpret_cast<const uint32_t *>(
        p.q + ((static_cast<size_t>(row0) + t0 + r + 8) * kHq + h) * kD);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qa[ks][0] = row_a ? __ldg(qra + (16 * ks + c2) / 2) : 0u;
      qa[ks][1] = row_b ? __ldg(qrb + (16 * ks + c2) / 2) : 0u;
      qa[ks][2] = row_a ? __ldg(qra + (16 * ks + 8 + c2) / 2) : 0u;
      qa[ks][3] = row_b ? __ldg(qrb + (16 * ks + 8 + c2) / 2) : 0u;
    }
  }
  float o[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m_a = p_neg_inf(), m_b = p_neg_inf(), l_a = 0.f, l_b = 0.f;
  bool ok = true;
  for (int j = 0; j < n_blocks; ++j) {
    const int stage = j % kPStages;
    const uint32_t phase = (j / kPStages) & 1;
    if (!mbar_wait(&sm.full[stage], phase)) {
      report(p.err, PA_DEV_TIMEOUT);
      ok = false;
      break;
    }
    if (sm.blk_of_stage[stage] >= 0) {
      unsigned char *tile = sm.kv[stage];
      const uint32_t ktile = smem_u32(tile);
      const uint32_t vtile = ktile + kBs * kHeadRowBytes;
      const int n_valid = min(kBs, last_pos + 1 - j * kBs);   // keys any row of the tile may see
      if (n_valid < kBs) {
        // slots past the tile's last position may hold anything (NaN
        // included) and meet P = 0: every warp writes the same zeros over
        // those V rows before it reads them
        uint4 *vrow = reinterpret_cast<uint4 *>(tile + kBs * kHeadRowBytes);
        for (int e = n_valid * 8 + lane; e < kBs * 8; e += 32) vrow[e] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int tok = (lm_i >> 1) * 8 + lm_r;
        const int chunk = 2 * ks + (lm_i & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ktile + tok * kHeadRowBytes + ((chunk ^ lm_r) << 4), b0, b1, b2, b3);
        mma_bf16_16816(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16_16816(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
      // s0: keys j*16 + c2, +1 (rows r, r+8); s1: the same keys + 8
      const int kp = j * kBs + c2;
      const float ninf = p_neg_inf();
      float xa0 = s0[0] * p.qscale, xa1 = s0[1] * p.qscale;
      float xa2 = s1[0] * p.qscale, xa3 = s1[1] * p.qscale;
      float xb0 = s0[2] * p.qscale, xb1 = s0[3] * p.qscale;
      float xb2 = s1[2] * p.qscale, xb3 = s1[3] * p.qscale;
      xa0 = (kp <= qpos_a) ? xa0 : ninf;
      xa1 = (kp + 1 <= qpos_a) ? xa1 : ninf;
      xa2 = (kp + 8 <= qpos_a) ? xa2 : ninf;
      xa3 = (kp + 9 <= qpos_a) ? xa3 : ninf;
      xb0 = (kp <= qpos_b) ? xb0 : ninf;
      xb1 = (kp + 1 <= qpos_b) ? xb1 : ninf;
      xb2 = (kp + 8 <= qpos_b) ? xb2 : ninf;
      xb3 = (kp + 9 <= qpos_b) ? xb3 : ninf;
      float mxa = fmaxf(fmaxf(xa0, xa1), fmaxf(xa2, xa3));
      float mxb = fmaxf(fmaxf(xb0, xb1), fmaxf(xb2, xb3));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
      mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
      mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
      // a row with no visible key so far (only after refused blocks) keeps
      // an empty state: its scale and its exponent base stay finite
      const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
      const float ala = (mna == ninf) ? 1.f : p_exp2(m_a - mna);
      const float alb = (mnb == ninf) ? 1.f : p_exp2(m_b - mnb);
      const float sa = (mna == ninf) ? 0.f : mna, sb = (mnb == ninf) ? 0.f : mnb;
      const uint32_t pa0 = float2_to_bf16x2(p_exp2(xa0 - sa), p_exp2(xa1 - sa));
      const uint32_t pa2 = float2_to_bf16x2(p_exp2(xa2 - sa), p_exp2(xa3 - sa));
      const uint32_t pb0 = float2_to_bf16x2(p_exp2(xb0 - sb), p_exp2(xb1 - sb));
      const uint32_t pb2 = float2_to_bf16x2(p_exp2(xb2 - sb), p_exp2(xb3 - sb));
      // l sums the probabilities as rounded for the P V product
      const float2 fa0 = bf16x2_to_float2(pa0), fa2 = bf16x2_to_float2(pa2);
      const float2 fb0 = bf16x2_to_float2(pb0), fb2 = bf16x2_to_float2(pb2);
      l_a = fmaf(l_a, ala, (fa0.x + fa0.y) + (fa2.x + fa2.y));
      l_b = fmaf(l_b, alb, (fb0.x + fb0.y) + (fb2.x + fb2.y));
      m_a = mna;
      m_b = mnb;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        o[t][0] *= ala;
        o[t][1] *= ala;
        o[t][2] *= alb;
        o[t][3] *= alb;
      }
#pragma unroll
      for (int dp = 0; dp < 4; ++dp) {
        const int tok = (lm_i & 1) * 8 + lm_r;
        const int chunk = 2 * dp + (lm_i >> 1);
        uint32_t v0, v1, v2, v3;
        ldsm_x4_trans(vtile + tok * kHeadRowBytes + ((chunk ^ lm_r) << 4), v0, v1, v2, v3);
        mma_bf16_16816(o[2 * dp], pa0, pb0, pa2, pb2, v0, v1);
        mma_bf16_16816(o[2 * dp + 1], pa0, pb0, pa2, pb2, v2, v3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);
  }
  if (!ok) return;
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
  // l == 0 only when every block the row sees was refused as out of range
  if (row_a) {
    const float inv = (l_a > 0.f) ? 1.f / l_a : 0.f;
    uint32_t *dst = reinterpret_cast<uint32_t *>(
        p.out + ((static_cast<size_t>(row0) + t0 + r) * kHq + h) * kD);
#pragma unroll
    for (int t = 0; t < 8; ++t) dst[(8 * t + c2) / 2] = float2_to_bf16x2(o[t][0] * inv, o[t][1] * inv);
  }
  if (row_b) {
    const float inv = (l_b > 0.f) ? 1.f / l_b : 0.f;
    uint32_t *dst = reinterpret_cast<uint32_t *>(
        p.out + ((static_cast<size_t>(row0) + t0 + r + 8) * kHq + h) * kD);
#pragma unroll
    for (int t = 0; t < 8; ++t) dst[(8 * t + c2) / 2] = float2_to_bf16x2(o[t][2] * inv, o[t][3] * inv);
  }
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
  static thread_local const void *map_pool = nullptr;
  static thread_local int map_blocks = 0;
  alignas(64) static thread_local CUtensorMap map;
  if (map_pool != kv_cache || map_blocks != num_blocks) {
    rc = make_kv_map(&map, kv_cache, num_blocks);
    if (rc != PA_OK) return rc;
    map_pool = kv_cache;
    map_blocks = num_blocks;
  }
  // every sequence's chunk ends in at most one partial tile
  const long long tiles = (static_cast<long long>(total_tokens) + kQTile - 1) / kQTile + num_seqs;
  if (tiles > INT_MAX) return PA_ERR_ARG;
  PrefillParams prm;
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.q = q;
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
                 dim3(kPThreads), smem, static_cast<cudaStream_t>(stream), map, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
