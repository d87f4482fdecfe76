// pa_decode.cu -- decode step of PagedAttention for one layer on sm_103a.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "What is in
// the box": pagedAttentionKernel computes one query token's attention over
// K/V stored in 16-token pages found through block_table, with an online
// softmax and __shfl_down_sync reductions; GQA_Q_TO_K_RATIO = 4.
//
// Design (GB300-first, not the page's kernel):
//  * Work is balanced by BLOCKS, not by sequences: the blocks of all
//    sequences are laid end to end and cut into gridDim.x equal ranges, one
//    per CTA ("stream-K" style).  A sequence whose blocks span several CTAs
//    gets one fp32 partial (m, l, acc) per CTA, merged by a second kernel
//    (split-context / flash-decoding merge).  Any length mix keeps every SM
//    busy.
//  * One physical block (16 tokens x 8 kv heads x K,V = 32 KiB, contiguous)
//    is fetched with ONE bulk async copy (TMA, non-tensor form) into a
//    shared-memory stage; a producer warp keeps kStages copies in flight
//    (mbarrier full/empty pipeline).  Each block is read from HBM once and
//    serves all 8 kv heads; each kv head's slice serves its 4 q heads.
//  * Eight consumer warps, one per kv head.  QK: lane (token t, dim quarter)
//    does 16-dim dot products for 4 heads with packed fp32x2 FMAs, then a
//    3-shuffle reduce-scatter leaves one (token, head) score per lane.  The
//    online softmax keeps (m, l) per head in the log2 domain.  PV: lane owns
//    2 output dims for all 4 heads, weights come from shared memory as one
//    broadcast float4 per token.
#include <cfloat>
#include <climits>
#include <cstdio>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kConsumerWarps = kHkv;                       // one per kv head
constexpr int kThreads = (kConsumerWarps + 1) * 32;        // + producer warp
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kScanThreads = kConsumerWarps * 32;          // 256
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kSegStart = 1;   // first block of this CTA's share of a sequence
constexpr int kSegEnd = 2;     // last block of that share
constexpr int kEndOfWork = 4;  // no more blocks; stage carries no data

struct StageDesc {
  int seq;
  int n_valid;   // tokens of the block inside the context, 1..16
  int flags;
  int n_parts;   // CTAs sharing this sequence
};

struct __align__(16) Smem {
  unsigned char kv[kStages][kBlockBytes];          // offset 0: 32 KiB-aligned stages
  float p[kConsumerWarps][kBs][kGqa];              // softmax weights, per warp
  float alpha[kConsumerWarps][kGqa];               // rescale factors, per warp
  StageDesc desc[kStages];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  long long warp_sum[kConsumerWarps];
  long long nb_total;
  long long first_b;
  int first_seq;
};

struct DecodeParams {
  __nv_bfloat16 *out;
  const uint16_t *q;
  const unsigned char *kv;
  const int32_t *block_table;
  const int32_t *context_lens;
  int2 *meta;        // [num_seqs] (first partial slot, number of partials)
  float2 *ml;        // [slots][32] (m, l), m in the log2 domain
  float2 *acc;       // [slots][32][32] unnormalised output, 2 dims per float2
  int32_t *err;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int num_seqs;
  int layer;
  float qscale;      // scale * log2(e), folded into q
};

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Context length clamped into [0, max_blocks * 16].
__device__ __forceinline__ int clamped_ctx(const DecodeParams &p, int s) {
  int t = p.context_lens[s];
  return min(max(t, 0), p.max_blocks * kBs);
}

// CTA whose block range [floor(c*NB/G), floor((c+1)*NB/G)) holds block b.
__device__ __forceinline__ int cta_of(long long b, long long nb_total, int g) {
  return static_cast<int>(((b + 1) * g + nb_total - 1) / nb_total) - 1;
}

__device__ __forceinline__ long long warp_incl_scan(long long v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

struct QRegs {
  float2 a[kGqa][4];   // q pairs matching the lane's first K load
  float2 b[kGqa][4];   // q pairs matching the lane's second K load
};

__device__ __forceinline__ float2 scaled_pair(uint32_t u, float sc) {
  float2 f = bf16x2_to_float2(u);
  return make_float2(f.x * sc, f.y * sc);
}

// Lane (t8 = lane/4, qq = lane%4) handles dims [8qq, 8qq+8) and
// [32+8qq, 32+8qq+8).  Lanes with odd t8 read the upper half first, which
// makes the shared-memory K reads bank-conflict free.
__device__ __forceinline__ void load_q(QRegs &qr, const DecodeParams &p, int s, int g, int lane) {
  const int qq = lane & 3;
  const bool odd = (lane >> 2) & 1;
#pragma unroll
  for (int h = 0; h < kGqa; ++h) {
    const uint4 *row =
        reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(s) * kHq + g * kGqa + h) * kD);
    uint4 lo = __ldg(row + qq);
    uint4 hi = __ldg(row + 4 + qq);
    uint4 A = odd ? hi : lo;
    uint4 B = odd ? lo : hi;
    qr.a[h][0] = scaled_pair(A.x, p.qscale);
    qr.a[h][1] = scaled_pair(A.y, p.qscale);
    qr.a[h][2] = scaled_pair(A.z, p.qscale);
    qr.a[h][3] = scaled_pair(A.w, p.qscale);
    qr.b[h][0] = scaled_pair(B.x, p.qscale);
    qr.b[h][1] = scaled_pair(B.y, p.qscale);
    qr.b[h][2] = scaled_pair(B.z, p.qscale);
    qr.b[h][3] = scaled_pair(B.w, p.qscale);
  }
}

// Score of token t (row of the stage) for this lane's head after the
// reduce-scatter over the 4 lanes that share t.
__device__ __forceinline__ float qk_score(const QRegs &qr, const unsigned char *krow, int lane) {
  const int qq = lane & 3;
  const bool odd = (lane >> 2) & 1;
  const uint4 ka = *reinterpret_cast<const uint4 *>(krow + qq * 16 + (odd ? 64 : 0));
  const uint4 kb = *reinterpret_cast<const uint4 *>(krow + qq * 16 + (odd ? 0 : 64));
  const float2 k0 = bf16x2_to_float2(ka.x), k1 = bf16x2_to_float2(ka.y);
  const float2 k2 = bf16x2_to_float2(ka.z), k3 = bf16x2_to_float2(ka.w);
  const float2 k4 = bf16x2_to_float2(kb.x), k5 = bf16x2_to_float2(kb.y);
  const float2 k6 = bf16x2_to_float2(kb.z), k7 = bf16x2_to_float2(kb.w);
  float v[kGqa];
#pragma unroll
  for (int h = 0; h < kGqa; ++h) {
    float2 acc = make_float2(0.f, 0.f);
    acc = fma2(qr.a[h][0], k0, acc);
    acc = fma2(qr.a[h][1], k1, acc);
    acc = fma2(qr.a[h][2], k2, acc);
    acc = fma2(qr.a[h][3], k3, acc);
    acc = fma2(qr.b[h][0], k4, acc);
    acc = fma2(qr.b[h][1], k5, acc);
    acc = fma2(qr.b[h][2], k6, acc);
    acc = fma2(qr.b[h][3], k7, acc);
    v[h] = acc.x + acc.y;
  }
  // reduce-scatter: after two exchange steps lane qq holds head qq's sum
  const bool b1 = qq & 2;
  float send0 = b1 ? v[0] : v[2];
  float send1 = b1 ? v[1] : v[3];
  float keep0 = b1 ? v[2] : v[0];
  float keep1 = b1 ? v[3] : v[1];
  keep0 += __shfl_xor_sync(0xffffffffu, send0, 2);
  keep1 += __shfl_xor_sync(0xffffffffu, send1, 2);
  const bool b0 = qq & 1;
  float send = b0 ? keep0 : keep1;
  float keep = b0 ? keep1 : keep0;
  keep += __shfl_xor_sync(0xffffffffu, send, 1);
  return keep;
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm) decode_split_kernel(DecodeParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int c = blockIdx.x;
  // everything this kernel reads may come from the previous kernel on the
  // stream; with programmatic launch only the CTA start-up overlaps it
  pdl_wait_primary();

  // ---- total number of blocks over all sequences ---------------------------
  long long mine = 0;
  if (tid < kScanThreads) {
    for (int i = tid; i < p.num_seqs; i += kScanThreads) {
      int t = p.context_lens[i];
      if ((t < 0 || t > p.max_blocks * kBs) && c == 0) report(p.err, PA_DEV_CTX_RANGE);
      mine += (clamped_ctx(p, i) + kBs - 1) / kBs;
    }
    #pragma unroll
    for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
    if (lane == 0) sm.warp_sum[warp] = mine;
  }
  if (tid == 0) sm.first_seq = INT_MAX;
  __syncthreads();
  long long nb_total = 0;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) nb_total += sm.warp_sum[w];
  const int G = static_cast<int>(min(static_cast<long long>(gridDim.x), max(nb_total, 1LL)));
  if (c >= G) return;
  const long long lo = nb_total * c / G;
  const long long hi = nb_total * (c + 1) / G;
  __syncthreads();   // warp_sum is reused below

  // ---- first sequence touching [lo, hi): smallest s with B[s+1] > lo or B[s] >= lo
  long long carry = 0;
  for (int base = 0; base < p.num_seqs; base += kScanThreads) {
    const int i = base + tid;
    long long nb = 0;
    if (tid < kScanThreads && i < p.num_seqs) nb = (clamped_ctx(p, i) + kBs - 1) / kBs;
    long long incl = 0;
    if (tid < kScanThreads) {
      incl = warp_incl_scan(nb, lane);
      if (lane == 31) sm.warp_sum[warp] = incl;
    }
    __syncthreads();
    long long woff = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      long long ws = sm.warp_sum[w];
      if (w < warp) woff += ws;
      chunk += ws;
    }
    const long long b_i = carry + woff + incl - nb;
    const bool cond = tid < kScanThreads && i < p.num_seqs && (b_i + nb > lo || b_i >= lo);
    if (cond) atomicMin(&sm.first_seq, i);
    __syncthreads();
    const int f = sm.first_seq;
    if (f != INT_MAX) {
      if (i == f && tid < kScanThreads) sm.first_b = b_i;
      __syncthreads();
      break;
    }
    carry += chunk;
    __syncthreads();   // warp_sum is rewritten by the next chunk
  }

  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&sm.full[st], 1);
      mbar_init(&sm.empty[st], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int s_first = sm.first_seq == INT_MAX ? p.num_seqs : sm.first_seq;

  if (warp == kConsumerWarps) {
    // ===================================================== producer warp ==
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    uint32_t issued = 0, issued_parity = 0;   // per stage: used / last phase parity
    long long B = (s_first < p.num_seqs) ? sm.first_b : nb_total;
    for (int s = s_first; s < p.num_seqs && ok; ++s) {
      if (B >= hi && c != G - 1) break;
      const int T = clamped_ctx(p, s);
      const int nb = (T + kBs - 1) / kBs;
      if (nb == 0) {
        // empty context: this CTA owns it, the output is zero
        uint4 *o = reinterpret_cast<uint4 *>(p.out + static_cast<size_t>(s) * kHq * kD);
        for (int k = lane; k < kHq * kD * 2 / 16; k += 32) o[k] = make_uint4(0, 0, 0, 0);
        if (lane == 0) p.meta[s] = make_int2(0, 0);
        continue;
      }
      const long long jb = max(lo, B) - B;
      const long long je = min(hi, B + nb) - B;
      const int c_first = cta_of(B, nb_total, G);
      const int c_last = cta_of(B + nb - 1, nb_total, G);
      const int n_parts = c_last - c_first + 1;
      if (c == c_first && lane == 0) p.meta[s] = make_int2(c_first + s, n_parts);
      const int32_t *row =
          p.block_table + (static_cast<size_t>(s) * p.n_layers + p.layer) * p.max_blocks;
      for (long long j0 = jb; j0 < je && ok; j0 += 32) {
        const long long jj = j0 + lane;
        const int my_blk = (jj < je) ? row[jj] : 0;
        const int cnt = static_cast<int>(min(32LL, je - j0));
        for (int k = 0; k < cnt; ++k) {
          const int blk = __shfl_sync(0xffffffffu, my_blk, k);
          const long long j = j0 + k;
          int good = 1;
          if (lane == 0) {
            if (!mbar_wait(&sm.empty[stage], phase ^ 1)) {
              good = 0;
            } else {
              StageDesc d;
              d.seq = s;
              d.n_valid = min(kBs, T - static_cast<int>(j) * kBs);
              d.flags = (j == jb ? kSegStart : 0) | (j == je - 1 ? kSegEnd : 0);
              d.n_parts = n_parts;
              sm.desc[stage] = d;
              if (blk >= 0 && blk < p.num_blocks) {
                mbar_arrive_expect_tx(&sm.full[stage], kBlockBytes);
                bulk_g2s(sm.kv[stage], p.kv + static_cast<size_t>(blk) * kBlockBytes, kBlockBytes,
                         &sm.full[stage]);
              } else {
                report(p.err, PA_DEV_BAD_BLOCK);
                sm.desc[stage].n_valid = -sm.desc[stage].n_valid;   // consumers skip it
                mbar_arrive(&sm.full[stage]);
              }
              issued |= 1u << stage;
              issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
            }
          }
          ok = __shfl_sync(0xffffffffu, good, 0) != 0;
          if (!ok) break;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      B += nb;
    }
    if (lane == 0) {
      if (ok && mbar_wait(&sm.empty[stage], phase ^ 1)) {
        sm.desc[stage].flags = kEndOfWork;
        mbar_arrive(&sm.full[stage]);
        // this arrive is now the stage's last phase; the copy before it on
        // the same stage has completed, or the consumers could not have freed it
        issued |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      } else {
        report(p.err, PA_DEV_TIMEOUT);
      }
      // no copy may still be landing in shared memory when the CTA exits
      for (int st = 0; st < kStages; ++st)
        if ((issued >> st) & 1u)
          if (!mbar_wait(&sm.full[st], (issued_parity >> st) & 1u)) report(p.err, PA_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ===================================================== consumer warps ==
    const int g = warp;                 // kv head
    const int t8 = lane >> 2;           // token within a half block
    const int qq = lane & 3;            // head within the group (after reduce-scatter)
    const unsigned char *khead = nullptr;
    QRegs qr;
    float2 o[kGqa];
    float m = neg_inf(), l = 0.f;
    int stage = 0;
    uint32_t phase = 0;
#pragma unroll
    for (int h = 0; h < kGqa; ++h) o[h] = make_float2(0.f, 0.f);
    while (true) {
      if (!mbar_wait(&sm.full[stage], phase)) {
        report(p.err, PA_DEV_TIMEOUT);
        break;
      }
      const StageDesc d = sm.desc[stage];
      if (d.flags & kEndOfWork) break;
      if (d.flags & kSegStart) {
        load_q(qr, p, d.seq, g, lane);
        m = neg_inf();
        l = 0.f;
#pragma unroll
        for (int h = 0; h < kGqa; ++h) o[h] = make_float2(0.f, 0.f);
      }
      const int n_valid = d.n_valid;
      if (n_valid > 0) {
        khead = sm.kv[stage] + g * kHeadRowBytes;
        // ---- scores of tokens t8 and t8 + 8 for head qq (log2 domain)
        float s0 = qk_score(qr, khead + t8 * kTokRowBytes, lane);
        float s1 = qk_score(qr, khead + (t8 + 8) * kTokRowBytes, lane);
        s0 = (t8 < n_valid) ? s0 : neg_inf();
        s1 = (t8 + 8 < n_valid) ? s1 : neg_inf();
        // ---- online softmax
        float bm = fmaxf(s0, s1);
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float m_new = fmaxf(m, bm);
        const float alpha = fast_exp2(m - m_new);
        const float p0 = fast_exp2(s0 - m_new);
        const float p1 = fast_exp2(s1 - m_new);
        l = l * alpha + p0 + p1;
        m = m_new;
        sm.p[g][t8][qq] = p0;
        sm.p[g][t8 + 8][qq] = p1;
        if (t8 == 0) sm.alpha[g][qq] = alpha;
        __syncwarp();
        // ---- PV: this lane owns dims 2*lane, 2*lane+1 of all 4 heads
        const float4 al = *reinterpret_cast<const float4 *>(sm.alpha[g]);
        o[0] = make_float2(o[0].x * al.x, o[0].y * al.x);
        o[1] = make_float2(o[1].x * al.y, o[1].y * al.y);
        o[2] = make_float2(o[2].x * al.z, o[2].y * al.z);
        o[3] = make_float2(o[3].x * al.w, o[3].y * al.w);
        const unsigned char *vcol = sm.kv[stage] + kHalfBlockBytes + g * kHeadRowBytes + lane * 4;
        if (n_valid == kBs) {
#pragma unroll
          for (int t = 0; t < kBs; ++t) {
            const float4 pw = *reinterpret_cast<const float4 *>(sm.p[g][t]);
            const float2 v = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(vcol + t * kTokRowBytes));
            o[0] = fma2(make_float2(pw.x, pw.x), v, o[0]);
            o[1] = fma2(make_float2(pw.y, pw.y), v, o[1]);
            o[2] = fma2(make_float2(pw.z, pw.z), v, o[2]);
            o[3] = fma2(make_float2(pw.w, pw.w), v, o[3]);
          }
        } else {
          for (int t = 0; t < n_valid; ++t) {
            const float4 pw = *reinterpret_cast<const float4 *>(sm.p[g][t]);
            const float2 v = bf16x2_to_float2(*reinterpret_cast<const uint32_t *>(vcol + t * kTokRowBytes));
            o[0] = fma2(make_float2(pw.x, pw.x), v, o[0]);
            o[1] = fma2(make_float2(pw.y, pw.y), v, o[1]);
            o[2] = fma2(make_float2(pw.z, pw.z), v, o[2]);
            o[3] = fma2(make_float2(pw.w, pw.w), v, o[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[stage]);
      if (d.flags & kSegEnd) {
        // ---- finish this CTA's share of sequence d.seq
        float lt = l;
        lt += __shfl_xor_sync(0xffffffffu, lt, 4);
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
        if (d.n_parts == 1) {
#pragma unroll
          for (int h = 0; h < kGqa; ++h) {
            const float inv = 1.f / __shfl_sync(0xffffffffu, lt, h);
            uint32_t *dst = reinterpret_cast<uint32_t *>(
                p.out + (static_cast<size_t>(d.seq) * kHq + g * kGqa + h) * kD);
            dst[lane] = float2_to_bf16x2(o[h].x * inv, o[h].y * inv);
          }
        } else {
          const size_t slot = static_cast<size_t>(c) + d.seq;
#pragma unroll
          for (int h = 0; h < kGqa; ++h)
            p.acc[(slot * kHq + g * kGqa + h) * (kD / 2) + lane] = o[h];
          if (lane < kGqa) p.ml[slot * kHq + g * kGqa + lane] = make_float2(m, lt);
        }
      }
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  pdl_launch_dependents();
}

// Combines the partials of every sequence split across CTAs.  Grid
// (num_seqs, 32 q heads), 256 threads.  All partials of one (sequence, head)
// are loaded in parallel: first the maxima (one per thread), then the
// weighted accumulators, 8 partials at a time across the warps.
constexpr int kMergeThreads = 256;
constexpr int kMaxParts = 1024;   // the grid never exceeds this many CTAs

__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(DecodeParams p) {
  pdl_wait_primary();
  __shared__ float wpart[kMaxParts];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float2 osum[kMergeThreads / 32][32];
  const int s = blockIdx.x;
  const int h = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int2 mt = p.meta[s];
  const int np = mt.y;
  if (np <= 1) return;
  const size_t slot0 = static_cast<size_t>(mt.x);

  float mloc = neg_inf();
  for (int k = tid; k < np; k += kMergeThreads) mloc = fmaxf(mloc, p.ml[(slot0 + k) * kHq + h].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();

  float lloc = 0.f;
  for (int k = tid; k < np; k += kMergeThreads) {
    const float2 mlk = p.ml[(slot0 + k) * kHq + h];
    const float wk = fast_exp2(mlk.x - M);
    wpart[k] = wk;
    lloc = fmaf(wk, mlk.y, lloc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
  if (lane == 0) red[warp] = lloc;
  __syncthreads();
  float L = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) L += red[w];

  float2 o = make_float2(0.f, 0.f);
  constexpr int kGroups = kMergeThreads / 32;
#pragma unroll 4
  for (int k = warp; k < np; k += kGroups) {
    const float2 a = p.acc[((slot0 + k) * kHq + h) * (kD / 2) + lane];
    const float wk = wpart[k];
    o.x = fmaf(wk, a.x, o.x);
    o.y = fmaf(wk, a.y, o.y);
  }
  osum[warp][lane] = o;
  __syncthreads();
  if (warp == 0) {
    float2 t = osum[0][lane];
#pragma unroll
    for (int w = 1; w < kGroups; ++w) {
      t.x += osum[w][lane].x;
      t.y += osum[w][lane].y;
    }
    const float inv = 1.f / L;
    uint32_t *dst = reinterpret_cast<uint32_t *>(p.out + (static_cast<size_t>(s) * kHq + h) * kD);
    dst[lane] = float2_to_bf16x2(t.x * inv, t.y * inv);
  }
}

int g_grid_limit = 0;

struct WsLayout {
  size_t meta_off, ml_off, acc_off, total;
};

constexpr size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int num_seqs, long long slots) {
  WsLayout w;
  w.meta_off = 0;
  w.ml_off = align256(sizeof(int2) * static_cast<size_t>(num_seqs));
  w.acc_off = w.ml_off + align256(sizeof(float2) * kHq * static_cast<size_t>(slots));
  w.total = w.acc_off + align256(sizeof(float) * kHq * kD * static_cast<size_t>(slots));
  return w;
}

int auto_grid(const DeviceInfo &di, int num_seqs, int max_blocks) {
  long long g = static_cast<long long>(di.sm_count) * kCtasPerSm;
  if (g_grid_limit > 0) g = min(g, static_cast<long long>(g_grid_limit));
  g = min(g, static_cast<long long>(num_seqs) * max_blocks);
  g = min(g, static_cast<long long>(kMaxParts));
  return static_cast<int>(max(g, 1LL));
}

}  // namespace

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

extern "C" size_t pa_decode_workspace_size(int num_seqs, int max_blocks_per_seq) {
  if (num_seqs <= 0 || max_blocks_per_seq <= 0) return 0;
  DeviceInfo di;
  if (current_device(&di) != PA_OK) di.sm_count = 1024;   // generous when no device answers
  const int G = auto_grid(di, num_seqs, max_blocks_per_seq);
  return ws_layout(num_seqs, static_cast<long long>(G) + num_seqs).total;
}

extern "C" int pa_decode_set_grid_limit(int max_ctas) {
  if (max_ctas < 0) return PA_ERR_ARG;
  g_grid_limit = max_ctas;
  return PA_OK;
}

extern "C" int pa_decode_attention(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                                   int num_blocks, const int32_t *block_table, int n_layers,
                                   int max_blocks_per_seq, const int32_t *context_lens,
                                   int num_seqs, int layer, float scale, void *workspace,
                                   size_t workspace_bytes, int32_t *err, void *stream) {
  if (num_seqs < 0 || num_blocks <= 0 || n_layers <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * kBs > INT_MAX) return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !kv_cache || !block_table || !context_lens || !err) return PA_ERR_NULL;
  if (!workspace) return PA_ERR_WORKSPACE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(kv_cache) || !aligned16(workspace))
    return PA_ERR_ALIGN;
  DeviceInfo di;
  int rc = current_device(&di);
  if (rc != PA_OK) return rc;

  int G = auto_grid(di, num_seqs, max_blocks_per_seq);
  WsLayout w = ws_layout(num_seqs, static_cast<long long>(G) + num_seqs);
  while (w.total > workspace_bytes && G > 1) {
    G = G / 2;
    w = ws_layout(num_seqs, static_cast<long long>(G) + num_seqs);
  }
  if (w.total > workspace_bytes) return PA_ERR_WORKSPACE;

  static bool attr_done[64] = {};
  const size_t smem = sizeof(Smem);
  if (!attr_done[di.device]) {
    if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return PA_ERR_CUDA;
    attr_done[di.device] = true;
  }

  DecodeParams prm;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  prm.out = reinterpret_cast<__nv_bfloat16 *>(out);
  prm.q = q;
  prm.kv = reinterpret_cast<const unsigned char *>(kv_cache);
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.meta = reinterpret_cast<int2 *>(ws + w.meta_off);
  prm.ml = reinterpret_cast<float2 *>(ws + w.ml_off);
  prm.acc = reinterpret_cast<float2 *>(ws + w.acc_off);
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.layer = layer;
  prm.qscale = scale * kLog2e;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_pdl(decode_split_kernel, dim3(G), dim3(kThreads), smem, st, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(decode_merge_kernel, dim3(num_seqs, kHq), dim3(kMergeThreads), 0, st, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
