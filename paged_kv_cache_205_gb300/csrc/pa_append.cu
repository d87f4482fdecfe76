// pa_append.cu -- KV append with Llama-3-scaled RoPE, and block release.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map".  "The path of
// one inference": the KV cache is one allocation cut into 16-token blocks
// numbered by an iota free list (free_blocks), and block_table entries
// start at -1 ("not assigned yet"); init_rope_frequencies(HEAD_DIM,
// MAX_SEQ_LEN, 500000, 32, 1, 4, 8192) sets up RoPE.  "What is in the box":
// RoPE with Llama 3 scaling (ropeKernel_llama3 / ropeKernelDecode).
//
// pa_kv_append_rope is two kernels:
//   append_alloc_kernel  (1 CTA)  serves the sequences whose position starts
//                                 a page, in ascending order, from the back
//                                 of the free list; writes the table entries
//                                 and the new free count.
//   append_store_kernel  (1 CTA per sequence, programmatic dependent launch)
//                                 rotates q and k while the first kernel
//                                 runs, then waits for it and stores K/V in
//                                 the slot the table names.
// pa_prefill_append_rope does the same for a prompt chunk per sequence
// ("The path of one inference": prefill pushes the whole prompt through at
// once; ropeKernel_llama3 is the prefill RoPE).
#include <climits>
#include <cmath>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kScanCta = 1024;
constexpr int kStoreThreads = (kHkv + kHq) * 8;   // 8 threads per head row, 40 rows
constexpr int kStoreRows = 8;                      // token rows per CTA of the prefill store

// Llama-3-scaled RoPE inverse frequencies of the 32 pairs, computed on the
// host in fp64 and passed by value (no device memory involved).
struct RopeFreqs {
  double f[PA_HEAD_DIM / 2];
};

struct AppendParams {
  RopeFreqs freqs;
  const uint16_t *k_new;
  const uint16_t *v_new;
  uint16_t *q;                 // may be null
  unsigned char *kv;
  int32_t *block_table;
  const int32_t *context_lens;
  int32_t *free_list;
  int32_t *free_count;
  int32_t *err;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int num_seqs;
  int layer;
};

__device__ __forceinline__ size_t table_row(int s, int n_layers, int layer, int max_blocks) {
  return (static_cast<size_t>(s) * n_layers + layer) * static_cast<size_t>(max_blocks);
}

// Exclusive prefix count of `flag` over a 1024-thread CTA; also returns the
// CTA total.  `tot` is 32 ints of shared scratch.
__device__ __forceinline__ int cta_exclusive_count(bool flag, int *tot, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int before_in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) tot[warp] = __popc(bal);
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < kScanCta / 32; ++w) {
    const int t = tot[w];
    if (w < warp) before += t;
    all += t;
  }
  __syncthreads();
  *total = all;
  return before + before_in_warp;
}

template <int BT>
__global__ void __launch_bounds__(kScanCta) append_alloc_kernel(AppendParams p) {
  __shared__ int tot[kScanCta / 32];
  pdl_wait_primary();        // the table and free list may come from the previous kernel
  pdl_launch_dependents();   // the store kernel may start its rotations now
  const int cap = p.max_blocks * BT;
  // a count outside [0, num_blocks] never indexes past the free list
  const int fc0 = min(max(*p.free_count, 0), p.num_blocks);
  int served = 0;
  for (int base = 0; base < p.num_seqs; base += kScanCta) {
    const int i = base + threadIdx.x;
    int pos = 0;
    bool need = false;
    if (i < p.num_seqs) {
      pos = p.context_lens[i];
      const bool in_range = pos >= 0 && pos < cap;
      if (!in_range) report(p.err, PA_DEV_CTX_RANGE);
      need = in_range && (pos % BT == 0);
    }
    int chunk = 0;
    const int rank = served + cta_exclusive_count(need, tot, &chunk);
    if (need) {
      int32_t *entry = p.block_table + table_row(i, p.n_layers, p.layer, p.max_blocks) + pos / BT;
      if (rank < fc0) {
        const int blk = p.free_list[fc0 - 1 - rank];
        *entry = blk;
        if (blk < 0 || blk >= p.num_blocks) report(p.err, PA_DEV_BAD_BLOCK);
      } else {
        *entry = -1;   // refused: the page stays unassigned
        report(p.err, PA_DEV_FREE_UNDERFLOW);
      }
    }
    served += chunk;
  }
  if (threadIdx.x == 0) *p.free_count = max(fc0 - served, 0);
}

// Llama 3 rescaling of the RoPE inverse frequency of pair i (head_dim 64):
// theta 500000, factor 32, low_freq_factor 1, high_freq_factor 4, original
// context 8192.  Wavelengths under 8192/4 keep their frequency, those over
// 8192/1 are slowed by the factor, and the band between blends the two
// linearly in 8192/wavelength.  Host code, run once.
RopeFreqs llama3_freqs() {
  RopeFreqs r;
  const double theta = 500000.0, factor = 32.0, low = 1.0, high = 4.0, orig = 8192.0;
  const double two_pi = 6.283185307179586476925;
  for (int i = 0; i < kD / 2; ++i) {
    const double f = std::pow(theta, -static_cast<double>(2 * i) / kD);
    const double wavelen = two_pi / f;
    if (wavelen < orig / high) {
      r.f[i] = f;
    } else if (wavelen > orig / low) {
      r.f[i] = f / factor;
    } else {
      const double w = (orig / wavelen - low) / (high - low);
      r.f[i] = (1.0 - w) * (f / factor) + w * f;
    }
  }
  return r;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint32_t float_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t *>(&h);
}

// Rotate 4 consecutive pairs (d, d + 32), d = 4j..4j+3, of one head row.
__device__ __forceinline__ void rotate4(uint2 lo, uint2 hi, const float2 *cs, int j, uint2 *out_lo,
                                        uint2 *out_hi) {
  const uint32_t lw[2] = {lo.x, lo.y}, hw[2] = {hi.x, hi.y};
  uint32_t ol[2], oh[2];
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t rl = 0, rh = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float a = bf16_bits_to_float((lw[w] >> (16 * half)) & 0xffffu);
      const float b = bf16_bits_to_float((hw[w] >> (16 * half)) & 0xffffu);
      const float2 c = cs[4 * j + 2 * w + half];   // (cos, sin)
      const float ra = fmaf(a, c.x, -b * c.y);
      const float rb = fmaf(b, c.x, a * c.y);
      rl |= float_to_bf16_bits(ra) << (16 * half);
      rh |= float_to_bf16_bits(rb) << (16 * half);
    }
    ol[w] = rl;
    oh[w] = rh;
  }
  *out_lo = make_uint2(ol[0], ol[1]);
  *out_hi = make_uint2(oh[0], oh[1]);
}

// (cos, sin) of the angle pos * f.  The angle is formed and reduced modulo
// 2*pi in fp64, so that positions in the tens of thousands keep their phase.
// The reduction is Cody and Waite's (W. J. Cody, W. Waite, "Software Manual
// for the Elementary Functions", 1980): 2*pi is split into a double head and
// the double nearest to the rest, and k*2*pi is taken off in two fused
// multiply-adds, head first.  The reduced angle (|r| <= pi) goes through
// fp32 sincosf, with a first-order correction for the part of it fp32 could
// not hold.
__device__ __forceinline__ float2 rope_cos_sin(int pos, double f) {
  const double two_pi_hi = 6.283185307179586232, two_pi_lo = 2.4492935982947064e-16;
  const double a = static_cast<double>(pos) * f;
  const double k = rint(a * 0.15915494309189533577);
  const double red = fma(-k, two_pi_lo, fma(-k, two_pi_hi, a));
  const float rf = static_cast<float>(red);
  const float rerr = static_cast<float>(red - static_cast<double>(rf));   // |rerr| <= 2^-23
  float sn, cn;
  sincosf(rf, &sn, &cn);
  return make_float2(fmaf(-sn, rerr, cn), fmaf(cn, rerr, sn));
}

template <int BT>
__global__ void __launch_bounds__(kStoreThreads) append_store_kernel(AppendParams p) {
  constexpr size_t kHalfPageBytes = static_cast<size_t>(BT) * kTokRowBytes;
  constexpr size_t kPageBytes = 2 * kHalfPageBytes;
  __shared__ float2 cs[kD / 2];
  pdl_launch_dependents();   // the next kernel may start its own set-up
  const int s = blockIdx.x;
  const int tid = threadIdx.x;
  const int pos = p.context_lens[s];
  const bool in_range = pos >= 0 && pos < p.max_blocks * BT;
  if (!in_range) {            // reported by the allocation kernel
    pdl_wait_primary();
    return;
  }
  if (tid < kD / 2) cs[tid] = rope_cos_sin(pos, p.freqs.f[tid]);
  __syncthreads();

  const int head = tid >> 3;   // 0..7 k heads, 8..39 q heads
  const int j = tid & 7;
  uint2 klo = make_uint2(0, 0), khi = make_uint2(0, 0);
  if (head < kHkv) {
    const uint16_t *row = p.k_new + (static_cast<size_t>(s) * kHkv + head) * kD;
    const uint2 lo = *reinterpret_cast<const uint2 *>(row + 4 * j);
    const uint2 hi = *reinterpret_cast<const uint2 *>(row + kD / 2 + 4 * j);
    rotate4(lo, hi, cs, j, &klo, &khi);
  } else if (p.q) {
    uint16_t *row = p.q + (static_cast<size_t>(s) * kHq + (head - kHkv)) * kD;
    const uint2 lo = *reinterpret_cast<const uint2 *>(row + 4 * j);
    const uint2 hi = *reinterpret_cast<const uint2 *>(row + kD / 2 + 4 * j);
    uint2 rlo, rhi;
    rotate4(lo, hi, cs, j, &rlo, &rhi);
    *reinterpret_cast<uint2 *>(row + 4 * j) = rlo;
    *reinterpret_cast<uint2 *>(row + kD / 2 + 4 * j) = rhi;
  }
  uint4 v = make_uint4(0, 0, 0, 0);
  if (tid < kTokRowBytes / 16)
    v = reinterpret_cast<const uint4 *>(p.v_new + static_cast<size_t>(s) * kHkv * kD)[tid];

  // the entry of a page that starts now is written by the allocation kernel;
  // an existing page's entry was written before that kernel started
  if (pos % BT == 0) pdl_wait_primary();
  const int blk =
      p.block_table[table_row(s, p.n_layers, p.layer, p.max_blocks) + pos / BT];
  if (blk < 0 || blk >= p.num_blocks) {
    // a new page that was refused or popped invalid is reported by the
    // allocation kernel; an invalid existing entry is reported here
    if (tid == 0 && pos % BT != 0) report(p.err, PA_DEV_BAD_BLOCK);
    pdl_wait_primary();   // this grid ends after the allocation kernel
    return;
  }
  unsigned char *block = p.kv + static_cast<size_t>(blk) * kPageBytes;
  const int slot = pos % BT;
  if (head < kHkv) {
    unsigned char *krow = block + slot * kTokRowBytes + head * kHeadRowBytes;
    *reinterpret_cast<uint2 *>(krow + 8 * j) = klo;
    *reinterpret_cast<uint2 *>(krow + kD + 8 * j) = khi;
  }
  if (tid < kTokRowBytes / 16)
    reinterpret_cast<uint4 *>(block + kHalfPageBytes + slot * kTokRowBytes)[tid] = v;
  pdl_wait_primary();   // this grid ends after the allocation kernel
}

// ------------------------------------------------------------------ prefill
// A prompt chunk per sequence: the tokens of sequence s are rows
// cu_tokens[s] .. cu_tokens[s+1]-1, at positions context_lens[s] + i.
//   prefill_alloc_kernel  (1 CTA)  ranks every page the chunks open over the
//                                  sequences in order and pops them from the
//                                  back of the free list, pages spread over
//                                  the threads.
//   prefill_store_kernel  (1 CTA per 8 token rows, programmatic
//                                  dependent launch) rotates the rows' k and
//                                  q, then stores K/V in the slots the table
//                                  names; the rows' loads are all in flight
//                                  before the table is read.

struct PrefillAppendParams {
  RopeFreqs freqs;
  const uint16_t *k_new;
  const uint16_t *v_new;
  uint16_t *q;                 // may be null
  unsigned char *kv;
  int32_t *block_table;
  const int32_t *cu_tokens;
  const int32_t *context_lens;
  int32_t *free_list;
  int32_t *free_count;
  int32_t *err;
  int total_tokens;
  int num_blocks;
  int n_layers;
  int max_blocks;
  int num_seqs;
  int layer;
};

// Whether sequence s's chunk is accepted: it fits the sequence's table (of
// max_blocks pages of BT tokens) and its rows lie inside [0, total_tokens).
// Sets the context and chunk length.
template <int BT>
__device__ __forceinline__ bool chunk_fits(const PrefillAppendParams &p, int s, int *ctx, int *n) {
  const int c0 = p.cu_tokens[s], c1 = p.cu_tokens[s + 1];
  *ctx = p.context_lens[s];
  *n = c1 - c0;
  return *ctx >= 0 && *n >= 0 && c0 >= 0 && c1 <= p.total_tokens &&
         static_cast<long long>(*ctx) + *n <= static_cast<long long>(p.max_blocks) * BT;
}

template <int BT>
__global__ void __launch_bounds__(kScanCta) prefill_alloc_kernel(PrefillAppendParams p) {
  __shared__ int tot[kScanCta / 32];
  __shared__ int incl_s[kScanCta];    // pages of the batch's sequences up to and including each
  __shared__ int first_s[kScanCta];   // each sequence's first new page
  pdl_wait_primary();        // the table and free list may come from the previous kernel
  pdl_launch_dependents();   // the store kernel may start its rotations now
  const int fc0 = min(max(*p.free_count, 0), p.num_blocks);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int served = 0;
  for (int base = 0; base < p.num_seqs; base += kScanCta) {
    const int s = base + threadIdx.x;
    int ctx = 0, n = 0, first = 0, pages = 0;
    if (s < p.num_seqs) {
      if (!chunk_fits<BT>(p, s, &ctx, &n)) {
        report(p.err, PA_DEV_CTX_RANGE);
      } else {
        first = (ctx + BT - 1) / BT;                 // pages already open
        pages = (ctx + n + BT - 1) / BT - first;     // pages this chunk opens
      }
    }
    // pages are ranked over the sequences in order: a prefix sum
    int incl = pages;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) tot[warp] = incl;
    __syncthreads();
    int before = 0, chunk = 0;
    for (int w = 0; w < kScanCta / 32; ++w) {
      const int t = tot[w];
      if (w < warp) before += t;
      chunk += t;
    }
    incl_s[threadIdx.x] = before + incl;
    first_s[threadIdx.x] = first;
    __syncthreads();
    // every thread takes pages e, e + 1024, ... of the batch: page e belongs
    // to the first sequence k of the batch with incl_s[k] > e
    for (int e = threadIdx.x; e < chunk; e += kScanCta) {
      int lo = 0, hi = kScanCta - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (incl_s[mid] > e) hi = mid;
        else lo = mid + 1;
      }
      const int j = e - (lo > 0 ? incl_s[lo - 1] : 0);
      int32_t *entry =
          p.block_table + table_row(base + lo, p.n_layers, p.layer, p.max_blocks) + first_s[lo] + j;
      const int rank = served + e;
      if (rank < fc0) {
        const int blk = p.free_list[fc0 - 1 - rank];
        *entry = blk;
        if (blk < 0 || blk >= p.num_blocks) report(p.err, PA_DEV_BAD_BLOCK);
      } else {
        *entry = -1;   // refused: the page stays unassigned
        report(p.err, PA_DEV_FREE_UNDERFLOW);
      }
    }
    served += chunk;
    __syncthreads();
  }
  if (threadIdx.x == 0) *p.free_count = max(fc0 - served, 0);
}

template <int BT>
__global__ void __launch_bounds__(kStoreThreads) prefill_store_kernel(PrefillAppendParams p) {
  constexpr size_t kPageBytes = static_cast<size_t>(BT) * 2 * kTokRowBytes;   // K and V
  constexpr size_t kHalfPageBytes = static_cast<size_t>(BT) * kTokRowBytes;
  __shared__ float2 cs[kStoreRows][kD / 2];
  __shared__ int row_seq[kStoreRows];     // -1: the row lies in no accepted chunk
  __shared__ int row_pos[kStoreRows];
  __shared__ int row_open[kStoreRows];    // the sequence's first page opened by this chunk
  __shared__ int row_blk[kStoreRows];     // -1: no valid page for the row
  pdl_launch_dependents();   // the next kernel may start its own set-up
  const int tid = threadIdx.x;
  const int r0 = blockIdx.x * kStoreRows;
  // thread i < kStoreRows: row r0 + i's sequence (the largest s with
  // cu_tokens[s] <= r: an empty chunk's start equals the next one's, so the
  // search passes over it) and position
  if (tid < kStoreRows) {
    const int r = r0 + tid;
    int seq = -1, pos = 0, open = 0;
    if (r < p.total_tokens) {
      int lo = 0, hi = p.num_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_tokens[mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      int ctx, n;
      // a refused chunk is reported by the allocation kernel
      if (chunk_fits<BT>(p, lo, &ctx, &n) && r >= p.cu_tokens[lo] && r < p.cu_tokens[lo + 1]) {
        seq = lo;
        pos = ctx + (r - p.cu_tokens[lo]);
        open = (ctx + BT - 1) / BT;
      }
    }
    row_seq[tid] = seq;
    row_pos[tid] = pos;
    row_open[tid] = open;
  }
  // every row's k / q half-rows and v, in flight before anything waits on them
  const int head = tid >> 3;   // 0..7 k heads, 8..39 q heads
  const int j = tid & 7;
  uint2 lo[kStoreRows], hi[kStoreRows];
  uint4 v[kStoreRows];
#pragma unroll
  for (int i = 0; i < kStoreRows; ++i) {
    const int r = r0 + i;
    lo[i] = hi[i] = make_uint2(0, 0);
    v[i] = make_uint4(0, 0, 0, 0);
    if (r < p.total_tokens) {
      const uint16_t *row = nullptr;
      if (head < kHkv) row = p.k_new + (static_cast<size_t>(r) * kHkv + head) * kD;
      else if (p.q) row = p.q + (static_cast<size_t>(r) * kHq + (head - kHkv)) * kD;
      if (row) {
        lo[i] = *reinterpret_cast<const uint2 *>(row + 4 * j);
        hi[i] = *reinterpret_cast<const uint2 *>(row + kD / 2 + 4 * j);
      }
      if (tid < kTokRowBytes / 16)
        v[i] = reinterpret_cast<const uint4 *>(p.v_new + static_cast<size_t>(r) * kHkv * kD)[tid];
    }
  }
  __syncthreads();
  // (cos, sin) of every row's position; thread i < kStoreRows: the row's page
  for (int e = tid; e < kStoreRows * (kD / 2); e += kStoreThreads) {
    const int i = e / (kD / 2), c = e % (kD / 2);
    if (row_seq[i] >= 0) cs[i][c] = rope_cos_sin(row_pos[i], p.freqs.f[c]);
  }
  if (tid < kStoreRows) {
    int blk = -1;
    const int s = row_seq[tid];
    if (s >= 0) {
      const int page = row_pos[tid] / BT;
      const bool new_page = page >= row_open[tid];
      if (new_page) pdl_wait_primary();   // its entry comes from the allocation kernel
      blk = p.block_table[table_row(s, p.n_layers, p.layer, p.max_blocks) + page];
      if (blk < 0 || blk >= p.num_blocks) {
        // a page of this chunk that was refused or popped invalid is reported
        // by the allocation kernel; an invalid page from before is reported here
        if (!new_page) report(p.err, PA_DEV_BAD_BLOCK);
        blk = -1;
      }
    }
    row_blk[tid] = blk;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kStoreRows; ++i) {
    if (row_seq[i] < 0) continue;
    uint2 rlo, rhi;
    if (head < kHkv || p.q) rotate4(lo[i], hi[i], cs[i], j, &rlo, &rhi);
    if (head >= kHkv && p.q) {   // q rotates in place whether or not the row's page is valid
      uint16_t *row = p.q + (static_cast<size_t>(r0 + i) * kHq + (head - kHkv)) * kD;
      *reinterpret_cast<uint2 *>(row + 4 * j) = rlo;
      *reinterpret_cast<uint2 *>(row + kD / 2 + 4 * j) = rhi;
    }
    const int blk = row_blk[i];
    if (blk < 0) continue;
    unsigned char *block = p.kv + static_cast<size_t>(blk) * kPageBytes;
    const int slot = row_pos[i] % BT;
    if (head < kHkv) {
      unsigned char *krow = block + slot * kTokRowBytes + head * kHeadRowBytes;
      *reinterpret_cast<uint2 *>(krow + 8 * j) = rlo;
      *reinterpret_cast<uint2 *>(krow + kD + 8 * j) = rhi;
    }
    if (tid < kTokRowBytes / 16)
      reinterpret_cast<uint4 *>(block + kHalfPageBytes + slot * kTokRowBytes)[tid] = v[i];
  }
  pdl_wait_primary();   // this grid ends after the allocation kernel
}

struct FreeParams {
  const int32_t *seq_ids;
  int32_t *block_table;
  const int32_t *context_lens;
  int32_t *free_list;
  int32_t *free_count;
  int32_t *err;
  int n_free;
  int n_layers;
  int max_blocks;
  int num_blocks;
};

template <int BT>
__global__ void __launch_bounds__(kScanCta) free_kernel(FreeParams p) {
  __shared__ int tot[kScanCta / 32];
  const int cap = p.max_blocks * BT;
  const int fc0 = *p.free_count;
  int pushed = 0;
  for (int i = 0; i < p.n_free; ++i) {
    const int s = p.seq_ids[i];
    if (s < 0) {
      if (threadIdx.x == 0) report(p.err, PA_DEV_CTX_RANGE);
      continue;
    }
    int T = p.context_lens[s];
    if (T < 0 || T > cap) {
      if (threadIdx.x == 0) report(p.err, PA_DEV_CTX_RANGE);
      T = min(max(T, 0), cap);
    }
    const int nb = (T + BT - 1) / BT;
    const long long entries = static_cast<long long>(nb) * p.n_layers;
    for (long long e0 = 0; e0 < entries; e0 += kScanCta) {
      const long long e = e0 + threadIdx.x;
      int32_t *entry = nullptr;
      int blk = -1;
      bool valid = false;
      if (e < entries) {
        const int layer = static_cast<int>(e / nb);
        const int jj = static_cast<int>(e % nb);
        entry = p.block_table + table_row(s, p.n_layers, layer, p.max_blocks) + jj;
        blk = *entry;
        valid = blk >= 0 && blk < p.num_blocks;
      }
      int chunk = 0;
      const int rank = cta_exclusive_count(valid, tot, &chunk);
      if (entry) {
        if (!valid) {
          report(p.err, PA_DEV_BAD_BLOCK);
          *entry = -1;
        } else {
          const long long at = static_cast<long long>(fc0) + pushed + rank;
          if (at >= 0 && at < p.num_blocks) {
            p.free_list[at] = blk;
            *entry = -1;
          } else {
            report(p.err, PA_DEV_FREE_OVERFLOW);
          }
        }
      }
      pushed += chunk;
    }
  }
  if (threadIdx.x == 0) {
    const long long n = static_cast<long long>(fc0) + pushed;
    *p.free_count = fc0 >= p.num_blocks ? fc0 : static_cast<int>(min(n, static_cast<long long>(p.num_blocks)));
  }
}

}  // namespace
}  // namespace pa

using namespace pa;

namespace {

template <int BT>
int kv_append_rope_impl(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                        uint16_t *kv_cache, int num_blocks, int32_t *block_table, int n_layers,
                        int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                        int layer, int32_t *free_list, int32_t *free_count, int32_t *err,
                        void *stream) {
  if (num_seqs < 0 || num_blocks <= 0 || n_layers <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * BT > INT_MAX) return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0) return PA_OK;
  if (!k_new || !v_new || !kv_cache || !block_table || !context_lens || !free_list ||
      !free_count || !err)
    return PA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_cache) ||
      (q_or_null && !aligned16(q_or_null)))
    return PA_ERR_ALIGN;
  DeviceInfo di;
  const int rc = current_device(&di);
  if (rc != PA_OK) return rc;

  static const RopeFreqs freqs = llama3_freqs();
  AppendParams prm;
  prm.freqs = freqs;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.q = q_or_null;
  prm.kv = reinterpret_cast<unsigned char *>(kv_cache);
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.free_list = free_list;
  prm.free_count = free_count;
  prm.err = err;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.layer = layer;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_pdl(append_alloc_kernel<BT>, dim3(1), dim3(kScanCta), 0, st, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(append_store_kernel<BT>, dim3(num_seqs), dim3(kStoreThreads), 0, st, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" int pa_kv_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                                 uint16_t *q_or_null, uint16_t *kv_cache, int num_blocks,
                                 int32_t *block_table, int n_layers, int max_blocks_per_seq,
                                 const int32_t *context_lens, int num_seqs, int layer,
                                 int32_t *free_list, int32_t *free_count, int32_t *err,
                                 void *stream) {
  return kv_append_rope_impl<kBs>(k_new, v_new, q_or_null, kv_cache, num_blocks, block_table,
                                  n_layers, max_blocks_per_seq, context_lens, num_seqs, layer,
                                  free_list, free_count, err, stream);
}

extern "C" int pa_kv_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                                    uint16_t *q_or_null, uint16_t *kv_cache, int num_blocks,
                                    int block_tokens, int32_t *block_table, int n_layers,
                                    int max_blocks_per_seq, const int32_t *context_lens,
                                    int num_seqs, int layer, int32_t *free_list,
                                    int32_t *free_count, int32_t *err, void *stream) {
  switch (block_tokens) {
    case 8:
      return kv_append_rope_impl<8>(k_new, v_new, q_or_null, kv_cache, num_blocks, block_table,
                                    n_layers, max_blocks_per_seq, context_lens, num_seqs, layer,
                                    free_list, free_count, err, stream);
    case 16:
      return kv_append_rope_impl<16>(k_new, v_new, q_or_null, kv_cache, num_blocks, block_table,
                                     n_layers, max_blocks_per_seq, context_lens, num_seqs, layer,
                                     free_list, free_count, err, stream);
    case 32:
      return kv_append_rope_impl<32>(k_new, v_new, q_or_null, kv_cache, num_blocks, block_table,
                                     n_layers, max_blocks_per_seq, context_lens, num_seqs, layer,
                                     free_list, free_count, err, stream);
    default:
      return PA_ERR_ARG;
  }
}

namespace {

template <int BT>
int prefill_append_impl(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                        int total_tokens, const int32_t *cu_tokens, uint16_t *kv_cache,
                        int num_blocks, int32_t *block_table, int n_layers,
                        int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                        int layer, int32_t *free_list, int32_t *free_count, int32_t *err,
                        void *stream) {
  if (num_seqs < 0 || total_tokens < 0 || num_blocks <= 0 || n_layers <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * BT > INT_MAX) return PA_ERR_ARG;
  if (layer < 0 || layer >= n_layers) return PA_ERR_LAYER;
  if (num_seqs == 0 || total_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !cu_tokens || !kv_cache || !block_table || !context_lens ||
      !free_list || !free_count || !err)
    return PA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_cache) ||
      (q_or_null && !aligned16(q_or_null)))
    return PA_ERR_ALIGN;
  DeviceInfo di;
  const int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  static const RopeFreqs freqs = llama3_freqs();
  PrefillAppendParams prm;
  prm.freqs = freqs;
  prm.k_new = k_new;
  prm.v_new = v_new;
  prm.q = q_or_null;
  prm.kv = reinterpret_cast<unsigned char *>(kv_cache);
  prm.block_table = block_table;
  prm.cu_tokens = cu_tokens;
  prm.context_lens = context_lens;
  prm.free_list = free_list;
  prm.free_count = free_count;
  prm.err = err;
  prm.total_tokens = total_tokens;
  prm.num_blocks = num_blocks;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_seqs = num_seqs;
  prm.layer = layer;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_pdl(prefill_alloc_kernel<BT>, dim3(1), dim3(kScanCta), 0, st, prm) != cudaSuccess)
    return PA_ERR_CUDA;
  if (launch_pdl(prefill_store_kernel<BT>, dim3((total_tokens + kStoreRows - 1) / kStoreRows),
                 dim3(kStoreThreads), 0, st, prm) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" int pa_prefill_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                                      uint16_t *q_or_null, int total_tokens,
                                      const int32_t *cu_tokens, uint16_t *kv_cache, int num_blocks,
                                      int32_t *block_table, int n_layers, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int layer,
                                      int32_t *free_list, int32_t *free_count, int32_t *err,
                                      void *stream) {
  return prefill_append_impl<kBs>(k_new, v_new, q_or_null, total_tokens, cu_tokens, kv_cache,
                                  num_blocks, block_table, n_layers, max_blocks_per_seq,
                                  context_lens, num_seqs, layer, free_list, free_count, err,
                                  stream);
}

extern "C" int pa_prefill_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                                         uint16_t *q_or_null, int total_tokens,
                                         const int32_t *cu_tokens, uint16_t *kv_cache,
                                         int num_blocks, int block_tokens, int32_t *block_table,
                                         int n_layers, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_seqs, int layer,
                                         int32_t *free_list, int32_t *free_count, int32_t *err,
                                         void *stream) {
  switch (block_tokens) {
    case 8:
      return prefill_append_impl<8>(k_new, v_new, q_or_null, total_tokens, cu_tokens, kv_cache,
                                    num_blocks, block_table, n_layers, max_blocks_per_seq,
                                    context_lens, num_seqs, layer, free_list, free_count, err,
                                    stream);
    case 16:
      return prefill_append_impl<16>(k_new, v_new, q_or_null, total_tokens, cu_tokens, kv_cache,
                                     num_blocks, block_table, n_layers, max_blocks_per_seq,
                                     context_lens, num_seqs, layer, free_list, free_count, err,
                                     stream);
    case 32:
      return prefill_append_impl<32>(k_new, v_new, q_or_null, total_tokens, cu_tokens, kv_cache,
                                     num_blocks, block_table, n_layers, max_blocks_per_seq,
                                     context_lens, num_seqs, layer, free_list, free_count, err,
                                     stream);
    default:
      return PA_ERR_ARG;
  }
}

namespace {

template <int BT>
int free_impl(const int32_t *seq_ids, int n_free, int32_t *block_table, int n_layers,
              int max_blocks_per_seq, const int32_t *context_lens, int32_t *free_list,
              int32_t *free_count, int num_blocks, int32_t *err, void *stream) {
  if (n_free < 0 || num_blocks <= 0 || n_layers <= 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * BT > INT_MAX) return PA_ERR_ARG;
  if (n_free == 0) return PA_OK;
  if (!seq_ids || !block_table || !context_lens || !free_list || !free_count || !err)
    return PA_ERR_NULL;
  DeviceInfo di;
  const int rc = current_device(&di);
  if (rc != PA_OK) return rc;
  FreeParams prm;
  prm.seq_ids = seq_ids;
  prm.block_table = block_table;
  prm.context_lens = context_lens;
  prm.free_list = free_list;
  prm.free_count = free_count;
  prm.err = err;
  prm.n_free = n_free;
  prm.n_layers = n_layers;
  prm.max_blocks = max_blocks_per_seq;
  prm.num_blocks = num_blocks;
  free_kernel<BT><<<1, kScanCta, 0, static_cast<cudaStream_t>(stream)>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

extern "C" int pa_free(const int32_t *seq_ids, int n_free, int32_t *block_table, int n_layers,
                       int max_blocks_per_seq, const int32_t *context_lens, int32_t *free_list,
                       int32_t *free_count, int num_blocks, int32_t *err, void *stream) {
  return free_impl<kBs>(seq_ids, n_free, block_table, n_layers, max_blocks_per_seq, context_lens,
                        free_list, free_count, num_blocks, err, stream);
}

extern "C" int pa_free_bt(const int32_t *seq_ids, int n_free, int block_tokens,
                          int32_t *block_table, int n_layers, int max_blocks_per_seq,
                          const int32_t *context_lens, int32_t *free_list, int32_t *free_count,
                          int num_blocks, int32_t *err, void *stream) {
  switch (block_tokens) {
    case 8:
      return free_impl<8>(seq_ids, n_free, block_table, n_layers, max_blocks_per_seq,
                          context_lens, free_list, free_count, num_blocks, err, stream);
    case 16:
      return free_impl<16>(seq_ids, n_free, block_table, n_layers, max_blocks_per_seq,
                           context_lens, free_list, free_count, num_blocks, err, stream);
    case 32:
      return free_impl<32>(seq_ids, n_free, block_table, n_layers, max_blocks_per_seq,
                           context_lens, free_list, free_count, num_blocks, err, stream);
    default:
      return PA_ERR_ARG;
  }
}

extern "C" const char *pa_error_string(int code) {
  switch (code) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "a required pointer is NULL";
    case PA_ERR_ARG: return "a size or count is out of range";
    case PA_ERR_LAYER: return "layer outside [0, n_layers)";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_ALIGN: return "a tensor pointer is not 16-byte aligned";
    case PA_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case PA_ERR_DEVICE: return "no usable sm_103 device";
    case PA_ERR_STATE: return "batcher call out of order";
    default: return "unknown error";
  }
}
