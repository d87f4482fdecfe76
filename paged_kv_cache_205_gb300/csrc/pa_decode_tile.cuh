// pa_decode_tile.cuh -- one 16-token tile of one kv head in the decode
// kernels: the 4 q heads of the GQA group against the tile's K and V, folded
// into a warp's running online-softmax state.
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "What is in
// the box": softmax(q . K^T * scale) V per query head with an online softmax,
// GQA_Q_TO_K_RATIO = 4.
//
// The 4 q heads are the M rows of m16n8k16 bf16 tensor-core MMAs: S = Q K^T
// (8 MMAs, rows 4..15 of Q are zero) and O += P V (8 MMAs) per tile, fed by
// ldmatrix from shared memory.  The softmax runs on the S fragments in fp32
// in the log2 domain (2 shuffles per tile).  The PV MMA takes P as two bf16
// parts: rows 0..3 of its A operand hold bf16(P) and rows 8..11 the bf16
// rounding of the remainder P - bf16(P), so D rows r and r + 8 accumulate
// the two parts of the same q head's output and their sum carries P to
// about 16 significant bits, at no extra MMA (the rows were idle).  l sums
// the fp32 weights.  With P in bf16 alone, short contexts (a few keys,
// outputs the size of single V entries) would add up to ~2e-3 of weight
// rounding to the output's own bf16 rounding.
#pragma once

#include "pa_device.cuh"

namespace pa {

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Q fragments of q heads (g*4 .. g*4+3) of one token: row r = lane / 4 holds
// columns 16ks + c2 (qa) and 16ks + 8 + c2 (qc), c2 = 2 (lane % 4); lanes of
// rows 4..7 hold zeros.  q: [32][64] bf16 of the token.
__device__ __forceinline__ void load_q_fragments(const uint16_t *q_token, int g, int lane,
                                                 uint32_t (&qa)[4], uint32_t (&qc)[4]) {
  const int r = lane >> 2, c2 = 2 * (lane & 3);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) qa[ks] = qc[ks] = 0u;
  if (r < kGqa) {
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(q_token + (g * kGqa + r) * kD);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qa[ks] = __ldg(qrow + (16 * ks + c2) / 2);
      qc[ks] = __ldg(qrow + (16 * ks + 8 + c2) / 2);
    }
  }
}

struct TileState {
  float o[8][4];   // O fragments, 8 tiles of 8 dims: row r (P's bf16 part) and
                   // row r + 8 (the remainder's part) of q head r
  float m;         // running max (log2 domain) of row r
  float l;         // running sum of this lane's columns of row r

  // Unnormalised output of q head r at dims 8t + c2 + k (k = 0, 1).
  __device__ __forceinline__ float out(int t, int k) const { return o[t][k] + o[t][k + 2]; }

  __device__ __forceinline__ void reset() {
    m = neg_inf();
    l = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  }
};

// Folds one tile into the warp's state.  ktile / vtile: shared addresses of
// the tile's 16 K rows and 16 V rows of 128 bytes, 16-byte chunk c of row t
// stored at chunk c ^ (t & 7).  Tokens used: 0 .. n_valid-1, or with
// kRowMask the set bits of `use` (8-token pages whose second page is
// missing).  The V rows of the other tokens are zeroed first (they may hold
// anything, NaN included) and their scores masked.  The caller synchronises
// the warp before the tile's buffer is released.
template <bool kRowMask>
__device__ __forceinline__ void attend_tile(uint32_t ktile, uint32_t vtile, int n_valid,
                                            unsigned use, const uint32_t (&qa)[4],
                                            const uint32_t (&qc)[4], float qscale, int lane,
                                            TileState &st) {
  const int c2 = 2 * (lane & 3);
  const int lm_i = lane >> 3, lm_r = lane & 7;
  if (kRowMask ? (use != 0xffffu) : (n_valid < kBs)) {
    uint4 *vrow = reinterpret_cast<uint4 *>(__cvta_shared_to_generic(vtile));
    if (kRowMask) {
      for (int e = lane; e < kBs * 8; e += 32)
        if (!((use >> (e >> 3)) & 1u)) vrow[e] = make_uint4(0, 0, 0, 0);
    } else {
      for (int e = n_valid * 8 + lane; e < kBs * 8; e += 32) vrow[e] = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();   // the next copy into this buffer comes through TMA
    __syncwarp();
  }
  // ---- S = Q K^T for tokens 0..7 (s0) and 8..15 (s1)
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) {
    const int tok = (lm_i >> 1) * 8 + lm_r;
    const int chunk = 2 * ks + (lm_i & 1);
    uint32_t b0, b1, b2, b3;
    ldsm_x4(ktile + tok * kHeadRowBytes + ((chunk ^ lm_r) << 4), b0, b1, b2, b3);
    mma_bf16_16816(s0, qa[ks], 0u, qc[ks], 0u, b0, b1);
    mma_bf16_16816(s1, qa[ks], 0u, qc[ks], 0u, b2, b3);
  }
  // ---- online softmax on row r, columns c2, c2+1, 8+c2, 9+c2
  const bool u0 = kRowMask ? ((use >> c2) & 1u) : (c2 < n_valid);
  const bool u1 = kRowMask ? ((use >> (c2 + 1)) & 1u) : (c2 + 1 < n_valid);
  const bool u2 = kRowMask ? ((use >> (c2 + 8)) & 1u) : (c2 + 8 < n_valid);
  const bool u3 = kRowMask ? ((use >> (c2 + 9)) & 1u) : (c2 + 9 < n_valid);
  const float x0 = u0 ? s0[0] * qscale : neg_inf();
  const float x1 = u1 ? s0[1] * qscale : neg_inf();
  const float x2 = u2 ? s1[0] * qscale : neg_inf();
  const float x3 = u3 ? s1[1] * qscale : neg_inf();
  float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(st.m, mx);
  const float alpha = fast_exp2(st.m - m_new);
  const float p0 = fast_exp2(x0 - m_new), p1 = fast_exp2(x1 - m_new);
  const float p2 = fast_exp2(x2 - m_new), p3 = fast_exp2(x3 - m_new);
  const uint32_t pa = float2_to_bf16x2(p0, p1);
  const uint32_t pc = float2_to_bf16x2(p2, p3);
  const float2 fa = bf16x2_to_float2(pa), fc = bf16x2_to_float2(pc);
  const uint32_t pa_lo = float2_to_bf16x2(p0 - fa.x, p1 - fa.y);
  const uint32_t pc_lo = float2_to_bf16x2(p2 - fc.x, p3 - fc.y);
  st.l = fmaf(st.l, alpha, (p0 + p1) + (p2 + p3));
  st.m = m_new;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    st.o[t][0] *= alpha;
    st.o[t][1] *= alpha;
    st.o[t][2] *= alpha;
    st.o[t][3] *= alpha;
  }
  // ---- O += P V, dims in 4 pairs of 8-dim tiles
#pragma unroll
  for (int dp = 0; dp < 4; ++dp) {
    const int tok = (lm_i & 1) * 8 + lm_r;
    const int chunk = 2 * dp + (lm_i >> 1);
    uint32_t v0, v1, v2, v3;
    ldsm_x4_trans(vtile + tok * kHeadRowBytes + ((chunk ^ lm_r) << 4), v0, v1, v2, v3);
    mma_bf16_16816(st.o[2 * dp], pa, pa_lo, pc, pc_lo, v0, v1);
    mma_bf16_16816(st.o[2 * dp + 1], pa, pa_lo, pc, pc_lo, v2, v3);
  }
}

// Row sum of the warp's state over the lane quad of row r.
__device__ __forceinline__ float row_sum(const TileState &st) {
  float lt = st.l;
  lt += __shfl_xor_sync(0xffffffffu, lt, 1);
  lt += __shfl_xor_sync(0xffffffffu, lt, 2);
  return lt;
}

}  // namespace pa
