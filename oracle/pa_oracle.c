/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle.  TEST INFRASTRUCTURE ONLY:
 * the tests, the smoke check and the benchmark's CPU baseline leg call it;
 * the CUDA library never does, and the two share no code.
 *
 * Every loop here follows the definition of the operation directly: gather
 * each token through the block table, take the full softmax over all scores,
 * sum p * v.  No blocking, no online rescaling, no fusion.
 *
 * Page cited throughout: "An Inference Engine in 1,500 Lines of CUDA: The
 * Map" (tiny-vllm series part 1).  See pa_oracle.h for the data layout.
 */
#include "pa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define BS    16   /* BLOCK_SIZE = 16 tokens per page ("The path of one inference", constants listing) */
#define HKV    8   /* kv heads */
#define HQ    32   /* q heads; GQA_Q_TO_K_RATIO = 4 ("What is in the box", GQA row) */
#define HD    64   /* head_dim */
#define GQA    4

/* Element (blk, K=0|V=1, tok, head, d) of a pool whose pages hold bt tokens. */
static size_t pool_index(int blk, int kv, int tok, int head, int d, int bt)
{
    return ((((size_t)blk * 2 + kv) * bt + tok) * HKV + head) * HD + d;
}

static size_t bt_row(int seq, int n_layers, int layer, int max_blocks)
{
    return ((size_t)seq * n_layers + layer) * (size_t)max_blocks;
}

double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to bf16, nearest-even.  First round to float (nearest-even),
 * then to bf16; when the float lands exactly on a bf16 half-way point that
 * the double did not sit on, the second rounding goes toward the double. */
uint16_t oracle_double_to_bf16(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf or nan */
        if (u & 0x007fffffu) return (uint16_t)((u >> 16) | 0x0040u);
        return (uint16_t)(u >> 16);
    }
    uint32_t low = u & 0xffffu;
    uint32_t hi = u >> 16;
    if (low == 0x8000u && (double)f != x) {
        /* the float is a tie only because of the first rounding */
        int away = fabs(x) > fabs((double)f);
        return (uint16_t)(away ? hi + 1 : hi);
    }
    if (low > 0x8000u || (low == 0x8000u && (hi & 1u))) hi += 1;
    return (uint16_t)hi;
}

/* ---------------------------------------------------------------- RoPE ---
 * init_rope_frequencies(HEAD_DIM, MAX_SEQ_LEN, 500000, 32, 1, 4, 8192)
 * ("The path of one inference", step (3)): theta, factor, low_freq_factor,
 * high_freq_factor, original context length.  The pages give only the
 * arguments; the rule applied to them is the published Llama 3.1 rescaling:
 * wavelengths shorter than original/high are kept, longer than original/low
 * are divided by factor, and the band between is blended linearly in
 * original/wavelength. */
double oracle_llama3_scale_freq(double inv_freq, double factor,
                                double low_freq_factor, double high_freq_factor,
                                double original_max_pos)
{
    const double pi = 3.14159265358979323846;
    double wavelen = 2.0 * pi / inv_freq;
    double high_wavelen = original_max_pos / high_freq_factor;   /* 2048 */
    double low_wavelen = original_max_pos / low_freq_factor;     /* 8192 */
    if (wavelen < high_wavelen) return inv_freq;
    if (wavelen > low_wavelen) return inv_freq / factor;
    double smooth = (original_max_pos / wavelen - low_freq_factor) /
                    (high_freq_factor - low_freq_factor);
    return (1.0 - smooth) * inv_freq / factor + smooth * inv_freq;
}

void oracle_llama3_inv_freq(int head_dim, double theta, double factor,
                            double low_freq_factor, double high_freq_factor,
                            double original_max_pos, double *inv_freq)
{
    for (int i = 0; i < head_dim / 2; ++i) {
        double base = pow(theta, -(2.0 * i) / (double)head_dim);
        inv_freq[i] = oracle_llama3_scale_freq(base, factor, low_freq_factor,
                                               high_freq_factor, original_max_pos);
    }
}

/* Rotate-half pairing: element i turns with element i + head_dim/2 through
 * the angle pos * inv_freq[i]. */
void oracle_rope_rotate(const double *x, int head_dim, double pos,
                        const double *inv_freq, double *out)
{
    int half = head_dim / 2;
    for (int i = 0; i < half; ++i) {
        double angle = pos * inv_freq[i];
        double c = cos(angle), s = sin(angle);
        double a = x[i], b = x[i + half];
        out[i] = a * c - b * s;
        out[i + half] = b * c + a * s;
    }
}

/* ----------------------------------------------------------- attention ---
 * The decode step of PagedAttention: one query token per sequence attends
 * over every cached token of that sequence, the K/V of token t living in
 * physical block block_table[seq][layer][t / 16] at slot t % 16 ("What is in
 * the box": 16-token pages plus a block_table index array; "The path of one
 * inference": -1 means not assigned yet).  q head h uses kv head h / 4. */

static int check_block(int blk, int num_blocks)
{
    return blk >= 0 && blk < num_blocks;
}

int oracle_attention_partial_bt(const uint16_t *q_head, const uint16_t *pool,
                                int num_blocks, const int32_t *row, int kv_head,
                                int t_begin, int t_end, double scale,
                                double *m_out, double *l_out, double *acc, int bt)
{
    int n = t_end - t_begin;
    for (int d = 0; d < HD; ++d) acc[d] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (n <= 0) return 0;

    double *score = (double *)malloc(sizeof(double) * (size_t)n);
    if (!score) return -1;
    int err = 0;
    for (int t = t_begin; t < t_end; ++t) {
        int blk = row[t / bt];
        if (!check_block(blk, num_blocks)) { err |= PAO_ERR_BAD_BLOCK; score[t - t_begin] = -INFINITY; continue; }
        double dot = 0.0;
        for (int d = 0; d < HD; ++d)
            dot += oracle_bf16_to_double(q_head[d]) *
                   oracle_bf16_to_double(pool[pool_index(blk, 0, t % bt, kv_head, d, bt)]);
        score[t - t_begin] = scale * dot;
    }
    double m = -INFINITY;
    for (int i = 0; i < n; ++i) if (score[i] > m) m = score[i];
    double l = 0.0;
    for (int t = t_begin; t < t_end; ++t) {
        int blk = row[t / bt];
        if (!check_block(blk, num_blocks)) continue;
        double p = exp(score[t - t_begin] - m);
        l += p;
        for (int d = 0; d < HD; ++d)
            acc[d] += p * oracle_bf16_to_double(pool[pool_index(blk, 1, t % bt, kv_head, d, bt)]);
    }
    free(score);
    *m_out = m;
    *l_out = l;
    return err;
}

int oracle_attention_partial(const uint16_t *q_head, const uint16_t *pool,
                             int num_blocks, const int32_t *row, int kv_head,
                             int t_begin, int t_end, double scale,
                             double *m_out, double *l_out, double *acc)
{
    return oracle_attention_partial_bt(q_head, pool, num_blocks, row, kv_head, t_begin, t_end,
                                       scale, m_out, l_out, acc, BS);
}

/* Split-context merge: the partials of disjoint token ranges combine into
 * the softmax over their union by rescaling each to the common maximum. */
void oracle_merge_partials(int n_parts, const double *m, const double *l,
                           const double *acc, double *out)
{
    double mmax = -INFINITY;
    for (int p = 0; p < n_parts; ++p) if (m[p] > mmax) mmax = m[p];
    double lsum = 0.0;
    for (int d = 0; d < HD; ++d) out[d] = 0.0;
    if (mmax == -INFINITY) return;
    for (int p = 0; p < n_parts; ++p) {
        if (m[p] == -INFINITY) continue;
        double w = exp(m[p] - mmax);
        lsum += w * l[p];
        for (int d = 0; d < HD; ++d) out[d] += w * acc[(size_t)p * HD + d];
    }
    for (int d = 0; d < HD; ++d) out[d] /= lsum;
}

int oracle_decode_attention_bt(double *out, const uint16_t *q, const uint16_t *pool,
                               int num_blocks, const int32_t *block_table,
                               int n_layers, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int layer,
                               double scale, int bt)
{
    int err = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        if (ctx < 0 || ctx > max_blocks_per_seq * bt) {
            err |= PAO_ERR_CTX_RANGE;
            ctx = ctx < 0 ? 0 : max_blocks_per_seq * bt;
        }
        const int32_t *row = block_table + bt_row(s, n_layers, layer, max_blocks_per_seq);
        for (int h = 0; h < HQ; ++h) {
            double *o = out + ((size_t)s * HQ + h) * HD;
            double m, l;
            int e = oracle_attention_partial_bt(q + ((size_t)s * HQ + h) * HD, pool,
                                                num_blocks, row, h / GQA, 0, ctx,
                                                scale, &m, &l, o, bt);
            if (e < 0) return e;
            err |= e;
            if (ctx == 0 || l == 0.0) {           /* empty context: zeros */
                for (int d = 0; d < HD; ++d) o[d] = 0.0;
                continue;
            }
            for (int d = 0; d < HD; ++d) o[d] /= l;
        }
    }
    return err;
}

int oracle_decode_attention(double *out, const uint16_t *q, const uint16_t *pool,
                            int num_blocks, const int32_t *block_table,
                            int n_layers, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int layer,
                            double scale)
{
    return oracle_decode_attention_bt(out, q, pool, num_blocks, block_table, n_layers,
                                      max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                      BS);
}

/* -------------------------------------------------------------- append ---
 * Each sequence adds the token at position pos = context_lens[s].  When pos
 * starts a new 16-token page the sequence takes a block from the free list
 * (free_blocks is an iota vector, "The path of one inference"; the reading
 * here pops from its back, sequences in ascending order), records it in
 * block_table[s][layer][pos / 16], then stores RoPE(k) and v at slot
 * pos % 16.  q, when given, is rotated in place at the same position; that
 * rotation depends on the position alone, so it happens even when the K/V
 * store is refused.  A refused allocation leaves the table entry at -1. */
int oracle_kv_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                             uint16_t *q_or_null, uint16_t *pool, int num_blocks,
                             int32_t *block_table, int n_layers, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int layer,
                             int32_t *free_list, int32_t *free_count,
                             const double *inv_freq, int bt)
{
    int err = 0;
    double x[HD], y[HD];
    for (int s = 0; s < num_seqs; ++s) {
        int pos = context_lens[s];
        if (pos < 0 || pos >= max_blocks_per_seq * bt) { err |= PAO_ERR_CTX_RANGE; continue; }
        if (q_or_null) {
            /* q turns at its position whatever happens to the K/V store */
            for (int h = 0; h < HQ; ++h) {
                uint16_t *qh = q_or_null + ((size_t)s * HQ + h) * HD;
                for (int d = 0; d < HD; ++d) x[d] = oracle_bf16_to_double(qh[d]);
                oracle_rope_rotate(x, HD, (double)pos, inv_freq, y);
                for (int d = 0; d < HD; ++d) qh[d] = oracle_double_to_bf16(y[d]);
            }
        }
        int32_t *row = block_table + bt_row(s, n_layers, layer, max_blocks_per_seq);
        int blk;
        if (pos % bt == 0) {
            if (*free_count <= 0) {
                /* refused: the page stays unassigned */
                err |= PAO_ERR_FREE_UNDERFLOW;
                row[pos / bt] = -1;
                continue;
            }
            blk = free_list[*free_count - 1];
            *free_count -= 1;
            row[pos / bt] = blk;
        } else {
            blk = row[pos / bt];
        }
        if (!check_block(blk, num_blocks)) { err |= PAO_ERR_BAD_BLOCK; continue; }

        int slot = pos % bt;
        for (int h = 0; h < HKV; ++h) {
            const uint16_t *k = k_new + ((size_t)s * HKV + h) * HD;
            const uint16_t *v = v_new + ((size_t)s * HKV + h) * HD;
            for (int d = 0; d < HD; ++d) x[d] = oracle_bf16_to_double(k[d]);
            oracle_rope_rotate(x, HD, (double)pos, inv_freq, y);
            for (int d = 0; d < HD; ++d) {
                pool[pool_index(blk, 0, slot, h, d, bt)] = oracle_double_to_bf16(y[d]);
                pool[pool_index(blk, 1, slot, h, d, bt)] = v[d];
            }
        }
    }
    return err;
}

int oracle_kv_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *q_or_null, uint16_t *pool, int num_blocks,
                          int32_t *block_table, int n_layers, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int layer,
                          int32_t *free_list, int32_t *free_count,
                          const double *inv_freq)
{
    return oracle_kv_append_rope_bt(k_new, v_new, q_or_null, pool, num_blocks, block_table,
                                    n_layers, max_blocks_per_seq, context_lens, num_seqs, layer,
                                    free_list, free_count, inv_freq, BS);
}

/* ------------------------------------------------------------- prefill ---
 * The prefill path of tiny-vllm pushes a whole prompt through at once
 * ("The path of one inference": prefill() is matrix x matrix, decode is
 * vector x matrix; ropeKernel_llama3 rotates all prompt tokens).  Here a
 * prompt chunk is appended to the paged cache and attends causally. */
int oracle_prefill_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                                  uint16_t *q_or_null, const int32_t *cu_tokens,
                                  uint16_t *pool, int num_blocks, int32_t *block_table,
                                  int n_layers, int max_blocks_per_seq,
                                  const int32_t *context_lens, int num_seqs, int layer,
                                  int32_t *free_list, int32_t *free_count,
                                  const double *inv_freq, int bt)
{
    int err = 0;
    double x[HD], y[HD];
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        int n = cu_tokens[s + 1] - cu_tokens[s];
        if (ctx < 0 || n < 0 || ctx + n > max_blocks_per_seq * bt) { err |= PAO_ERR_CTX_RANGE; continue; }
        int32_t *row = block_table + bt_row(s, n_layers, layer, max_blocks_per_seq);
        int refused = -1;   /* page of this chunk the free list could not give */
        for (int i = 0; i < n; ++i) {
            int pos = ctx + i;
            size_t r = (size_t)cu_tokens[s] + (size_t)i;
            if (q_or_null) {
                for (int h = 0; h < HQ; ++h) {
                    uint16_t *qh = q_or_null + (r * HQ + h) * HD;
                    for (int d = 0; d < HD; ++d) x[d] = oracle_bf16_to_double(qh[d]);
                    oracle_rope_rotate(x, HD, (double)pos, inv_freq, y);
                    for (int d = 0; d < HD; ++d) qh[d] = oracle_double_to_bf16(y[d]);
                }
            }
            if (pos % bt == 0) {
                if (*free_count <= 0) {
                    err |= PAO_ERR_FREE_UNDERFLOW;
                    row[pos / bt] = -1;
                    refused = pos / bt;
                    continue;
                }
                row[pos / bt] = free_list[*free_count - 1];
                *free_count -= 1;
            }
            if (pos / bt == refused) continue;          /* already reported */
            int blk = row[pos / bt];
            if (!check_block(blk, num_blocks)) { err |= PAO_ERR_BAD_BLOCK; continue; }
            int slot = pos % bt;
            for (int h = 0; h < HKV; ++h) {
                const uint16_t *k = k_new + (r * HKV + h) * HD;
                const uint16_t *v = v_new + (r * HKV + h) * HD;
                for (int d = 0; d < HD; ++d) x[d] = oracle_bf16_to_double(k[d]);
                oracle_rope_rotate(x, HD, (double)pos, inv_freq, y);
                for (int d = 0; d < HD; ++d) {
                    pool[pool_index(blk, 0, slot, h, d, bt)] = oracle_double_to_bf16(y[d]);
                    pool[pool_index(blk, 1, slot, h, d, bt)] = v[d];
                }
            }
        }
    }
    return err;
}

int oracle_prefill_attention_bt(double *out, const uint16_t *q, const int32_t *cu_tokens,
                                const uint16_t *pool, int num_blocks,
                                const int32_t *block_table, int n_layers,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                int num_seqs, int layer, double scale, int bt)
{
    int err = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        int n = cu_tokens[s + 1] - cu_tokens[s];
        if (ctx < 0 || n < 0 || ctx + n > max_blocks_per_seq * bt) { err |= PAO_ERR_CTX_RANGE; continue; }
        const int32_t *row = block_table + bt_row(s, n_layers, layer, max_blocks_per_seq);
        for (int i = 0; i < n; ++i) {
            size_t r = (size_t)cu_tokens[s] + (size_t)i;
            for (int h = 0; h < HQ; ++h) {
                double *o = out + (r * HQ + h) * HD;
                double m, l;
                int e = oracle_attention_partial_bt(q + (r * HQ + h) * HD, pool, num_blocks, row,
                                                    h / GQA, 0, ctx + i + 1, scale, &m, &l, o, bt);
                if (e < 0) return e;
                err |= e;
                for (int d = 0; d < HD; ++d) o[d] = (l > 0.0) ? o[d] / l : 0.0;
            }
        }
    }
    return err;
}

int oracle_prefill_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                               uint16_t *q_or_null, const int32_t *cu_tokens,
                               uint16_t *pool, int num_blocks, int32_t *block_table,
                               int n_layers, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int layer,
                               int32_t *free_list, int32_t *free_count,
                               const double *inv_freq)
{
    return oracle_prefill_append_rope_bt(k_new, v_new, q_or_null, cu_tokens, pool, num_blocks,
                                         block_table, n_layers, max_blocks_per_seq,
                                         context_lens, num_seqs, layer, free_list, free_count,
                                         inv_freq, BS);
}

int oracle_prefill_attention(double *out, const uint16_t *q, const int32_t *cu_tokens,
                             const uint16_t *pool, int num_blocks,
                             const int32_t *block_table, int n_layers,
                             int max_blocks_per_seq, const int32_t *context_lens,
                             int num_seqs, int layer, double scale)
{
    return oracle_prefill_attention_bt(out, q, cu_tokens, pool, num_blocks, block_table, n_layers,
                                       max_blocks_per_seq, context_lens, num_seqs, layer, scale,
                                       BS);
}

/* ---------------------------------------------------------------- free ---
 * A finished sequence hands its blocks back: for each listed sequence in the
 * given order, layer 0..n_layers-1, logical block 0..ceil(ctx/16)-1, push the
 * block onto the back of the free list and mark the table entry -1 (the
 * "not assigned yet" value). */
int oracle_free_bt(const int32_t *seq_ids, int n_free, int32_t *block_table,
                   int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                   int32_t *free_list, int32_t *free_count, int num_blocks, int bt)
{
    int err = 0;
    for (int i = 0; i < n_free; ++i) {
        int s = seq_ids[i];
        int ctx = context_lens[s];
        if (ctx < 0 || ctx > max_blocks_per_seq * bt) {
            err |= PAO_ERR_CTX_RANGE;
            ctx = ctx < 0 ? 0 : max_blocks_per_seq * bt;
        }
        int nb = (ctx + bt - 1) / bt;
        for (int layer = 0; layer < n_layers; ++layer) {
            int32_t *row = block_table + bt_row(s, n_layers, layer, max_blocks_per_seq);
            for (int j = 0; j < nb; ++j) {
                int blk = row[j];
                if (!check_block(blk, num_blocks)) { err |= PAO_ERR_BAD_BLOCK; row[j] = -1; continue; }
                if (*free_count >= num_blocks) { err |= PAO_ERR_FREE_OVERFLOW; continue; }
                free_list[*free_count] = blk;
                *free_count += 1;
                row[j] = -1;
            }
        }
    }
    return err;
}

int oracle_free(const int32_t *seq_ids, int n_free, int32_t *block_table,
                int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                int32_t *free_list, int32_t *free_count, int num_blocks)
{
    return oracle_free_bt(seq_ids, n_free, block_table, n_layers, max_blocks_per_seq,
                          context_lens, free_list, free_count, num_blocks, BS);
}
