/*
 * pa_oracle.h -- plain CPU oracle for the PagedAttention decode step and the
 * KV append with Llama-3-scaled RoPE.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library; the few constants below are restated here on purpose.
 *
 * Source pages: "An Inference Engine in 1,500 Lines of CUDA: The Map"
 * (jaehun.me, tiny-vllm series part 1), sections "What is in the box" (the
 * 16-token pages + block_table, GQA ratio 4, online softmax, Llama-3 RoPE
 * rows) and "The path of one inference" (the init_rope_frequencies arguments,
 * the 2 GB pool cut into 16-token blocks, the iota free list, the block_table
 * filled with -1).
 *
 * All floating point is fp64.  bf16 values travel as their raw 16-bit
 * patterns (uint16_t).
 *
 * Data layout (the pages do not state one; this is the reading used):
 *   pool        [num_blocks][2 (K=0, V=1)][16 tokens][8 kv heads][64] bf16
 *   block_table [num_seqs][n_layers][max_blocks_per_seq] int32, -1 = unassigned
 *   q           [num_seqs][32 q heads][64] bf16
 *   k_new/v_new [num_seqs][8 kv heads][64] bf16
 *   q head h reads kv head h / 4.
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* error bits, same meaning as the library's device error word */
#define PAO_ERR_BAD_BLOCK      1  /* block id outside [0, num_blocks) inside a context */
#define PAO_ERR_CTX_RANGE      2  /* context < 0 or beyond max_blocks_per_seq * 16 */
#define PAO_ERR_FREE_UNDERFLOW 4  /* append needed a block but the free list was empty */
#define PAO_ERR_FREE_OVERFLOW  8  /* free pushed more than num_blocks entries */

/* Llama-3 RoPE inverse frequencies, inv_freq[head_dim/2]. */
void oracle_llama3_inv_freq(int head_dim, double theta, double factor,
                            double low_freq_factor, double high_freq_factor,
                            double original_max_pos, double *inv_freq);

/* Llama-3 rescaling of one unscaled inverse frequency. */
double oracle_llama3_scale_freq(double inv_freq, double factor,
                                double low_freq_factor, double high_freq_factor,
                                double original_max_pos);

/* Rotate-half RoPE of one head vector x[head_dim] at position pos. */
void oracle_rope_rotate(const double *x, int head_dim, double pos,
                        const double *inv_freq, double *out);

/* bf16 <-> double (round to nearest even, exact from double). */
double   oracle_bf16_to_double(uint16_t b);
uint16_t oracle_double_to_bf16(double x);

/* Decode attention for one layer.  out[num_seqs][32][64] fp64.
 * Returns the error bits found (0 on success). */
int oracle_decode_attention(double *out, const uint16_t *q, const uint16_t *pool,
                            int num_blocks, const int32_t *block_table,
                            int n_layers, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int layer,
                            double scale);

/* Unnormalised partial of one q head over tokens [t_begin, t_end):
 * m = max score, l = sum exp(score - m), acc[64] = sum exp(score - m) v. */
int oracle_attention_partial(const uint16_t *q_head, const uint16_t *pool,
                             int num_blocks, const int32_t *bt_row, int kv_head,
                             int t_begin, int t_end, double scale,
                             double *m, double *l, double *acc);

/* Merge n_parts partials (m[p], l[p], acc[p][64]) into out[64]. */
void oracle_merge_partials(int n_parts, const double *m, const double *l,
                           const double *acc, double *out);

/* KV append with RoPE for one layer (block allocation, K rotation, store).
 * Rotates q in place when q_or_null is not NULL.  Returns error bits. */
int oracle_kv_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                          uint16_t *q_or_null, uint16_t *pool, int num_blocks,
                          int32_t *block_table, int n_layers, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int layer,
                          int32_t *free_list, int32_t *free_count,
                          const double *inv_freq);

/* Prefill (a prompt chunk per sequence).  Tokens of all sequences are
 * packed: those of sequence s are rows cu_tokens[s] .. cu_tokens[s+1]-1 of
 * k_new / v_new [rows][8][64] and q [rows][32][64]; token i of s sits at
 * position context_lens[s] + i.
 *
 * Append: positions are taken in (sequence, position) order; a position that
 * starts a page pops the back of the free list.  A chunk that does not fit
 * the sequence's table (context < 0 or context + tokens > max_blocks * 16)
 * is refused whole (PAO_ERR_CTX_RANGE: nothing popped, stored or rotated).
 * A refused page (free list empty) is -1 in the table and its tokens are not
 * stored; q is rotated for every token of an accepted chunk. */
int oracle_prefill_append_rope(const uint16_t *k_new, const uint16_t *v_new,
                               uint16_t *q_or_null, const int32_t *cu_tokens,
                               uint16_t *pool, int num_blocks, int32_t *block_table,
                               int n_layers, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int layer,
                               int32_t *free_list, int32_t *free_count,
                               const double *inv_freq);

/* Causal attention of every chunk token over positions 0..context+i of its
 * sequence (the cached tokens and the chunk's tokens up to itself).
 * out[rows][32][64] fp64. */
int oracle_prefill_attention(double *out, const uint16_t *q, const int32_t *cu_tokens,
                             const uint16_t *pool, int num_blocks,
                             const int32_t *block_table, int n_layers,
                             int max_blocks_per_seq, const int32_t *context_lens,
                             int num_seqs, int layer, double scale);

/* The same with pages of bt tokens (the page's BLOCK_SIZE, 16, being a
 * tunable: pool [num_blocks][2][bt][8][64], token t of a sequence in block
 * row[t / bt], slot t % bt; a page starts at positions that are multiples
 * of bt).  The functions above are these with bt = 16. */
int oracle_attention_partial_bt(const uint16_t *q_head, const uint16_t *pool,
                                int num_blocks, const int32_t *bt_row, int kv_head,
                                int t_begin, int t_end, double scale,
                                double *m, double *l, double *acc, int bt);
int oracle_decode_attention_bt(double *out, const uint16_t *q, const uint16_t *pool,
                               int num_blocks, const int32_t *block_table,
                               int n_layers, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int layer,
                               double scale, int bt);
int oracle_kv_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                             uint16_t *q_or_null, uint16_t *pool, int num_blocks,
                             int32_t *block_table, int n_layers, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int layer,
                             int32_t *free_list, int32_t *free_count,
                             const double *inv_freq, int bt);
int oracle_free_bt(const int32_t *seq_ids, int n_free, int32_t *block_table,
                   int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                   int32_t *free_list, int32_t *free_count, int num_blocks, int bt);
int oracle_prefill_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new,
                                  uint16_t *q_or_null, const int32_t *cu_tokens,
                                  uint16_t *pool, int num_blocks, int32_t *block_table,
                                  int n_layers, int max_blocks_per_seq,
                                  const int32_t *context_lens, int num_seqs, int layer,
                                  int32_t *free_list, int32_t *free_count,
                                  const double *inv_freq, int bt);
int oracle_prefill_attention_bt(double *out, const uint16_t *q, const int32_t *cu_tokens,
                                const uint16_t *pool, int num_blocks,
                                const int32_t *block_table, int n_layers,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                int num_seqs, int layer, double scale, int bt);

/* Release the blocks of finished sequences.  Returns error bits. */
int oracle_free(const int32_t *seq_ids, int n_free, int32_t *block_table,
                int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                int32_t *free_list, int32_t *free_count, int num_blocks);

#ifdef __cplusplus
}
#endif
#endif
