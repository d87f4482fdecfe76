/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) PagedAttention decode library.
 *
 * The operations follow "An Inference Engine in 1,500 Lines of CUDA: The
 * Map" (jaehun.me, tiny-vllm series part 1):
 *   - "What is in the box": PagedAttention as 16-token pages plus a
 *     block_table index array; GQA_Q_TO_K_RATIO = 4; online softmax inside
 *     pagedAttentionKernel; RoPE with Llama 3 scaling.
 *   - "The path of one inference": init_rope_frequencies(HEAD_DIM,
 *     MAX_SEQ_LEN, 500000, 32, 1, 4, 8192); one 2 GB cudaMalloc cut into
 *     16-token blocks numbered by an iota free list; a block_table of
 *     MAX_SEQUENCES * N_LAYERS * MAX_BLOCKS_PER_SEQ ints set to -1 ("not
 *     assigned yet"); decode handles one token per active slot per step.
 *
 * Fixed shapes (Llama 3.2 1B): 32 query heads, 8 kv heads (q head h reads
 * kv head h / 4), head_dim 64, 16 tokens per block, bf16 storage.
 *
 * Layouts (all row-major, all device memory owned by the caller):
 *   kv_cache     [num_blocks][2][16][8][64] bf16   (index 0 = K, 1 = V);
 *                one block is 32 KiB, contiguous
 *   block_table  [num_seqs][n_layers][max_blocks_per_seq] int32, -1 = none;
 *                sequence i of a call uses row i
 *   q, out       [num_seqs][32][64] bf16
 *   k_new, v_new [num_seqs][8][64] bf16
 *   context_lens [num_seqs] int32
 *   free_list    [num_blocks] int32, a stack: entries [0, *free_count) free
 *
 * bf16 values are passed as their 16-bit patterns (uint16_t).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless stated; the library allocates and
 *     frees nothing and keeps no pointer after the call returns.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and the call returns without synchronising.
 *   - The return value reports host-detectable faults (PA_ERR_*).  Faults
 *     found by the kernels (bad block id, context out of range, free-list
 *     underflow/overflow, a wait that ran out) are OR-ed as PA_DEV_* bits into
 *     the caller's device word `*err`; the kernels never trap.  The caller
 *     zeroes *err when it wants a fresh report.
 *   - num_seqs == 0 (or n_free == 0) is a no-op that returns PA_OK.
 *   - Tensor pointers must be 16-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_NUM_Q_HEADS   32
#define PA_NUM_KV_HEADS  8
#define PA_HEAD_DIM      64
#define PA_BLOCK_TOKENS  16
#define PA_BLOCK_BYTES   (2 * PA_BLOCK_TOKENS * PA_NUM_KV_HEADS * PA_HEAD_DIM * 2)

/* host-side return codes */
#define PA_OK              0
#define PA_ERR_NULL       -1   /* a required pointer is NULL */
#define PA_ERR_ARG        -2   /* a size or count is out of range */
#define PA_ERR_LAYER      -3   /* layer outside [0, n_layers) */
#define PA_ERR_WORKSPACE  -4   /* workspace NULL or smaller than pa_decode_workspace_size */
#define PA_ERR_ALIGN      -5   /* a tensor pointer is not 16-byte aligned */
#define PA_ERR_CUDA       -6   /* a CUDA runtime call or kernel launch failed */
#define PA_ERR_DEVICE     -7   /* no usable device, or not an sm_103 GPU */
#define PA_ERR_STATE      -8   /* batcher call out of order (run without a plan, plan twice) */

/* device-side error bits, OR-ed into *err */
#define PA_DEV_BAD_BLOCK       1   /* block id outside [0, num_blocks) inside a context */
#define PA_DEV_CTX_RANGE       2   /* context < 0 or beyond max_blocks_per_seq * 16 */
#define PA_DEV_FREE_UNDERFLOW  4   /* append needed a block and the free list was empty */
#define PA_DEV_FREE_OVERFLOW   8   /* free pushed past num_blocks entries */
#define PA_DEV_TIMEOUT        16   /* an internal pipeline wait ran out; output invalid */

/*
 * pa_kv_append_rope -- append one new token per sequence to the paged cache.
 *
 * Page: "The path of one inference" (free_blocks / block_table set-up,
 * init_rope_frequencies arguments) and "What is in the box" (RoPE with
 * Llama 3 scaling; ropeKernelDecode is the decode-time RoPE).
 *
 * For each sequence s, pos = context_lens[s] (tokens already cached):
 *   1. If pos % 16 == 0, a block is taken from the free list: sequences that
 *      need one are served in ascending s, each taking
 *      free_list[*free_count - 1] and decrementing *free_count; the id is
 *      written to block_table[s][layer][pos / 16].
 *   2. k_new[s] is rotated with rotate-half RoPE at angle pos * f_i, f_i the
 *      Llama-3-scaled inverse frequencies (theta 500000, factor 32, low 1,
 *      high 4, original context 8192), rounded to bf16, and stored with
 *      v_new[s] (copied bit for bit) at slot pos % 16 of that block.
 *   3. If q_or_null is not NULL, q[s] (all 32 heads) is rotated in place at
 *      the same position.
 * Device errors: PA_DEV_CTX_RANGE (pos < 0 or pos >= max_blocks_per_seq*16;
 * nothing written), PA_DEV_FREE_UNDERFLOW (no block left; nothing written),
 * PA_DEV_BAD_BLOCK (existing table entry invalid; nothing written).
 * Two kernels on `stream`; the second starts early with programmatic
 * dependent launch and waits for the first before touching the cache.
 */
int pa_kv_append_rope(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                      uint16_t *kv_cache, int num_blocks,
                      int32_t *block_table, int n_layers, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int layer,
                      int32_t *free_list, int32_t *free_count, int32_t *err,
                      void *stream);

/*
 * pa_decode_attention -- the decode step of PagedAttention for one layer.
 *
 * Page: "What is in the box" (pagedAttentionKernel: online softmax, warp
 * shuffle reductions, 16-token pages + block_table; GQA ratio 4).
 *
 * out[s][h] = sum_t softmax_t(scale * q[s][h] . K_t) V_t over the
 * context_lens[s] tokens t of sequence s, K_t/V_t read from block
 * block_table[s][layer][t / 16], slot t % 16, kv head h / 4.  fp32
 * accumulation, output rounded to bf16.  A sequence with context 0 gets a
 * zero output.  Long contexts are split across CTAs and merged (split
 * context); the split only changes rounding.  Which kernel runs is set by
 * pa_decode_set_path (automatic by default).
 * workspace: device scratch of at least pa_decode_workspace_size(num_seqs,
 * max_blocks_per_seq) bytes, owned by the caller.  It must be zero-filled
 * once before its first use (it holds the work counter that spreads blocks
 * over CTAs); every call returns it to a state the next call accepts.
 * Calls that share one workspace must not overlap in time.
 * num_seqs is at most 2048 per call.
 * Device errors: PA_DEV_BAD_BLOCK (that block's tokens are dropped),
 * PA_DEV_CTX_RANGE (context clamped), PA_DEV_TIMEOUT.
 */
int pa_decode_attention(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                        int num_blocks, const int32_t *block_table, int n_layers,
                        int max_blocks_per_seq, const int32_t *context_lens,
                        int num_seqs, int layer, float scale,
                        void *workspace, size_t workspace_bytes, int32_t *err,
                        void *stream);

/*
 * pa_decode_attention_static -- pa_decode_attention for callers that cannot
 * allocate device memory where they run the decode step.
 *
 * The pages have no counterpart to this entry point.  It serves callers that
 * may not call cudaMalloc at that point -- an engine whose memory map is fixed
 * at start-up, a serving thread that must not trigger the device-wide
 * synchronisation an allocation can cause, a plugin handed only its tensors.
 * It computes exactly what pa_decode_attention computes, with the same
 * arguments minus the workspace: the split partials and the work counter live
 * in a 16 MiB array in the library's device memory, held by every GPU that
 * loads the library until the process exits.
 *   - num_seqs at most PA_STATIC_MAX_SEQS; more returns PA_ERR_WORKSPACE.
 *   - Calls no cudaMalloc / cudaFree or allocating library routine.
 *   - The first call on a device looks up the array's device address (with
 *     that device current).  Under CUDA's lazy module loading that first call
 *     may also load the library's device code and back the 16 MiB array, which
 *     can allocate and synchronise the device: make one warm-up call on each
 *     device at start-up, before serving and before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; each call clears its work counter on `stream` first.  Calls
 *     whose kernels could overlap on the GPU race on the array: serialise them.
 */
#define PA_STATIC_MAX_SEQS 512
int pa_decode_attention_static(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                               int num_blocks, const int32_t *block_table, int n_layers,
                               int max_blocks_per_seq, const int32_t *context_lens,
                               int num_seqs, int layer, float scale, int32_t *err,
                               void *stream);

/*
 * Page size as a tunable: pa_kv_append_rope_bt, pa_decode_attention_bt,
 * pa_free_bt and pa_decode_workspace_size_bt are the entry points above with
 * pages of block_tokens = 8, 16 or 32 tokens (the page's BLOCK_SIZE is 16,
 * "What is in the box": 16-token pages; the four calls above are these with
 * 16).  The pool is then [num_blocks][2][block_tokens][8][64] bf16 (a block
 * is block_tokens * 2 KiB), token t of a sequence lives in block
 * block_table[s][layer][t / block_tokens], slot t % block_tokens, and an
 * append at position pos takes a new block when pos % block_tokens == 0.
 * Everything else (arguments, layouts, errors) is as above; another
 * block_tokens returns PA_ERR_ARG (0 from the workspace size).  The prefill
 * entry points have the same variants (pa_prefill_append_rope_bt,
 * pa_prefill_attention_bt, declared with them below); the batcher uses
 * 16-token pages.
 */
int pa_kv_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                         uint16_t *kv_cache, int num_blocks, int block_tokens,
                         int32_t *block_table, int n_layers, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int layer,
                         int32_t *free_list, int32_t *free_count, int32_t *err,
                         void *stream);
int pa_decode_attention_bt(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                           int num_blocks, int block_tokens, const int32_t *block_table,
                           int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                           int num_seqs, int layer, float scale,
                           void *workspace, size_t workspace_bytes, int32_t *err,
                           void *stream);
int pa_free_bt(const int32_t *seq_ids, int n_free, int block_tokens, int32_t *block_table,
               int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
               int32_t *free_list, int32_t *free_count, int num_blocks,
               int32_t *err, void *stream);
size_t pa_decode_workspace_size_bt(int num_seqs, int max_blocks_per_seq, int block_tokens);

/*
 * pa_prefill_append_rope -- append a prompt chunk per sequence to the paged
 * cache (the prefill counterpart of pa_kv_append_rope).
 *
 * Page: "The path of one inference" (prefill pushes the whole prompt through
 * at once, matrix x matrix; ropeKernel_llama3 is the prefill RoPE, paired with
 * ropeKernelDecode) and "What is in the box" (16-token pages + block_table).
 *
 * Packed tokens: cu_tokens[num_seqs + 1] (device) is non-decreasing with
 * cu_tokens[0] = 0 and cu_tokens[num_seqs] = total_tokens; the chunk of
 * sequence s is rows cu_tokens[s] .. cu_tokens[s+1]-1 of
 *   k_new, v_new [total_tokens][8][64] bf16, q [total_tokens][32][64] bf16,
 * and row cu_tokens[s] + i sits at position context_lens[s] + i
 * (context_lens[s] = tokens already cached for s; 0 for a fresh prompt).
 *   1. Every position of a chunk that starts a page (position % 16 == 0)
 *      takes a block from the back of the free list, in (sequence, position)
 *      order, and writes it to block_table[s][layer][position / 16].
 *   2. Each k_new row is rotated (rotate-half RoPE with the Llama-3-scaled
 *      frequencies of pa_kv_append_rope), rounded to bf16 and stored with its
 *      v_new row at slot position % 16 of its page.
 *   3. If q_or_null is not NULL, every q row of an accepted chunk is rotated
 *      in place at its position.
 * Device errors: PA_DEV_CTX_RANGE (context < 0, context + chunk beyond
 * max_blocks_per_seq * 16, or rows outside [0, total_tokens): the whole chunk
 * is refused, nothing popped, stored or rotated), PA_DEV_FREE_UNDERFLOW (no
 * block left: that page stays -1 and its tokens are not stored),
 * PA_DEV_BAD_BLOCK (a table entry the chunk writes into is invalid: its
 * tokens are not stored).  Two kernels on `stream`, the second started early
 * with programmatic dependent launch.
 */
int pa_prefill_append_rope(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                           int total_tokens, const int32_t *cu_tokens,
                           uint16_t *kv_cache, int num_blocks, int32_t *block_table,
                           int n_layers, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs, int layer,
                           int32_t *free_list, int32_t *free_count, int32_t *err,
                           void *stream);

/*
 * pa_prefill_attention -- causal attention of a prompt chunk per sequence
 * over its pages (the prefill counterpart of pa_decode_attention).
 *
 * Page: "The path of one inference" (prefill: the whole prompt at once,
 * matrix x matrix) and "What is in the box" (16-token pages + block_table;
 * GQA ratio 4; online softmax).
 *
 * With the packed layout of pa_prefill_append_rope (q and out
 * [total_tokens][32][64] bf16), for row r = cu_tokens[s] + i:
 *   out[r][h] = sum_t softmax_t(scale * q[r][h] . K_t) V_t
 * over positions t = 0 .. context_lens[s] + i of sequence s, read from block
 * block_table[s][layer][t / 16], slot t % 16, kv head h / 4.  The chunk's own
 * K/V must already be in the cache (pa_prefill_append_rope before this call
 * on the same stream).  fp32 accumulation, output rounded to bf16.
 * num_seqs is at most 2048 per call; scale must be positive and finite
 * (PA_ERR_ARG otherwise); no workspace.
 * Device errors: PA_DEV_CTX_RANGE (a chunk that does not fit its table, or
 * rows outside [0, total_tokens): its rows are not written),
 * PA_DEV_BAD_BLOCK (that block's tokens are dropped), PA_DEV_TIMEOUT.
 */
int pa_prefill_attention(uint16_t *out, const uint16_t *q, int total_tokens,
                         const int32_t *cu_tokens, const uint16_t *kv_cache, int num_blocks,
                         const int32_t *block_table, int n_layers, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int layer, float scale,
                         int32_t *err, void *stream);

/*
 * pa_prefill_append_rope_bt / pa_prefill_attention_bt -- the two prefill
 * entry points above with pages of block_tokens = 8, 16 or 32 tokens (the
 * page's BLOCK_SIZE, 16, as a tunable; the pool [num_blocks][2][block_tokens]
 * [8][64] bf16, token t of a sequence in block block_table[s][layer]
 * [t / block_tokens], slot t % block_tokens; a chunk opens a page at every
 * position that is a multiple of block_tokens).  Arguments, layouts, errors
 * and stream behaviour are those of the calls above; another block_tokens
 * returns PA_ERR_ARG before any launch.
 */
int pa_prefill_append_rope_bt(const uint16_t *k_new, const uint16_t *v_new, uint16_t *q_or_null,
                              int total_tokens, const int32_t *cu_tokens, uint16_t *kv_cache,
                              int num_blocks, int block_tokens, int32_t *block_table,
                              int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                              int num_seqs, int layer, int32_t *free_list, int32_t *free_count,
                              int32_t *err, void *stream);
int pa_prefill_attention_bt(uint16_t *out, const uint16_t *q, int total_tokens,
                            const int32_t *cu_tokens, const uint16_t *kv_cache, int num_blocks,
                            int block_tokens, const int32_t *block_table, int n_layers,
                            int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                            int layer, float scale, int32_t *err, void *stream);

/*
 * Test hook for the prefill kernel's bounded waits (no counterpart on the
 * pages).  With chunk >= 0 the prefill attention kernel's CTA 0 announces the
 * bytes of its chunk-th 128-key chunk (counted over its items) without
 * issuing the copies, so the barriers waited on for that chunk never
 * complete; every wait of the kernel then gives up after wait_limit_ns
 * (1 us .. 1 s), sets PA_DEV_TIMEOUT in *err, and each warp waits (again
 * bounded) for its own copies and MMAs in flight before the CTA frees its
 * tensor memory and exits; the outputs of that call are undefined.  chunk =
 * -1 restores normal operation (waits of 1 s, no copy left out).
 * Process-wide; for tests only.  Returns PA_ERR_ARG for a bad chunk or limit.
 */
int pa_prefill_set_test_fault(int chunk, long long wait_limit_ns);

/* Bytes of workspace pa_decode_attention needs on the current device. */
size_t pa_decode_workspace_size(int num_seqs, int max_blocks_per_seq);

/*
 * pa_free -- return finished sequences' blocks to the free list.
 *
 * Page: "The path of one inference" (free_blocks numbered by iota; -1 =
 * not assigned yet) and the slot recycling of the decode loop.
 * For i = 0..n_free-1 in order, s = seq_ids[i] (a block_table row), every
 * layer 0..n_layers-1 and logical block j < ceil(context_lens[s] / 16):
 * push block_table[s][layer][j] onto the back of the free list and set the
 * entry to -1.  num_blocks bounds the free list.  seq_ids and context_lens
 * are device arrays.  Device errors: PA_DEV_BAD_BLOCK (entry invalid; reset
 * to -1, not pushed), PA_DEV_FREE_OVERFLOW (free list full; entry kept),
 * PA_DEV_CTX_RANGE (negative seq id or context out of range).
 */
int pa_free(const int32_t *seq_ids, int n_free, int32_t *block_table, int n_layers,
            int max_blocks_per_seq, const int32_t *context_lens,
            int32_t *free_list, int32_t *free_count, int num_blocks,
            int32_t *err, void *stream);

/*
 * Continuous batching -- the host loop that feeds prefill and decode from a
 * queue of requests through a fixed set of block-table rows (slots).
 *
 * Page: "The path of one inference": prompts wait in a queue; while a slot
 * is free and a prompt is queued, prefill() takes the whole prompt at once;
 * otherwise one decode step produces one token for every active slot; a
 * finished slot is free again; the loop ends when no slot is active and the
 * queue is empty.  Where the page is silent:
 *   - A request is (request_id, prompt_len P >= 1, decode_steps G >= 1); it
 *     is finished after its G-th decode step (a generation length stands in
 *     for the end-of-text token: no model runs here).
 *   - Active requests hold block-table rows 0..n-1 in admission order.  A
 *     step first releases the requests that finished in the step before
 *     (pa_free over their rows, ascending), then closes the gaps keeping the
 *     order (the rows' table entries move with them).
 *   - Admission is first-in first-out and stops at the first queued request
 *     that lacks a free row, n_layers * ceil((P + G) / 16) pages not yet
 *     promised to admitted requests (so decode never runs out of pages), or
 *     P tokens of the step's prefill budget.
 *   - The step prefills the admitted prompts together (every layer:
 *     pa_prefill_append_rope then pa_prefill_attention on their rows), then
 *     every active row takes one decode step (every layer:
 *     pa_kv_append_rope at position = tokens cached, pa_decode_attention
 *     over position + 1, with the kernel pa_decode_kernel_for_lengths picks
 *     for the rows' contexts unless pa_decode_set_path forces one).
 * A batcher is host memory (created and owned by the library, freed by
 * pa_batcher_destroy); it is not thread-safe.  Use per step:
 *   pa_batcher_plan   decides the step (host only);
 *   pa_batcher_rows   tells which request each row holds and its decode
 *                     position, so the caller can fill the step's q/k/v;
 *   pa_batcher_run    enqueues the step's device work on `stream`
 *                     (or pa_batcher_commit, when the caller runs it).
 * After a failed pa_batcher_run the batcher's state is undefined: destroy it.
 */
typedef struct pa_batcher pa_batcher;

typedef struct pa_batch_plan {
    int n_retired;       /* requests released at the start of the step */
    int n_keep;          /* rows active before admission: 0 .. n_keep-1 */
    int n_admitted;      /* rows n_keep .. n_rows-1, prefilled this step */
    int n_rows;          /* rows taking the decode step: 0 .. n_rows-1 */
    int prefill_tokens;  /* prompt tokens of the admitted rows, packed in row order */
    int done;            /* 1: queue empty and nothing active; nothing to run */
} pa_batch_plan;

typedef struct pa_batch_buffers {
    uint16_t *kv_cache;            /* the pool (pa_decode_attention's layout) */
    int num_blocks;
    int32_t *block_table;          /* [max_slots][n_layers][max_blocks_per_seq], -1 filled */
    int32_t *block_table_tmp;      /* same size: rows move through it */
    void *ctl;                     /* device control area of pa_batcher_ctl_bytes */
    size_t ctl_bytes;
    int32_t *free_list;            /* holds at least the pages the batcher was given */
    int32_t *free_count;
    int32_t *err;                  /* device error word (PA_DEV_* bits) */
    void *decode_workspace;        /* pa_decode_workspace_size(max_slots, max_blocks_per_seq) bytes, zeroed once */
    size_t decode_workspace_bytes;
    /* the step's inputs and outputs, bf16, layer-major:
     *   prefill_*  [n_layers][prefill_budget][32 or 8][64]: row t of a layer
     *              is packed prompt token t (pa_prefill_attention's layout);
     *   decode_*   [n_layers][max_slots][32 or 8][64]: row i is block-table
     *              row i's token of the step.
     * q is rotated in place; out receives the attention outputs. */
    uint16_t *prefill_q, *prefill_k, *prefill_v, *prefill_out;
    uint16_t *decode_q, *decode_k, *decode_v, *decode_out;
    float scale;
} pa_batch_buffers;

/* Bytes of the device control area a batcher with max_slots rows uses. */
size_t pa_batcher_ctl_bytes(int max_slots);

/* max_slots rows (at most 2048) of a block table with n_layers and
 * max_blocks_per_seq; pages_free = pages on the free list when the loop
 * starts (the batcher promises no more than that); prefill_budget = prompt
 * tokens prefilled per step at most.  PA_ERR_ARG on bad sizes. */
int pa_batcher_create(int max_slots, int n_layers, int max_blocks_per_seq, int pages_free,
                      int prefill_budget, pa_batcher **out);
/* The same with pages of block_tokens = 8, 16 or 32 tokens ("The path of one
 * inference" marks BLOCK_SIZE as a tunable): lifetime pages are counted in
 * such pages, and every step runs the page-size (_bt) entry points over a
 * kv_cache of [num_blocks][2][block_tokens][8][64].  PA_ERR_ARG for another
 * size. */
int pa_batcher_create_bt(int max_slots, int n_layers, int max_blocks_per_seq, int pages_free,
                         int prefill_budget, int block_tokens, pa_batcher **out);
int pa_batcher_destroy(pa_batcher *b);

/* Queue a request.  PA_ERR_ARG when it could never run: P < 1, G < 1,
 * P > prefill_budget, P + G beyond max_blocks_per_seq * block_tokens, or
 * more pages than pages_free. */
int pa_batcher_submit(pa_batcher *b, int64_t request_id, int prompt_len, int decode_steps);

/* Decide the next step.  PA_ERR_STATE if the previous plan was not run. */
int pa_batcher_plan(pa_batcher *b, pa_batch_plan *plan);

/* Request id and decode position (tokens cached before the step's token)
 * of rows 0..n_rows-1 of the planned step; returns n_rows, or PA_ERR_ARG if
 * cap is smaller.  Either output may be NULL. */
int pa_batcher_rows(const pa_batcher *b, int64_t *request_ids, int32_t *positions, int cap);

/* Request ids released by the planned step; returns their number. */
int pa_batcher_retired(const pa_batcher *b, int64_t *request_ids, int cap);

/* Requests still queued. */
int pa_batcher_pending(const pa_batcher *b);

/* Enqueue the planned step on `stream`: one host-to-device copy of the
 * control block, pa_free and two row-moving kernels when requests leave, the
 * prefill of the admitted rows, the decode step; then pa_batcher_commit.
 * Host faults as PA_ERR_*; device faults OR-ed into buf->err.  The buffers
 * must stay untouched until the stream reaches the end of the step. */
int pa_batcher_run(pa_batcher *b, const pa_batch_buffers *buf, void *stream);

/* Decode-only steps (no request leaves or enters) are replayed from CUDA
 * graphs once one such step has run eagerly: one graph per batch size and
 * buffer set, captured on first use, its control-block copy fed from a
 * small ring of pinned host buffers the batcher owns.  Enabled by default;
 * enable = 0 runs every step by direct launches.  If capture is not
 * possible (for instance, `stream` is being captured by the caller) the
 * batcher switches to direct launches for good. */
int pa_batcher_set_graphs(pa_batcher *b, int enable);

/* Mark the planned step as done without enqueuing anything, for callers
 * that run the step's device work with their own kernels: the admitted
 * prompts count as cached and every row as one decode step further. */
int pa_batcher_commit(pa_batcher *b);

/* Cap on the CTAs one pa_decode_attention launch uses (0 = automatic: two
 * per SM).  Process-wide; affects only how contexts are split. */
int pa_decode_set_grid_limit(int max_ctas);

/*
 * Which decode-attention kernel pa_decode_attention runs (process-wide).
 * All compute the same attention and differ only in rounding order.
 *   PA_DECODE_AUTO     the per-head cluster kernel when every (sequence, kv
 *                      head) pair of the call gets at least two CTAs at once
 *                      (num_seqs * 16 <= 2 CTAs per SM, within the grid
 *                      limit) and pages hold 16 or 32 tokens; the
 *                      split-context kernel otherwise.
 *   PA_DECODE_SPLIT    always the split-context kernel: the batch's blocks
 *                      laid end to end and cut into chunks over all CTAs,
 *                      fp32 partials merged by a second kernel.  Balances any
 *                      mix of context lengths.
 *   PA_DECODE_CLUSTER  the per-head cluster kernel: one thread-block cluster
 *                      of 1, 2, 4 or 8 CTAs per (sequence, kv head), its CTAs
 *                      combined in shared memory; no workspace use.
 *   PA_DECODE_SEQ      the per-sequence cluster kernel: one cluster of 1 to
 *                      16 CTAs per sequence, one 32 KiB copy per page, each
 *                      CTA combining the q heads it owns; no workspace use.
 *                      Fastest when the batch's contexts are of similar
 *                      length; slow when a few contexts are much longer
 *                      than the rest (their clusters finish last).
 * The per-sequence kernel needs 16-token pages; the per-head one takes 8-,
 * 16- or 32-token pages (a 16-token tile is two pages or half a page), 8
 * only when forced (its four 1 KiB copies per tile make it slower than the
 * split kernel there); where a path's kernel does not take the page size
 * the call runs the split-context kernel.  Returns PA_ERR_ARG for any other
 * value.
 */
#define PA_DECODE_AUTO     0
#define PA_DECODE_SPLIT    1
#define PA_DECODE_CLUSTER  2
#define PA_DECODE_SEQ      3
int pa_decode_set_path(int path);

/* The kernel (PA_DECODE_SPLIT, _CLUSTER or _SEQ) that pa_decode_attention
 * (block_tokens 16) or pa_decode_attention_bt would run for num_seqs
 * sequences on the current device under the current path and grid limit;
 * PA_ERR_ARG for a bad count or page size, PA_ERR_CUDA / PA_ERR_DEVICE when
 * no sm_103 device answers. */
int pa_decode_kernel_for(int num_seqs, int block_tokens);

/* The decode kernel for a batch whose context lengths the caller knows on the
 * host (context_lens: num_seqs host ints, the lengths the attention covers),
 * for pages of block_tokens tokens; the caller passes it to
 * pa_decode_set_path (the continuous batcher applies it to every decode step
 * while the path is PA_DECODE_AUTO).  PA_DECODE_AUTO alone sees only
 * num_seqs; this rule also
 * sees how far the longest context lies above the mean (rho = max / mean,
 * in 16-token tiles):
 *   8-token pages, or rho > 3 (a few contexts far above the rest): the
 *     split-context kernel, the only one that spreads a long context over
 *     the whole GPU;
 *   else, while every (sequence, kv head) pair gets two CTAs at once (the
 *     PA_DECODE_AUTO bound): the per-head cluster kernel;
 *   else, 16-token pages and at most one sequence per CTA of the grid
 *     (two CTAs per SM, or the grid limit): the per-sequence cluster kernel
 *     (one 32 KiB copy per page);
 *   else the split-context kernel.
 * Measured on GB300 over 36 batches of 4..128 sequences with contexts
 * U[256, 2048], log-uniform in [1, 8192], all 1024 and all 4096: within 5 %
 * of the fastest kernel in 34 of them (the two others at 12 sequences: 5.0
 * and 9 % above the per-sequence kernel).  Ignores the process-wide path;
 * respects the grid limit.  PA_ERR_ARG for a bad count, page size or a null
 * pointer with num_seqs > 0; PA_ERR_CUDA / PA_ERR_DEVICE when no sm_103
 * device answers.  Host code only: no device work. */
int pa_decode_kernel_for_lengths(const int32_t *context_lens, int num_seqs, int block_tokens);

/*
 * Test hook for the bounded waits (no counterpart on the pages; they
 * build no failure detection).  With stage >= 0 the split-context kernel's
 * CTA 0 publishes its stage-th shared-memory stage without issuing the copies
 * for it, so the barrier the consumers wait on never completes; every wait of
 * the split kernel then gives up after wait_limit_ns (1 us .. 1 s), sets
 * PA_DEV_TIMEOUT in *err and returns, and the outputs of that call are
 * undefined.  No other kernel is affected.  stage = -1 restores normal
 * operation (waits of 1 s, no copy left out).  Process-wide; for tests only.
 * Returns PA_ERR_ARG for a bad stage or limit.
 */
int pa_decode_set_test_fault(int stage, long long wait_limit_ns);

/*
 * Test hook of the per-head cluster kernel's speculative plan (no
 * counterpart on the pages).  With mode = 1, its packed plan (the batches
 * where every (sequence, kv head) pair gets two CTAs on average) is first
 * worked out from the first sequence's length in place of every length, as
 * if the lengths had changed after they were read, so that the check after
 * the dependency wait finds the plan moved: CTAs change role mid-call (the
 * consumers drop what they accumulated and reload q) or are left without a
 * part.  Outputs stay exact.  mode = 0 restores normal operation.
 * Process-wide; for tests only.  PA_ERR_ARG for another mode.
 */
int pa_decode_set_test_plan(int mode);

/* Human-readable name of a PA_ERR_* code. */
const char *pa_error_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
