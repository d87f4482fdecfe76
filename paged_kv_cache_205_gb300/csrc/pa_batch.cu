// pa_batch.cu -- continuous batching over the paged cache: the host loop
// that feeds prefill and decode from a queue of requests through a fixed set
// of block-table rows (slots).
//
// Page: "An Inference Engine in 1,500 Lines of CUDA: The Map", "The path of
// one inference": prompts wait in a queue; while a slot is free and a prompt
// is queued, prefill() takes the whole prompt at once; otherwise one decode
// step produces one token per active slot; a finished slot is free again;
// the loop ends when no slot is active and the queue is empty.
//
// What the page leaves open is fixed as follows.
//   * A request is (id, P prompt tokens, G decode steps), G >= 1; it is
//     finished after its G-th decode step (no model here: a generation length
//     stands in for the end-of-text token).
//   * Active requests hold rows 0..n-1 in admission order.  A step first
//     releases the requests that finished in the step before (pa_free over
//     their rows, ascending), then closes the gaps keeping the order.
//   * Admission is first-in first-out and stops at the first request that
//     lacks a free row, L * ceil((P + G) / B) pages (B tokens per page, 16
//     unless the batcher was created with another size) not yet promised to the
//     admitted requests (so a decode step never runs out of pages), or P
//     tokens of the step's prefill budget.
//   * The admitted prompts are prefilled together (all layers:
//     pa_prefill_append_rope, pa_prefill_attention), then every active row
//     takes one decode step (all layers: pa_kv_append_rope at position ctx,
//     pa_decode_attention over ctx + 1).
//
// The loop's decisions are host code; every step's device work is enqueued
// on one stream from here: one host-to-device copy of the step's control
// block, the release, two row-moving kernels, then the library's entry points.
#include <algorithm>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "pa_device.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kMoveThreads = 256;

// Control block of one step, one copy to the device (int32 words):
//   [0, S)        rows released this step, ascending
//   [S, 2S)       cached tokens per row before the release (pa_free's context)
//   [2S, 3S)      source row of each kept row, after the gaps close
//   [3S, 4S)      decode position per row (tokens cached before the step's token)
//   [4S, 5S)      decode attention context per row (position + 1)
//   [5S, 6S + 1)  cu_tokens of the admitted prompts
//   [6S + 1, 7S + 1) zeros: the admitted rows' cached context
struct CtlLayout {
  int S;
  size_t retired() const { return 0; }
  size_t free_ctx() const { return static_cast<size_t>(S); }
  size_t keep() const { return 2 * static_cast<size_t>(S); }
  size_t pos() const { return 3 * static_cast<size_t>(S); }
  size_t attn() const { return 4 * static_cast<size_t>(S); }
  size_t cu() const { return 5 * static_cast<size_t>(S); }
  size_t zero() const { return 6 * static_cast<size_t>(S) + 1; }
  size_t words() const { return 7 * static_cast<size_t>(S) + 1; }
  size_t bytes() const { return (words() * 4 + 255) & ~static_cast<size_t>(255); }
};

// Rows [first, n_keep) of `tmp` take rows keep[first..n_keep) of `table`.
__global__ void __launch_bounds__(kMoveThreads) gather_rows_kernel(
    const int32_t *__restrict__ table, int32_t *__restrict__ tmp, const int32_t *__restrict__ keep,
    int first, int n_keep, int row_words) {
  const int r = first + blockIdx.y;
  if (r >= n_keep) return;
  const int32_t *src = table + static_cast<size_t>(keep[r]) * row_words;
  int32_t *dst = tmp + static_cast<size_t>(r) * row_words;
  for (int i = blockIdx.x * kMoveThreads + threadIdx.x; i < row_words; i += gridDim.x * kMoveThreads)
    dst[i] = src[i];
}

// Rows [first, n_keep) of `table` take them back from `tmp`; rows
// [n_keep, n_prev) (left behind by the moves) become -1.
__global__ void __launch_bounds__(kMoveThreads) place_rows_kernel(
    int32_t *__restrict__ table, const int32_t *__restrict__ tmp, int first, int n_keep,
    int n_prev, int row_words) {
  const int r = first + blockIdx.y;
  if (r >= n_prev) return;
  int32_t *dst = table + static_cast<size_t>(r) * row_words;
  const int32_t *src = tmp + static_cast<size_t>(r) * row_words;
  for (int i = blockIdx.x * kMoveThreads + threadIdx.x; i < row_words; i += gridDim.x * kMoveThreads)
    dst[i] = (r < n_keep) ? src[i] : -1;
}

struct Request {
  int64_t id;
  int prompt_len;
  int decode_steps;
};

struct Row {
  Request req;
  int ctx = 0;    // tokens cached
  int done = 0;   // decode steps taken
};

}  // namespace
}  // namespace pa

using namespace pa;

namespace {

constexpr int kCtlRing = 4;   // pinned control blocks in flight for replayed steps

// A decode-only step captured as a CUDA graph, for one batch size and one
// set of buffers.
struct DecodeGraph {
  int n_rows = 0;
  int path = 0;        // the decode kernel the graph runs
  int device = -1;
  pa_batch_buffers bufs{};
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t ctl_copy = nullptr;   // the control-block copy, repointed per replay
};

}  // namespace

struct pa_batcher {
  int max_slots, n_layers, max_blocks, pages_free, prefill_budget;
  int block_tokens = kBs;   // tokens per page
  std::deque<Request> queue;
  std::vector<Row> rows;
  long long promised = 0;
  // the planned step
  bool planned = false;
  pa_batch_plan plan{};
  std::vector<int64_t> retired_ids;
  int first_moved = 0;
  int n_prev = 0;
  std::vector<int32_t> ctl;   // host image of the control block
  // decode-only steps replayed from CUDA graphs
  bool graphs = true;
  bool eager_decode_done = false;   // the kernels' one-time set-up has run
  std::vector<DecodeGraph> decode_graphs;
  int32_t *pinned[kCtlRing] = {};
  cudaEvent_t ring_done[kCtlRing] = {};
  int ring_next = 0;
  cudaStream_t capture_stream = nullptr;
};

namespace {

long long pages_needed(const pa_batcher *b, int prompt_len, int decode_steps) {
  const int B = b->block_tokens;
  return static_cast<long long>(b->n_layers) * ((prompt_len + decode_steps + B - 1) / B);
}

}  // namespace

extern "C" size_t pa_batcher_ctl_bytes(int max_slots) {
  if (max_slots <= 0) return 0;
  return CtlLayout{max_slots}.bytes();
}

extern "C" int pa_batcher_create_bt(int max_slots, int n_layers, int max_blocks_per_seq,
                                    int pages_free, int prefill_budget, int block_tokens,
                                    pa_batcher **out) {
  if (!out) return PA_ERR_NULL;
  *out = nullptr;
  if (max_slots <= 0 || max_slots > 2048 || n_layers <= 0 || max_blocks_per_seq <= 0 ||
      pages_free < 0 || prefill_budget <= 0)
    return PA_ERR_ARG;
  if (block_tokens != 8 && block_tokens != 16 && block_tokens != 32) return PA_ERR_ARG;
  if (static_cast<long long>(max_blocks_per_seq) * block_tokens > (1LL << 30)) return PA_ERR_ARG;
  pa_batcher *b = new (std::nothrow) pa_batcher;
  if (!b) return PA_ERR_ARG;
  b->block_tokens = block_tokens;
  b->max_slots = max_slots;
  b->n_layers = n_layers;
  b->max_blocks = max_blocks_per_seq;
  b->pages_free = pages_free;
  b->prefill_budget = prefill_budget;
  b->ctl.assign(CtlLayout{max_slots}.words(), 0);
  *out = b;
  return PA_OK;
}

extern "C" int pa_batcher_create(int max_slots, int n_layers, int max_blocks_per_seq,
                                 int pages_free, int prefill_budget, pa_batcher **out) {
  return pa_batcher_create_bt(max_slots, n_layers, max_blocks_per_seq, pages_free,
                              prefill_budget, kBs, out);
}

extern "C" int pa_batcher_destroy(pa_batcher *b) {
  if (!b) return PA_OK;
  for (DecodeGraph &g : b->decode_graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    if (g.graph) cudaGraphDestroy(g.graph);
  }
  for (int i = 0; i < kCtlRing; ++i) {
    if (b->ring_done[i]) {
      cudaEventSynchronize(b->ring_done[i]);
      cudaEventDestroy(b->ring_done[i]);
    }
    if (b->pinned[i]) cudaFreeHost(b->pinned[i]);
  }
  if (b->capture_stream) cudaStreamDestroy(b->capture_stream);
  delete b;
  return PA_OK;
}

extern "C" int pa_batcher_set_graphs(pa_batcher *b, int enable) {
  if (!b) return PA_ERR_NULL;
  b->graphs = enable != 0;
  return PA_OK;
}

extern "C" int pa_batcher_submit(pa_batcher *b, int64_t request_id, int prompt_len,
                                 int decode_steps) {
  if (!b) return PA_ERR_NULL;
  if (prompt_len < 1 || decode_steps < 1 || prompt_len > b->prefill_budget) return PA_ERR_ARG;
  if (static_cast<long long>(prompt_len) + decode_steps >
      static_cast<long long>(b->max_blocks) * b->block_tokens)
    return PA_ERR_ARG;
  if (pages_needed(b, prompt_len, decode_steps) > b->pages_free) return PA_ERR_ARG;
  b->queue.push_back(Request{request_id, prompt_len, decode_steps});
  return PA_OK;
}

extern "C" int pa_batcher_plan(pa_batcher *b, pa_batch_plan *plan) {
  if (!b || !plan) return PA_ERR_NULL;
  if (b->planned) return PA_ERR_STATE;
  const CtlLayout L{b->max_slots};
  int32_t *ctl = b->ctl.data();
  std::fill(b->ctl.begin(), b->ctl.end(), 0);
  // 1. release what finished in the step before; the rest keep their order
  b->retired_ids.clear();
  std::vector<Row> kept;
  kept.reserve(b->rows.size());
  int n_ret = 0;
  for (int i = 0; i < static_cast<int>(b->rows.size()); ++i) {
    const Row &r = b->rows[i];
    if (r.done >= r.req.decode_steps) {
      ctl[L.retired() + n_ret++] = i;
      ctl[L.free_ctx() + i] = r.ctx;
      b->retired_ids.push_back(r.req.id);
      b->promised -= pages_needed(b, r.req.prompt_len, r.req.decode_steps);
    } else {
      ctl[L.keep() + kept.size()] = i;
      kept.push_back(r);
    }
  }
  b->n_prev = static_cast<int>(b->rows.size());
  const int n_keep = static_cast<int>(kept.size());
  int first = 0;
  while (first < n_keep && ctl[L.keep() + first] == first) ++first;
  b->first_moved = first;
  b->rows.swap(kept);
  // 2. admit from the head of the queue while it fits
  int budget = b->prefill_budget, tokens = 0;
  while (!b->queue.empty()) {
    const Request &q = b->queue.front();
    const long long need = pages_needed(b, q.prompt_len, q.decode_steps);
    if (static_cast<int>(b->rows.size()) >= b->max_slots || b->promised + need > b->pages_free ||
        q.prompt_len > budget)
      break;
    Row r;
    r.req = q;
    b->rows.push_back(r);
    b->promised += need;
    budget -= q.prompt_len;
    tokens += q.prompt_len;
    b->queue.pop_front();
  }
  const int n_rows = static_cast<int>(b->rows.size());
  // 3. the step's positions and packed prompts
  for (int i = 0; i < n_rows; ++i) {
    const int pos = (i >= n_keep) ? b->rows[i].req.prompt_len : b->rows[i].ctx;
    ctl[L.pos() + i] = pos;
    ctl[L.attn() + i] = pos + 1;
  }
  int acc = 0;
  for (int i = n_keep; i < n_rows; ++i) {
    ctl[L.cu() + (i - n_keep)] = acc;
    acc += b->rows[i].req.prompt_len;
  }
  ctl[L.cu() + (n_rows - n_keep)] = acc;
  pa_batch_plan p{};
  p.n_retired = n_ret;
  p.n_keep = n_keep;
  p.n_admitted = n_rows - n_keep;
  p.n_rows = n_rows;
  p.prefill_tokens = tokens;
  p.done = (n_rows == 0 && n_ret == 0) ? 1 : 0;
  b->plan = p;
  b->planned = !p.done;
  *plan = p;
  return PA_OK;
}

extern "C" int pa_batcher_rows(const pa_batcher *b, int64_t *request_ids, int32_t *positions,
                               int cap) {
  if (!b) return PA_ERR_NULL;
  const int n = static_cast<int>(b->rows.size());
  if (cap < n) return PA_ERR_ARG;
  const CtlLayout L{b->max_slots};
  for (int i = 0; i < n; ++i) {
    if (request_ids) request_ids[i] = b->rows[i].req.id;
    if (positions)
      positions[i] = b->planned ? b->ctl[L.pos() + i] : b->rows[i].ctx;
  }
  return n;
}

extern "C" int pa_batcher_retired(const pa_batcher *b, int64_t *request_ids, int cap) {
  if (!b) return PA_ERR_NULL;
  const int n = static_cast<int>(b->retired_ids.size());
  if (cap < n) return PA_ERR_ARG;
  for (int i = 0; i < n; ++i)
    if (request_ids) request_ids[i] = b->retired_ids[i];
  return n;
}

extern "C" int pa_batcher_pending(const pa_batcher *b) {
  if (!b) return PA_ERR_NULL;
  return static_cast<int>(b->queue.size());
}

extern "C" int pa_batcher_commit(pa_batcher *b) {
  if (!b) return PA_ERR_NULL;
  if (!b->planned) return PA_ERR_STATE;
  // prompts are cached, every row took its decode step
  const pa_batch_plan &p = b->plan;
  for (int i = 0; i < p.n_rows; ++i) {
    Row &r = b->rows[i];
    if (i >= p.n_keep) r.ctx = r.req.prompt_len;
    r.ctx += 1;
    r.done += 1;
  }
  b->planned = false;
  return PA_OK;
}

namespace {

// The decode kernel for the planned step's rows: the process-wide path when
// one is forced, else the choice from their attention contexts in the host
// image of the control block.
int decode_path_of(const pa_batcher *b, int n_rows) {
  const int forced = decode_path_setting();
  if (forced != PA_DECODE_AUTO) return forced;
  const CtlLayout L{b->max_slots};
  const int k = pa_decode_kernel_for_lengths(b->ctl.data() + L.attn(), n_rows, b->block_tokens);
  return k > 0 ? k : PA_DECODE_AUTO;
}

// The decode step of rows 0..n_rows-1, every layer: append, then attention
// with the decode kernel `path`.
int enqueue_decode(pa_batcher *b, const pa_batch_buffers *buf, int32_t *ctl, int n_rows,
                   int path, void *stream) {
  const CtlLayout L{b->max_slots};
  const int Lyr = b->n_layers, mb = b->max_blocks;
  const size_t dq = static_cast<size_t>(b->max_slots) * kHq * kD;
  const size_t dk = static_cast<size_t>(b->max_slots) * kHkv * kD;
  for (int l = 0; l < Lyr && n_rows > 0; ++l) {
    int rc = pa_kv_append_rope_bt(buf->decode_k + l * dk, buf->decode_v + l * dk,
                                  buf->decode_q + l * dq, buf->kv_cache, buf->num_blocks,
                                  b->block_tokens, buf->block_table, Lyr, mb, ctl + L.pos(),
                                  n_rows, l, buf->free_list, buf->free_count, buf->err, stream);
    if (rc != PA_OK) return rc;
    rc = decode_attention_path(buf->decode_out + l * dq, buf->decode_q + l * dq, buf->kv_cache,
                               buf->num_blocks, b->block_tokens, buf->block_table, Lyr, mb,
                               ctl + L.attn(), n_rows, l, buf->scale, buf->decode_workspace,
                               buf->decode_workspace_bytes, buf->err, stream, path);
    if (rc != PA_OK) return rc;
  }
  return PA_OK;
}

bool same_buffers(const pa_batch_buffers &a, const pa_batch_buffers &b) {
  return std::memcmp(&a, &b, sizeof(pa_batch_buffers)) == 0;
}

// A decode-only step from a CUDA graph: the control block goes through a
// ring of pinned host buffers (the graph's copy node is repointed at the
// buffer of this step), the graph is captured the first time a batch size
// and buffer set is seen.  Returns PA_OK, or an error before anything was
// enqueued on `stream` (the caller then runs the step eagerly).
int run_decode_graph(pa_batcher *b, const pa_batch_buffers *buf, void *stream) {
  const CtlLayout L{b->max_slots};
  const size_t bytes = L.words() * sizeof(int32_t);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (!b->pinned[0]) {
    for (int i = 0; i < kCtlRing; ++i) {
      if (cudaHostAlloc(reinterpret_cast<void **>(&b->pinned[i]), bytes, cudaHostAllocDefault) !=
              cudaSuccess ||
          cudaEventCreateWithFlags(&b->ring_done[i], cudaEventDisableTiming) != cudaSuccess)
        return PA_ERR_CUDA;
    }
  }
  if (!b->capture_stream &&
      cudaStreamCreateWithFlags(&b->capture_stream, cudaStreamNonBlocking) != cudaSuccess)
    return PA_ERR_CUDA;
  const int slot = b->ring_next;
  if (cudaEventSynchronize(b->ring_done[slot]) != cudaSuccess) return PA_ERR_CUDA;
  std::memcpy(b->pinned[slot], b->ctl.data(), bytes);
  const int n_rows = b->plan.n_rows;
  const int path = decode_path_of(b, n_rows);
  DecodeGraph *g = nullptr;
  for (DecodeGraph &c : b->decode_graphs)
    if (c.n_rows == n_rows && c.path == path && c.device == dev && same_buffers(c.bufs, *buf))
      g = &c;
  int32_t *ctl = static_cast<int32_t *>(buf->ctl);
  if (!g) {
    DecodeGraph ng;
    ng.n_rows = n_rows;
    ng.path = path;
    ng.device = dev;
    ng.bufs = *buf;
    cudaStream_t cs = b->capture_stream;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return PA_ERR_CUDA;
    const bool copied =
        cudaMemcpyAsync(ctl, b->pinned[slot], bytes, cudaMemcpyHostToDevice, cs) == cudaSuccess;
    const int rc = copied ? enqueue_decode(b, buf, ctl, n_rows, path, cs) : PA_ERR_CUDA;
    const cudaError_t ec = cudaStreamEndCapture(cs, &ng.graph);
    if (rc != PA_OK || ec != cudaSuccess) {
      if (ng.graph) cudaGraphDestroy(ng.graph);
      cudaGetLastError();
      return rc != PA_OK ? rc : PA_ERR_CUDA;
    }
    size_t n_nodes = 0;
    cudaGraphGetNodes(ng.graph, nullptr, &n_nodes);
    std::vector<cudaGraphNode_t> nodes(n_nodes);
    cudaGraphGetNodes(ng.graph, nodes.data(), &n_nodes);
    for (cudaGraphNode_t nd : nodes) {
      cudaGraphNodeType t;
      if (cudaGraphNodeGetType(nd, &t) == cudaSuccess && t == cudaGraphNodeTypeMemcpy) {
        ng.ctl_copy = nd;
        break;
      }
    }
    if (!ng.ctl_copy || cudaGraphInstantiate(&ng.exec, ng.graph, 0) != cudaSuccess) {
      cudaGraphDestroy(ng.graph);
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    b->decode_graphs.push_back(ng);
    g = &b->decode_graphs.back();
  } else if (cudaGraphExecMemcpyNodeSetParams1D(g->exec, g->ctl_copy, ctl, b->pinned[slot], bytes,
                                                cudaMemcpyHostToDevice) != cudaSuccess) {
    return PA_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaGraphLaunch(g->exec, st) != cudaSuccess) return PA_ERR_CUDA;
  cudaEventRecord(b->ring_done[slot], st);
  b->ring_next = (slot + 1) % kCtlRing;
  return PA_OK;
}

}  // namespace

extern "C" int pa_batcher_run(pa_batcher *b, const pa_batch_buffers *buf, void *stream) {
  if (!b || !buf) return PA_ERR_NULL;
  if (!b->planned) return PA_ERR_STATE;
  const pa_batch_plan &p = b->plan;
  const CtlLayout L{b->max_slots};
  if (!buf->kv_cache || !buf->block_table || !buf->block_table_tmp || !buf->ctl ||
      !buf->free_list || !buf->free_count || !buf->err)
    return PA_ERR_NULL;
  if (buf->ctl_bytes < L.bytes()) return PA_ERR_ARG;
  if (p.n_admitted > 0 &&
      (!buf->prefill_q || !buf->prefill_k || !buf->prefill_v || !buf->prefill_out))
    return PA_ERR_NULL;
  if (p.n_rows > 0 && (!buf->decode_q || !buf->decode_k || !buf->decode_v || !buf->decode_out))
    return PA_ERR_NULL;
  // a decode-only step (nothing leaves, nothing enters) replays a graph once
  // the kernels' one-time set-up has run eagerly
  if (b->graphs && b->eager_decode_done && p.n_rows > 0 && p.n_retired == 0 &&
      p.n_admitted == 0) {
    if (run_decode_graph(b, buf, stream) == PA_OK) return pa_batcher_commit(b);
    b->graphs = false;   // graphs unavailable here: every step runs eagerly from now on
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t *ctl = static_cast<int32_t *>(buf->ctl);
  // the control block: pageable host memory, staged by the copy before it returns
  if (cudaMemcpyAsync(ctl, b->ctl.data(), L.words() * sizeof(int32_t), cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return PA_ERR_CUDA;
  const int Lyr = b->n_layers, mb = b->max_blocks;
  const int row_words = Lyr * mb;
  int rc;
  // 1. release, then close the gaps
  if (p.n_retired > 0) {
    rc = pa_free_bt(ctl + L.retired(), p.n_retired, b->block_tokens, buf->block_table, Lyr, mb,
                    ctl + L.free_ctx(), buf->free_list, buf->free_count, buf->num_blocks,
                    buf->err, stream);
    if (rc != PA_OK) return rc;
    const int first = b->first_moved;
    if (first < b->n_prev) {
      const int gx = std::min((row_words + kMoveThreads - 1) / kMoveThreads, 64);
      if (first < p.n_keep) {
        gather_rows_kernel<<<dim3(gx, p.n_keep - first), kMoveThreads, 0, st>>>(
            buf->block_table, buf->block_table_tmp, ctl + L.keep(), first, p.n_keep, row_words);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
      }
      place_rows_kernel<<<dim3(gx, b->n_prev - first), kMoveThreads, 0, st>>>(
          buf->block_table, buf->block_table_tmp, first, p.n_keep, b->n_prev, row_words);
      if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
  }
  // 2. prefill of the admitted prompts
  const size_t tq = static_cast<size_t>(b->prefill_budget) * kHq * kD;
  const size_t tk = static_cast<size_t>(b->prefill_budget) * kHkv * kD;
  int32_t *table_new = buf->block_table + static_cast<size_t>(p.n_keep) * row_words;
  for (int l = 0; l < Lyr && p.n_admitted > 0; ++l) {
    rc = pa_prefill_append_rope_bt(buf->prefill_k + l * tk, buf->prefill_v + l * tk,
                                   buf->prefill_q + l * tq, p.prefill_tokens, ctl + L.cu(),
                                   buf->kv_cache, buf->num_blocks, b->block_tokens, table_new,
                                   Lyr, mb, ctl + L.zero(), p.n_admitted, l, buf->free_list,
                                   buf->free_count, buf->err, stream);
    if (rc != PA_OK) return rc;
    rc = pa_prefill_attention_bt(buf->prefill_out + l * tq, buf->prefill_q + l * tq,
                                 p.prefill_tokens, ctl + L.cu(), buf->kv_cache, buf->num_blocks,
                                 b->block_tokens, table_new, Lyr, mb, ctl + L.zero(),
                                 p.n_admitted, l, buf->scale, buf->err, stream);
    if (rc != PA_OK) return rc;
  }
  // 3. one decode step for every active row
  rc = enqueue_decode(b, buf, ctl, p.n_rows, decode_path_of(b, p.n_rows), stream);
  if (rc != PA_OK) return rc;
  if (p.n_rows > 0 && p.n_retired == 0 && p.n_admitted == 0) b->eager_decode_done = true;
  return pa_batcher_commit(b);
}
