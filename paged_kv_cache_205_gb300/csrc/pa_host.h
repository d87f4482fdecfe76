// pa_host.h -- host-side helpers shared by the library's translation units:
// per-device attribute cache, argument checks and launch with programmatic
// dependent launch.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

#include "../../include/pagedkv.h"

namespace pa {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0;
  int minor = 0;
};

// Current device's attributes (cached per device).  Returns PA_OK,
// PA_ERR_CUDA or PA_ERR_DEVICE (not an sm_103 GPU).
int current_device(DeviceInfo *info);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over a pool of num_blocks blocks: dims (d 64, kv head 8, token
// 16, K|V 2, block), box (64, 1, 16, 2, 1) = one kv head's K and V tiles of
// one block, 128-byte swizzle.  Returns PA_OK or PA_ERR_CUDA.
int make_kv_map(CUtensorMap *map, const void *kv_cache, int num_blocks);

// The same over a pool of bt-token pages (8, 16 or 32): box (64, 1, 16, 2, 1)
// for 16, one kv head's K or V rows of a 16-token tile (64, 1, 8 or 16, 1, 1)
// for 8 and 32.
int make_kv_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt);

// Over a pool of 16-token pages, box (64, 1, 16, 1, 1): one kv head's K rows
// (or V rows) of one page, 2 KiB.
int make_kv_rows_map(CUtensorMap *map, const void *kv_cache, int num_blocks);
// The same for pages of bt (8, 16 or 32) tokens: box (64, 1, bt, 1, 1).
int make_kv_rows_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt);
// Over a pool of bt-token pages (16 or 32), box (64, 1, 16, 2, 1): one kv
// head's K and V rows of a 16-token tile (tokens tok0 .. tok0+15 of a page).
int make_kv_tile_map_bt(CUtensorMap *map, const void *kv_cache, int num_blocks, int bt);

// Decode attention with one thread-block cluster per (sequence, kv head)
// (pa_decode_pair.cu), for 16-token pages.  decode_pair_cluster: the cluster
// size for a batch (1, 2, 4 or 8 CTAs per pair), or 0 when the pairs do not
// all fit on the GPU at once (max_ctas > 0 caps the CTAs).
int decode_pair_cluster(int num_seqs, int sm_count, int max_ctas);
// One cluster per sequence (pa_decode_pair.cu): cluster size 1..16 for a
// batch (0: more sequences than CTAs), and the launch over a page map.
int decode_seq_cluster(int num_seqs, int sm_count, int max_ctas);
int launch_decode_seq(const CUtensorMap &page_map, uint16_t *out, const uint16_t *q,
                      const void *kv_cache, int num_blocks, const int32_t *block_table,
                      int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                      int num_seqs, int layer, float scale, int32_t *err, int cluster,
                      cudaStream_t stream);
// Tensor map over a pool of 16-token pages whose box is one whole page:
// dims (d 64, token 16, kv head 8, K|V 2, page), so that shared memory holds
// [K|V][head][token][64] with each head's 16 token rows 128-byte swizzled.
int make_kv_page_map(CUtensorMap *map, const void *kv_cache, int num_blocks);
int launch_decode_pair(const CUtensorMap &map, uint16_t *out, const uint16_t *q,
                       int num_blocks, int block_tokens, const int32_t *block_table, int n_layers,
                       int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                       int layer, float scale, int32_t *err, int cluster, cudaStream_t stream);

// The process-wide decode path set by pa_decode_set_path (pa_decode.cu).
int decode_path_setting();

// pa_decode_attention_bt with the kernel given by `path` (PA_DECODE_*) instead
// of the process-wide setting (pa_decode.cu).
int decode_attention_path(uint16_t *out, const uint16_t *q, const uint16_t *kv_cache,
                          int num_blocks, int block_tokens, const int32_t *block_table,
                          int n_layers, int max_blocks_per_seq, const int32_t *context_lens,
                          int num_seqs, int layer, float scale, void *workspace,
                          size_t workspace_bytes, int32_t *err, void *stream, int path);

// Launch `kernel` with the programmatic-stream-serialization attribute, so it
// may start while the previous kernel on the stream finishes; the kernel
// itself must wait (griddepcontrol.wait) before reading that kernel's output.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pa
