"""ctypes binding of libpagedkv.so (argument marshalling only).

Each function takes torch CUDA tensors, checks dtype / device / layout,
turns them into device pointers and calls the C entry point of the same
name on the current torch CUDA stream (or the stream given).  A non-zero
return code raises PagedKVError.
"""
from __future__ import annotations

import ctypes
import os
import threading

PA_NUM_Q_HEADS = 32
PA_NUM_KV_HEADS = 8
PA_HEAD_DIM = 64
PA_BLOCK_TOKENS = 16
PA_BLOCK_BYTES = 2 * PA_BLOCK_TOKENS * PA_NUM_KV_HEADS * PA_HEAD_DIM * 2

PA_DEV_BAD_BLOCK = 1
PA_DEV_CTX_RANGE = 2
PA_DEV_FREE_UNDERFLOW = 4
PA_DEV_FREE_OVERFLOW = 8
PA_DEV_TIMEOUT = 16

_EXPORTS = (
    "pa_kv_append_rope",
    "pa_decode_attention",
    "pa_decode_attention_static",
    "pa_prefill_append_rope",
    "pa_prefill_attention",
    "pa_decode_workspace_size",
    "pa_free",
    "pa_decode_set_grid_limit",
    "pa_error_string",
)

_lock = threading.Lock()
_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code}: {pa_error_string(code)}")
        self.code = code


def library_path() -> str:
    from . import build
    return build.LIB


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads the in-tree library (building it first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build
        if not os.path.exists(build.LIB) or not build.up_to_date():
            if not build_if_missing:
                raise OSError(f"{build.LIB} is missing; run __graft_entry__.build()")
            build.build_library()
        lib = ctypes.CDLL(build.LIB)
        P, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        lib.pa_kv_append_rope.argtypes = [P, P, P, P, I, P, I, I, P, I, I, P, P, P, P]
        lib.pa_kv_append_rope.restype = I
        lib.pa_decode_attention.argtypes = [P, P, P, I, P, I, I, P, I, I, F, P, Z, P, P]
        lib.pa_decode_attention.restype = I
        lib.pa_prefill_append_rope.argtypes = [P, P, P, I, P, P, I, P, I, I, P, I, I, P, P, P, P]
        lib.pa_prefill_append_rope.restype = I
        lib.pa_prefill_attention.argtypes = [P, P, I, P, P, I, P, I, I, P, I, I, F, P, P]
        lib.pa_prefill_attention.restype = I
        lib.pa_decode_workspace_size.argtypes = [I, I]
        lib.pa_decode_workspace_size.restype = Z
        lib.pa_free.argtypes = [P, I, P, I, I, P, P, P, I, P, P]
        lib.pa_free.restype = I
        lib.pa_decode_set_grid_limit.argtypes = [I]
        lib.pa_decode_set_grid_limit.restype = I
        lib.pa_error_string.argtypes = [I]
        lib.pa_error_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def exported_symbols() -> dict:
    lib = library()
    return {name: hasattr(lib, name) for name in _EXPORTS}


def pa_error_string(code: int) -> str:
    return library().pa_error_string(int(code)).decode()


# ------------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _dev(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if dtype is not None and t.dtype not in dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, rc):
    if rc != 0:
        raise PagedKVError(fn, rc)


def _bf16():
    torch = _torch()
    return (torch.bfloat16, torch.int16, torch.uint16) if hasattr(torch, "uint16") else \
        (torch.bfloat16, torch.int16)


def _i32():
    return (_torch().int32,)


# ------------------------------------------------------------- entry points
def pa_kv_append_rope(k_new, v_new, q_or_null, kv_cache, block_table, context_lens, layer,
                      free_list, free_count, err, stream=None):
    """kv_cache [num_blocks][2][16][8][64] bf16; block_table [n][L][max_blocks] int32;
    k_new/v_new [n][8][64]; q_or_null [n][32][64] or None; free_count, err: int32[1]."""
    n, n_layers, max_blocks = block_table.shape
    rc = library().pa_kv_append_rope(
        _dev(k_new, "k_new", _bf16()), _dev(v_new, "v_new", _bf16()),
        _dev(q_or_null, "q_or_null", _bf16(), optional=True),
        _dev(kv_cache, "kv_cache", _bf16()), int(kv_cache.shape[0]),
        _dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
        _dev(context_lens, "context_lens", _i32()), int(n), int(layer),
        _dev(free_list, "free_list", _i32()), _dev(free_count, "free_count", _i32()),
        _dev(err, "err", _i32()), _stream(stream))
    _check("pa_kv_append_rope", rc)


def pa_prefill_append_rope(k_new, v_new, q_or_null, cu_tokens, kv_cache, block_table,
                           context_lens, layer, free_list, free_count, err, stream=None):
    """Packed prompt chunks: k_new/v_new [T][8][64], q_or_null [T][32][64] or None,
    cu_tokens int32 [n+1] (rows of sequence s: cu_tokens[s] .. cu_tokens[s+1]-1);
    block_table [n][L][max_blocks] int32."""
    n, n_layers, max_blocks = block_table.shape
    if cu_tokens.numel() != n + 1:
        raise ValueError("cu_tokens must hold num_seqs + 1 entries")
    rc = library().pa_prefill_append_rope(
        _dev(k_new, "k_new", _bf16()), _dev(v_new, "v_new", _bf16()),
        _dev(q_or_null, "q_or_null", _bf16(), optional=True), int(k_new.shape[0]),
        _dev(cu_tokens, "cu_tokens", _i32()),
        _dev(kv_cache, "kv_cache", _bf16()), int(kv_cache.shape[0]),
        _dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
        _dev(context_lens, "context_lens", _i32()), int(n), int(layer),
        _dev(free_list, "free_list", _i32()), _dev(free_count, "free_count", _i32()),
        _dev(err, "err", _i32()), _stream(stream))
    _check("pa_prefill_append_rope", rc)


def pa_prefill_attention(out, q, cu_tokens, kv_cache, block_table, context_lens, layer, scale,
                         err, stream=None):
    """out/q [T][32][64] bf16, packed as for pa_prefill_append_rope."""
    n, n_layers, max_blocks = block_table.shape
    if cu_tokens.numel() != n + 1:
        raise ValueError("cu_tokens must hold num_seqs + 1 entries")
    rc = library().pa_prefill_attention(
        _dev(out, "out", _bf16()), _dev(q, "q", _bf16()), int(q.shape[0]),
        _dev(cu_tokens, "cu_tokens", _i32()), _dev(kv_cache, "kv_cache", _bf16()),
        int(kv_cache.shape[0]), _dev(block_table, "block_table", _i32()), int(n_layers),
        int(max_blocks), _dev(context_lens, "context_lens", _i32()), int(n), int(layer),
        float(scale), _dev(err, "err", _i32()), _stream(stream))
    _check("pa_prefill_attention", rc)


def pa_decode_workspace_size(num_seqs: int, max_blocks_per_seq: int) -> int:
    return int(library().pa_decode_workspace_size(int(num_seqs), int(max_blocks_per_seq)))


def decode_workspace(num_seqs: int, max_blocks_per_seq: int, device=None):
    """A zero-filled uint8 CUDA tensor of pa_decode_workspace_size bytes, the
    state pa_decode_attention expects on first use."""
    torch = _torch()
    n = pa_decode_workspace_size(num_seqs, max_blocks_per_seq)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode_attention(out, q, kv_cache, block_table, context_lens, layer, scale, workspace,
                        err, stream=None, num_seqs=None):
    """out/q [n][32][64] bf16; workspace: a CUDA uint8 tensor of at least
    pa_decode_workspace_size bytes.  num_seqs defaults to block_table rows."""
    n_rows, n_layers, max_blocks = block_table.shape
    n = n_rows if num_seqs is None else int(num_seqs)
    rc = library().pa_decode_attention(
        _dev(out, "out", _bf16()), _dev(q, "q", _bf16()), _dev(kv_cache, "kv_cache", _bf16()),
        int(kv_cache.shape[0]), _dev(block_table, "block_table", _i32()), int(n_layers),
        int(max_blocks), _dev(context_lens, "context_lens", _i32()), n, int(layer),
        float(scale), _dev(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
        _dev(err, "err", _i32()), _stream(stream))
    _check("pa_decode_attention", rc)


def pa_free(seq_ids, block_table, context_lens, free_list, free_count, num_blocks, err,
            stream=None):
    n, n_layers, max_blocks = block_table.shape
    rc = library().pa_free(
        _dev(seq_ids, "seq_ids", _i32()), int(seq_ids.numel()),
        _dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
        _dev(context_lens, "context_lens", _i32()), _dev(free_list, "free_list", _i32()),
        _dev(free_count, "free_count", _i32()), int(num_blocks), _dev(err, "err", _i32()),
        _stream(stream))
    _check("pa_free", rc)


def pa_decode_set_grid_limit(max_ctas: int) -> None:
    _check("pa_decode_set_grid_limit", library().pa_decode_set_grid_limit(int(max_ctas)))
