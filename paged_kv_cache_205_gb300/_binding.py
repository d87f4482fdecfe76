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
    "pa_kv_append_rope_bt",
    "pa_decode_attention_bt",
    "pa_free_bt",
    "pa_decode_workspace_size_bt",
    "pa_prefill_append_rope_bt",
    "pa_prefill_attention_bt",
    "pa_prefill_set_test_fault",
    "pa_decode_set_grid_limit",
    "pa_error_string",
    "pa_batcher_ctl_bytes",
    "pa_batcher_create",
    "pa_batcher_create_bt",
    "pa_batcher_destroy",
    "pa_batcher_submit",
    "pa_batcher_plan",
    "pa_batcher_rows",
    "pa_batcher_retired",
    "pa_batcher_pending",
    "pa_batcher_run",
    "pa_batcher_commit",
    "pa_batcher_set_graphs",
)

_lock = threading.Lock()
_lib = None


class BatchPlan(ctypes.Structure):
    _fields_ = [("n_retired", ctypes.c_int), ("n_keep", ctypes.c_int),
                ("n_admitted", ctypes.c_int), ("n_rows", ctypes.c_int),
                ("prefill_tokens", ctypes.c_int), ("done", ctypes.c_int)]


class BatchBuffers(ctypes.Structure):
    _fields_ = [("kv_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int),
                ("block_table", ctypes.c_void_p), ("block_table_tmp", ctypes.c_void_p),
                ("ctl", ctypes.c_void_p), ("ctl_bytes", ctypes.c_size_t),
                ("free_list", ctypes.c_void_p), ("free_count", ctypes.c_void_p),
                ("err", ctypes.c_void_p), ("decode_workspace", ctypes.c_void_p),
                ("decode_workspace_bytes", ctypes.c_size_t),
                ("prefill_q", ctypes.c_void_p), ("prefill_k", ctypes.c_void_p),
                ("prefill_v", ctypes.c_void_p), ("prefill_out", ctypes.c_void_p),
                ("decode_q", ctypes.c_void_p), ("decode_k", ctypes.c_void_p),
                ("decode_v", ctypes.c_void_p), ("decode_out", ctypes.c_void_p),
                ("scale", ctypes.c_float)]


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
        lib.pa_kv_append_rope_bt.argtypes = [P, P, P, P, I, I, P, I, I, P, I, I, P, P, P, P]
        lib.pa_kv_append_rope_bt.restype = I
        lib.pa_decode_attention_bt.argtypes = [P, P, P, I, I, P, I, I, P, I, I, F, P, Z, P, P]
        lib.pa_decode_attention_bt.restype = I
        lib.pa_prefill_append_rope_bt.argtypes = [P, P, P, I, P, P, I, I, P, I, I, P, I, I, P, P, P,
                                                  P]
        lib.pa_prefill_append_rope_bt.restype = I
        lib.pa_prefill_attention_bt.argtypes = [P, P, I, P, P, I, I, P, I, I, P, I, I, F, P, P]
        lib.pa_prefill_attention_bt.restype = I
        lib.pa_free_bt.argtypes = [P, I, I, P, I, I, P, P, P, I, P, P]
        lib.pa_free_bt.restype = I
        lib.pa_decode_workspace_size_bt.argtypes = [I, I, I]
        lib.pa_decode_workspace_size_bt.restype = Z
        lib.pa_decode_workspace_size.argtypes = [I, I]
        lib.pa_decode_workspace_size.restype = Z
        lib.pa_free.argtypes = [P, I, P, I, I, P, P, P, I, P, P]
        lib.pa_free.restype = I
        lib.pa_decode_set_grid_limit.argtypes = [I]
        lib.pa_decode_set_grid_limit.restype = I
        lib.pa_decode_set_path.argtypes = [I]
        lib.pa_decode_set_path.restype = I
        lib.pa_decode_set_test_fault.argtypes = [I, ctypes.c_longlong]
        lib.pa_decode_set_test_fault.restype = I
        lib.pa_prefill_set_test_fault.argtypes = [I, ctypes.c_longlong]
        lib.pa_prefill_set_test_fault.restype = I
        lib.pa_decode_set_test_plan.argtypes = [I]
        lib.pa_decode_set_test_plan.restype = I
        lib.pa_decode_kernel_for.argtypes = [I, I]
        lib.pa_decode_kernel_for.restype = I
        lib.pa_decode_kernel_for_lengths.argtypes = [P, I, I]
        lib.pa_decode_kernel_for_lengths.restype = I
        lib.pa_error_string.argtypes = [I]
        lib.pa_error_string.restype = ctypes.c_char_p
        PP = ctypes.POINTER(ctypes.c_void_p)
        lib.pa_batcher_ctl_bytes.argtypes = [I]
        lib.pa_batcher_ctl_bytes.restype = Z
        lib.pa_batcher_create.argtypes = [I, I, I, I, I, PP]
        lib.pa_batcher_create.restype = I
        lib.pa_batcher_create_bt.argtypes = [I, I, I, I, I, I, PP]
        lib.pa_batcher_create_bt.restype = I
        lib.pa_batcher_destroy.argtypes = [P]
        lib.pa_batcher_destroy.restype = I
        lib.pa_batcher_submit.argtypes = [P, ctypes.c_int64, I, I]
        lib.pa_batcher_submit.restype = I
        lib.pa_batcher_plan.argtypes = [P, ctypes.POINTER(BatchPlan)]
        lib.pa_batcher_plan.restype = I
        lib.pa_batcher_rows.argtypes = [P, P, P, I]
        lib.pa_batcher_rows.restype = I
        lib.pa_batcher_retired.argtypes = [P, P, I]
        lib.pa_batcher_retired.restype = I
        lib.pa_batcher_pending.argtypes = [P]
        lib.pa_batcher_pending.restype = I
        lib.pa_batcher_run.argtypes = [P, ctypes.POINTER(BatchBuffers), P]
        lib.pa_batcher_run.restype = I
        lib.pa_batcher_commit.argtypes = [P]
        lib.pa_batcher_commit.restype = I
        lib.pa_batcher_set_graphs.argtypes = [P, I]
        lib.pa_batcher_set_graphs.restype = I
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
def _page_tokens(kv_cache) -> int:
    """Tokens per page of a pool [num_blocks][2][page][8][64]."""
    return int(kv_cache.shape[2]) if kv_cache.dim() == 5 else PA_BLOCK_TOKENS


def pa_kv_append_rope(k_new, v_new, q_or_null, kv_cache, block_table, context_lens, layer,
                      free_list, free_count, err, stream=None):
    """kv_cache [num_blocks][2][page][8][64] bf16 (page 16: pa_kv_append_rope;
    8 or 32: pa_kv_append_rope_bt); block_table [n][L][max_blocks] int32;
    k_new/v_new [n][8][64]; q_or_null [n][32][64] or None; free_count, err: int32[1]."""
    n, n_layers, max_blocks = block_table.shape
    page = _page_tokens(kv_cache)
    args = (_dev(k_new, "k_new", _bf16()), _dev(v_new, "v_new", _bf16()),
            _dev(q_or_null, "q_or_null", _bf16(), optional=True),
            _dev(kv_cache, "kv_cache", _bf16()), int(kv_cache.shape[0]))
    rest = (_dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
            _dev(context_lens, "context_lens", _i32()), int(n), int(layer),
            _dev(free_list, "free_list", _i32()), _dev(free_count, "free_count", _i32()),
            _dev(err, "err", _i32()), _stream(stream))
    if page == PA_BLOCK_TOKENS:
        _check("pa_kv_append_rope", library().pa_kv_append_rope(*args, *rest))
    else:
        _check("pa_kv_append_rope_bt", library().pa_kv_append_rope_bt(*args, page, *rest))


def pa_prefill_append_rope(k_new, v_new, q_or_null, cu_tokens, kv_cache, block_table,
                           context_lens, layer, free_list, free_count, err, stream=None):
    """Packed prompt chunks: k_new/v_new [T][8][64], q_or_null [T][32][64] or None,
    cu_tokens int32 [n+1] (rows of sequence s: cu_tokens[s] .. cu_tokens[s+1]-1);
    kv_cache [num_blocks][2][page][8][64] bf16 (page 16: pa_prefill_append_rope;
    8 or 32: pa_prefill_append_rope_bt); block_table [n][L][max_blocks] int32."""
    n, n_layers, max_blocks = block_table.shape
    if cu_tokens.numel() != n + 1:
        raise ValueError("cu_tokens must hold num_seqs + 1 entries")
    page = _page_tokens(kv_cache)
    args = (_dev(k_new, "k_new", _bf16()), _dev(v_new, "v_new", _bf16()),
            _dev(q_or_null, "q_or_null", _bf16(), optional=True), int(k_new.shape[0]),
            _dev(cu_tokens, "cu_tokens", _i32()),
            _dev(kv_cache, "kv_cache", _bf16()), int(kv_cache.shape[0]))
    rest = (_dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
            _dev(context_lens, "context_lens", _i32()), int(n), int(layer),
            _dev(free_list, "free_list", _i32()), _dev(free_count, "free_count", _i32()),
            _dev(err, "err", _i32()), _stream(stream))
    if page == PA_BLOCK_TOKENS:
        _check("pa_prefill_append_rope", library().pa_prefill_append_rope(*args, *rest))
    else:
        _check("pa_prefill_append_rope_bt",
               library().pa_prefill_append_rope_bt(*args, page, *rest))


def pa_prefill_attention(out, q, cu_tokens, kv_cache, block_table, context_lens, layer, scale,
                         err, stream=None):
    """out/q [T][32][64] bf16, packed as for pa_prefill_append_rope; kv_cache
    [num_blocks][2][page][8][64] (page 16: pa_prefill_attention; 8 or 32:
    pa_prefill_attention_bt)."""
    n, n_layers, max_blocks = block_table.shape
    if cu_tokens.numel() != n + 1:
        raise ValueError("cu_tokens must hold num_seqs + 1 entries")
    page = _page_tokens(kv_cache)
    args = (_dev(out, "out", _bf16()), _dev(q, "q", _bf16()), int(q.shape[0]),
            _dev(cu_tokens, "cu_tokens", _i32()), _dev(kv_cache, "kv_cache", _bf16()),
            int(kv_cache.shape[0]))
    rest = (_dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
            _dev(context_lens, "context_lens", _i32()), int(n), int(layer), float(scale),
            _dev(err, "err", _i32()), _stream(stream))
    if page == PA_BLOCK_TOKENS:
        _check("pa_prefill_attention", library().pa_prefill_attention(*args, *rest))
    else:
        _check("pa_prefill_attention_bt", library().pa_prefill_attention_bt(*args, page, *rest))


def pa_decode_workspace_size(num_seqs: int, max_blocks_per_seq: int,
                             block_tokens: int = PA_BLOCK_TOKENS) -> int:
    if block_tokens == PA_BLOCK_TOKENS:
        return int(library().pa_decode_workspace_size(int(num_seqs), int(max_blocks_per_seq)))
    return int(library().pa_decode_workspace_size_bt(int(num_seqs), int(max_blocks_per_seq),
                                                     int(block_tokens)))


def decode_workspace(num_seqs: int, max_blocks_per_seq: int, device=None,
                     block_tokens: int = PA_BLOCK_TOKENS):
    """A zero-filled uint8 CUDA tensor of pa_decode_workspace_size bytes, the
    state pa_decode_attention expects on first use."""
    torch = _torch()
    n = pa_decode_workspace_size(num_seqs, max_blocks_per_seq, block_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode_attention(out, q, kv_cache, block_table, context_lens, layer, scale, workspace,
                        err, stream=None, num_seqs=None):
    """out/q [n][32][64] bf16; workspace: a CUDA uint8 tensor of at least
    pa_decode_workspace_size bytes.  num_seqs defaults to block_table rows."""
    n_rows, n_layers, max_blocks = block_table.shape
    n = n_rows if num_seqs is None else int(num_seqs)
    page = _page_tokens(kv_cache)
    head = (_dev(out, "out", _bf16()), _dev(q, "q", _bf16()),
            _dev(kv_cache, "kv_cache", _bf16()), int(kv_cache.shape[0]))
    rest = (_dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
            _dev(context_lens, "context_lens", _i32()), n, int(layer), float(scale),
            _dev(workspace, "workspace"), int(workspace.numel() * workspace.element_size()),
            _dev(err, "err", _i32()), _stream(stream))
    if page == PA_BLOCK_TOKENS:
        _check("pa_decode_attention", library().pa_decode_attention(*head, *rest))
    else:
        _check("pa_decode_attention_bt", library().pa_decode_attention_bt(*head, page, *rest))


def pa_free(seq_ids, block_table, context_lens, free_list, free_count, num_blocks, err,
            stream=None, block_tokens=PA_BLOCK_TOKENS):
    n, n_layers, max_blocks = block_table.shape
    ids = (_dev(seq_ids, "seq_ids", _i32()), int(seq_ids.numel()))
    rest = (_dev(block_table, "block_table", _i32()), int(n_layers), int(max_blocks),
            _dev(context_lens, "context_lens", _i32()), _dev(free_list, "free_list", _i32()),
            _dev(free_count, "free_count", _i32()), int(num_blocks), _dev(err, "err", _i32()),
            _stream(stream))
    if block_tokens == PA_BLOCK_TOKENS:
        _check("pa_free", library().pa_free(*ids, *rest))
    else:
        _check("pa_free_bt", library().pa_free_bt(*ids, int(block_tokens), *rest))


def pa_decode_set_grid_limit(max_ctas: int) -> None:
    _check("pa_decode_set_grid_limit", library().pa_decode_set_grid_limit(int(max_ctas)))


PA_DECODE_AUTO, PA_DECODE_SPLIT, PA_DECODE_CLUSTER, PA_DECODE_SEQ = 0, 1, 2, 3


def pa_decode_kernel_for(num_seqs: int, block_tokens: int = PA_BLOCK_TOKENS) -> int:
    """PA_DECODE_SPLIT or PA_DECODE_CLUSTER: the kernel a decode call on
    num_seqs sequences would run now."""
    r = library().pa_decode_kernel_for(int(num_seqs), int(block_tokens))
    _check("pa_decode_kernel_for", min(r, 0))
    return int(r)


def pa_decode_set_test_fault(stage: int, wait_limit_ns: int = 0) -> None:
    """Test hook of the bounded waits (see include/pagedkv.h): stage >= 0
    leaves that stage of the split kernel's CTA 0 without its copies and
    shortens every wait of the split kernel to wait_limit_ns; -1 restores."""
    _check("pa_decode_set_test_fault",
           library().pa_decode_set_test_fault(int(stage), int(wait_limit_ns)))


def pa_prefill_set_test_fault(chunk: int, wait_limit_ns: int = 0) -> None:
    """Test hook of the prefill kernel's bounded waits (see
    include/pagedkv.h): chunk >= 0 leaves that chunk of CTA 0 without its
    copies and shortens every wait of the kernel to wait_limit_ns; -1
    restores."""
    _check("pa_prefill_set_test_fault",
           library().pa_prefill_set_test_fault(int(chunk), int(wait_limit_ns)))


def pa_decode_set_test_plan(mode: int) -> None:
    """Test hook of the per-head kernel's speculative plan (see
    include/pagedkv.h): 1 makes the plan move after the dependency wait, 0
    restores."""
    _check("pa_decode_set_test_plan", library().pa_decode_set_test_plan(int(mode)))


def pa_decode_kernel_for_lengths(context_lens, block_tokens: int = PA_BLOCK_TOKENS) -> int:
    """The decode kernel for a batch whose context lengths are known on the
    host (a sequence of ints); see include/pagedkv.h."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(context_lens, dtype=np.int32))
    rc = library().pa_decode_kernel_for_lengths(a.ctypes.data if a.size else None, int(a.size),
                                                int(block_tokens))
    if rc < 0:
        raise PagedKVError("pa_decode_kernel_for_lengths", rc)
    return rc


def pa_decode_set_path(path: int) -> None:
    """Selects the decode-attention kernel: PA_DECODE_AUTO (default),
    PA_DECODE_SPLIT or PA_DECODE_CLUSTER (process-wide)."""
    _check("pa_decode_set_path", library().pa_decode_set_path(int(path)))


# -------------------------------------------------------- continuous batching
def pa_batcher_ctl_bytes(max_slots: int) -> int:
    return int(library().pa_batcher_ctl_bytes(int(max_slots)))


class Batcher:
    """The library's continuous-batching loop (pa_batcher_*): a queue of
    requests, block-table rows as slots, one planned step at a time."""

    def __init__(self, max_slots, n_layers, max_blocks_per_seq, pages_free, prefill_budget,
                 block_tokens=PA_BLOCK_TOKENS):
        h = ctypes.c_void_p()
        _check("pa_batcher_create_bt", library().pa_batcher_create_bt(
            int(max_slots), int(n_layers), int(max_blocks_per_seq), int(pages_free),
            int(prefill_budget), int(block_tokens), ctypes.byref(h)))
        self._h = h
        self.block_tokens = int(block_tokens)
        self.max_slots = int(max_slots)
        self.n_layers = int(n_layers)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        self.prefill_budget = int(prefill_budget)

    def close(self):
        if self._h:
            library().pa_batcher_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def submit(self, request_id: int, prompt_len: int, decode_steps: int):
        _check("pa_batcher_submit", library().pa_batcher_submit(
            self._h, int(request_id), int(prompt_len), int(decode_steps)))

    def plan(self) -> BatchPlan:
        p = BatchPlan()
        _check("pa_batcher_plan", library().pa_batcher_plan(self._h, ctypes.byref(p)))
        return p

    def rows(self):
        """(request id per row, decode position per row) of the planned step."""
        import numpy as np
        ids = np.zeros(self.max_slots, dtype=np.int64)
        pos = np.zeros(self.max_slots, dtype=np.int32)
        n = library().pa_batcher_rows(self._h, ids.ctypes.data, pos.ctypes.data, self.max_slots)
        if n < 0:
            raise PagedKVError("pa_batcher_rows", n)
        return ids[:n], pos[:n]

    def retired(self):
        import numpy as np
        ids = np.zeros(self.max_slots, dtype=np.int64)
        n = library().pa_batcher_retired(self._h, ids.ctypes.data, self.max_slots)
        if n < 0:
            raise PagedKVError("pa_batcher_retired", n)
        return ids[:n].tolist()

    def pending(self) -> int:
        return int(library().pa_batcher_pending(self._h))

    def commit(self):
        _check("pa_batcher_commit", library().pa_batcher_commit(self._h))

    def set_graphs(self, enable: bool):
        """Replay decode-only steps from CUDA graphs (the default) or not."""
        _check("pa_batcher_set_graphs", library().pa_batcher_set_graphs(self._h, int(bool(enable))))

    def run(self, bufs: "BatchBuffers", stream=None):
        _check("pa_batcher_run", library().pa_batcher_run(self._h, ctypes.byref(bufs),
                                                          _stream(stream)))


def batch_buffers(kv_cache, block_table, block_table_tmp, ctl, free_list, free_count, err,
                  decode_workspace, prefill_q, prefill_k, prefill_v, prefill_out,
                  decode_q, decode_k, decode_v, decode_out, scale) -> BatchBuffers:
    """The pa_batch_buffers of a batcher from torch CUDA tensors (see
    include/pagedkv.h for shapes).  The tensors must outlive every step run
    with the returned structure."""
    b = BatchBuffers()
    b.kv_cache = _dev(kv_cache, "kv_cache", _bf16())
    b.num_blocks = int(kv_cache.shape[0])
    b.block_table = _dev(block_table, "block_table", _i32())
    b.block_table_tmp = _dev(block_table_tmp, "block_table_tmp", _i32())
    b.ctl = _dev(ctl, "ctl")
    b.ctl_bytes = int(ctl.numel() * ctl.element_size())
    b.free_list = _dev(free_list, "free_list", _i32())
    b.free_count = _dev(free_count, "free_count", _i32())
    b.err = _dev(err, "err", _i32())
    b.decode_workspace = _dev(decode_workspace, "decode_workspace")
    b.decode_workspace_bytes = int(decode_workspace.numel() * decode_workspace.element_size())
    for name, t in (("prefill_q", prefill_q), ("prefill_k", prefill_k), ("prefill_v", prefill_v),
                    ("prefill_out", prefill_out), ("decode_q", decode_q), ("decode_k", decode_k),
                    ("decode_v", decode_v), ("decode_out", decode_out)):
        setattr(b, name, _dev(t, name, _bf16()))
    b.scale = float(scale)
    return b
