"""CPU oracle for the PagedAttention decode step and the KV append with RoPE.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product
package ``paged_kv_cache_205_gb300`` never does, and the two share no code.

The arithmetic lives in plain C (``pa_oracle.c``, fp64 throughout), built
with gcc into ``oracle/_build/liboracle.so``; this module only marshals
numpy arrays.  bf16 tensors are passed as ``uint16`` arrays of raw bits.

Page followed: "An Inference Engine in 1,500 Lines of CUDA: The Map"
(tiny-vllm series part 1), sections "What is in the box" and "The path of
one inference".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

# the same error bits as pa_oracle.h
ERR_BAD_BLOCK = 1
ERR_CTX_RANGE = 2
ERR_FREE_UNDERFLOW = 4
ERR_FREE_OVERFLOW = 8

# Llama-3 RoPE arguments of init_rope_frequencies ("The path of one inference")
ROPE_THETA = 500000.0
ROPE_FACTOR = 32.0
ROPE_LOW = 1.0
ROPE_HIGH = 4.0
ROPE_ORIGINAL = 8192.0

N_KV = 8
N_Q = 32
HEAD_DIM = 64
BLOCK = 16


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(_SRC[:-1] + "h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_llama3_inv_freq.argtypes = [I, D, D, D, D, D, P]
        lib.oracle_llama3_inv_freq.restype = None
        lib.oracle_llama3_scale_freq.argtypes = [D, D, D, D, D]
        lib.oracle_llama3_scale_freq.restype = D
        lib.oracle_rope_rotate.argtypes = [P, I, D, P, P]
        lib.oracle_rope_rotate.restype = None
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = D
        lib.oracle_double_to_bf16.argtypes = [D]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_decode_attention_bt.argtypes = [P, P, P, I, P, I, I, P, I, I, D, I]
        lib.oracle_decode_attention_bt.restype = I
        lib.oracle_attention_partial_bt.argtypes = [P, P, I, P, I, I, I, D, P, P, P, I]
        lib.oracle_attention_partial_bt.restype = I
        lib.oracle_merge_partials.argtypes = [I, P, P, P, P]
        lib.oracle_merge_partials.restype = None
        lib.oracle_kv_append_rope_bt.argtypes = [P, P, P, P, I, P, I, I, P, I, I, P, P, P, I]
        lib.oracle_kv_append_rope_bt.restype = I
        lib.oracle_prefill_append_rope_bt.argtypes = [P, P, P, P, P, I, P, I, I, P, I, I, P, P, P,
                                                       I]
        lib.oracle_prefill_append_rope_bt.restype = I
        lib.oracle_prefill_attention_bt.argtypes = [P, P, P, P, I, P, I, I, P, I, I, D, I]
        lib.oracle_prefill_attention_bt.restype = I
        lib.oracle_free_bt.argtypes = [P, I, P, I, I, P, P, P, I, I]
        lib.oracle_free_bt.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ RoPE
def llama3_inv_freq(head_dim: int = HEAD_DIM, theta: float = ROPE_THETA,
                    factor: float = ROPE_FACTOR, low: float = ROPE_LOW,
                    high: float = ROPE_HIGH, original: float = ROPE_ORIGINAL) -> np.ndarray:
    out = np.zeros(head_dim // 2, dtype=np.float64)
    _load().oracle_llama3_inv_freq(head_dim, theta, factor, low, high, original, _ptr(out))
    return out


def llama3_scale_freq(inv_freq: float, factor: float = ROPE_FACTOR, low: float = ROPE_LOW,
                      high: float = ROPE_HIGH, original: float = ROPE_ORIGINAL) -> float:
    return _load().oracle_llama3_scale_freq(float(inv_freq), factor, low, high, original)


def rope_rotate(x: np.ndarray, pos: float, inv_freq: np.ndarray | None = None) -> np.ndarray:
    x = _c(x, np.float64)
    inv = llama3_inv_freq(x.shape[-1]) if inv_freq is None else _c(inv_freq, np.float64)
    out = np.zeros_like(x)
    _load().oracle_rope_rotate(_ptr(x), x.shape[-1], float(pos), _ptr(inv), _ptr(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (pure bit shift, no rounding)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.fromiter((lib.oracle_double_to_bf16(float(v)) for v in flat),
                      dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(x))


# ------------------------------------------------------------- attention
def decode_attention(q, pool, block_table, context_lens, layer, scale=0.125,
                     num_blocks=None, block_tokens=BLOCK):
    """out[num_seqs][32][64] fp64, plus the error bits.  pool
    [num_blocks][2][block_tokens][8][64]."""
    q = _c(q, np.uint16)
    pool = _c(pool, np.uint16)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    n, n_layers, max_blocks = bt.shape
    nb = pool.shape[0] if num_blocks is None else num_blocks
    out = np.zeros((n, N_Q, HEAD_DIM), dtype=np.float64)
    err = _load().oracle_decode_attention_bt(_ptr(out), _ptr(q), _ptr(pool), nb, _ptr(bt),
                                             n_layers, max_blocks, _ptr(ctx), n, layer,
                                             float(scale), int(block_tokens))
    if err < 0:
        raise MemoryError("oracle allocation failed")
    return out, err


def attention_partial(q_head, pool, bt_row, kv_head, t_begin, t_end, scale=0.125,
                      block_tokens=BLOCK):
    q_head = _c(q_head, np.uint16)
    pool = _c(pool, np.uint16)
    row = _c(bt_row, np.int32)
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(HEAD_DIM)
    err = _load().oracle_attention_partial_bt(_ptr(q_head), _ptr(pool), pool.shape[0],
                                              _ptr(row), kv_head, t_begin, t_end, float(scale),
                                              _ptr(m), _ptr(l), _ptr(acc), int(block_tokens))
    return float(m[0]), float(l[0]), acc, err


def merge_partials(m, l, acc):
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    acc = _c(acc, np.float64)
    out = np.zeros(HEAD_DIM)
    _load().oracle_merge_partials(len(m), _ptr(m), _ptr(l), _ptr(acc), _ptr(out))
    return out


# ---------------------------------------------------------------- append
def kv_append_rope(k_new, v_new, q, pool, block_table, context_lens, layer,
                   free_list, free_count, num_blocks=None, block_tokens=BLOCK):
    """In-place on copies: returns (q_rot or None, pool, block_table, free_list,
    free_count, err).  Inputs are not modified."""
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    qc = None if q is None else np.array(q, dtype=np.uint16, copy=True, order="C")
    poolc = np.array(pool, dtype=np.uint16, copy=True, order="C")
    btc = np.array(block_table, dtype=np.int32, copy=True, order="C")
    flc = np.array(free_list, dtype=np.int32, copy=True, order="C")
    fc = np.array([free_count], dtype=np.int32)
    ctx = _c(context_lens, np.int32)
    inv = llama3_inv_freq()
    n, n_layers, max_blocks = btc.shape
    nb = poolc.shape[0] if num_blocks is None else num_blocks
    err = _load().oracle_kv_append_rope_bt(_ptr(k_new), _ptr(v_new), _ptr(qc), _ptr(poolc), nb,
                                           _ptr(btc), n_layers, max_blocks, _ptr(ctx), n, layer,
                                           _ptr(flc), _ptr(fc), _ptr(inv), int(block_tokens))
    return qc, poolc, btc, flc, int(fc[0]), err


def prefill_append_rope(k_new, v_new, q, cu_tokens, pool, block_table, context_lens, layer,
                        free_list, free_count, num_blocks=None, block_tokens=BLOCK):
    """Returns (q_rot or None, pool, block_table, free_list, free_count, err)
    on copies; the inputs are not modified.  Pages of block_tokens tokens:
    pool [num_blocks][2][block_tokens][8][64]."""
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    qc = None if q is None else np.array(q, dtype=np.uint16, copy=True, order="C")
    cu = _c(cu_tokens, np.int32)
    poolc = np.array(pool, dtype=np.uint16, copy=True, order="C")
    btc = np.array(block_table, dtype=np.int32, copy=True, order="C")
    flc = np.array(free_list, dtype=np.int32, copy=True, order="C")
    fc = np.array([free_count], dtype=np.int32)
    ctx = _c(context_lens, np.int32)
    inv = llama3_inv_freq()
    n, n_layers, max_blocks = btc.shape
    nb = poolc.shape[0] if num_blocks is None else num_blocks
    err = _load().oracle_prefill_append_rope_bt(_ptr(k_new), _ptr(v_new), _ptr(qc), _ptr(cu),
                                                _ptr(poolc), nb, _ptr(btc), n_layers, max_blocks,
                                                _ptr(ctx), n, layer, _ptr(flc), _ptr(fc), _ptr(inv),
                                                int(block_tokens))
    return qc, poolc, btc, flc, int(fc[0]), err


def prefill_attention(q, cu_tokens, pool, block_table, context_lens, layer, scale=0.125,
                      num_blocks=None, block_tokens=BLOCK):
    """out[rows][32][64] fp64 and the error bits; pages of block_tokens tokens."""
    q = _c(q, np.uint16)
    cu = _c(cu_tokens, np.int32)
    pool = _c(pool, np.uint16)
    bt = _c(block_table, np.int32)
    ctx = _c(context_lens, np.int32)
    n, n_layers, max_blocks = bt.shape
    nb = pool.shape[0] if num_blocks is None else num_blocks
    out = np.zeros((q.shape[0], N_Q, HEAD_DIM), dtype=np.float64)
    err = _load().oracle_prefill_attention_bt(_ptr(out), _ptr(q), _ptr(cu), _ptr(pool), nb,
                                              _ptr(bt), n_layers, max_blocks, _ptr(ctx), n, layer,
                                              float(scale), int(block_tokens))
    if err < 0:
        raise MemoryError("oracle allocation failed")
    return out, err


def free(seq_ids, block_table, context_lens, free_list, free_count, num_blocks,
         block_tokens=BLOCK):
    """Returns (block_table, free_list, free_count, err) on copies."""
    ids = _c(seq_ids, np.int32)
    btc = np.array(block_table, dtype=np.int32, copy=True, order="C")
    flc = np.array(free_list, dtype=np.int32, copy=True, order="C")
    fc = np.array([free_count], dtype=np.int32)
    ctx = _c(context_lens, np.int32)
    n, n_layers, max_blocks = btc.shape
    err = _load().oracle_free_bt(_ptr(ids), len(ids), _ptr(btc), n_layers, max_blocks,
                                 _ptr(ctx), _ptr(flc), _ptr(fc), num_blocks, int(block_tokens))
    return btc, flc, int(fc[0]), err
