"""GB300 (sm_103a) PagedAttention decode: Python binding of ``libpagedkv.so``.

The functions below carry the names of the C ABI in ``include/pagedkv.h``
and only marshal arguments: torch CUDA tensors become device pointers and
the current torch stream becomes the ``stream`` argument.  Every step of
the computation runs in the library's CUDA kernels; there is no CPU or
PyTorch fallback, and a missing or unloadable library raises.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    BatchBuffers,
    Batcher,
    BatchPlan,
    batch_buffers,
    pa_batcher_ctl_bytes,
    PA_BLOCK_BYTES,
    PA_BLOCK_TOKENS,
    PA_DEV_BAD_BLOCK,
    PA_DEV_CTX_RANGE,
    PA_DEV_FREE_OVERFLOW,
    PA_DEV_FREE_UNDERFLOW,
    PA_DEV_TIMEOUT,
    PA_HEAD_DIM,
    PA_NUM_KV_HEADS,
    PA_NUM_Q_HEADS,
    PagedKVError,
    decode_workspace,
    exported_symbols,
    library,
    library_path,
    pa_decode_attention,
    pa_decode_set_grid_limit,
    pa_decode_set_path,
    pa_decode_set_test_fault,
    pa_decode_set_test_plan,
    pa_prefill_set_test_fault,
    pa_decode_kernel_for,
    pa_decode_kernel_for_lengths,
    PA_DECODE_AUTO,
    PA_DECODE_SPLIT,
    PA_DECODE_CLUSTER,
    PA_DECODE_SEQ,
    pa_decode_workspace_size,
    pa_error_string,
    pa_free,
    pa_kv_append_rope,
    pa_prefill_append_rope,
    pa_prefill_attention,
)
