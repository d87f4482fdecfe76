"""The seeded input generator's tables: every (sequence, layer) of a
workload holds ceil(tokens / page) distinct pages of the pool, no page
serves two (sequence, layer) slots unless the workload shares pages across
layers on purpose, the free list holds exactly the rest, and a page size
other than 16 keeps the pool's bytes.  Runs on the CPU."""
import numpy as np
import pytest

import pa_workloads as wl


def _check_tables(bt, ctx, num_blocks, page, free_list, free_count, per_layer_distinct=True):
    n, L, mb = bt.shape
    need = (np.asarray(ctx) + page - 1) // page
    used = []
    for s in range(n):
        for layer in range(L):
            row = bt[s, layer]
            k = int(need[s])
            assert np.all(row[:k] >= 0) and np.all(row[:k] < num_blocks)
            assert np.all(row[k:] == -1)
            used.append(row[:k])
    used = np.concatenate(used) if used else np.zeros(0, np.int32)
    if per_layer_distinct:
        assert len(np.unique(used)) == len(used), "a page serves two slots"
        free = free_list[:free_count]
        assert len(np.unique(free)) == free_count
        assert not np.intersect1d(free, used).size
        assert free_count + len(used) == num_blocks


@pytest.mark.parametrize("page", [8, 16, 32])
@pytest.mark.parametrize("name", ["prompts17_14", "prefill8x2k", "chunked32x512"])
def test_prefill_workload_tables(name, page):
    w = wl.make_prefill_workload(name, block_tokens=page)
    w16 = wl.make_prefill_workload(name)
    assert w.block_tokens == page
    assert w.num_blocks * page == w16.num_blocks * 16            # the pool keeps its bytes
    assert np.array_equal(w.context_lens, w16.context_lens)
    assert np.array_equal(w.chunk_lens, w16.chunk_lens)
    # room in every table row for the chunk's pages
    assert ((w.context_lens + w.chunk_lens + page - 1) // page).max() < w.max_blocks_per_seq
    _check_tables(w.block_table, w.context_lens, w.num_blocks, page, w.free_list, w.free_count)
    # the free list can serve every page the chunks open
    opened = ((w.context_lens + w.chunk_lens + page - 1) // page
              - (w.context_lens + page - 1) // page).sum() * w.n_layers
    assert w.free_count >= opened


@pytest.mark.parametrize("page", [8, 16, 32])
@pytest.mark.parametrize("name", ["llama1b", "long32k", "ragged"])
def test_decode_workload_tables(name, page):
    w = wl.make_workload(name, block_tokens=page)
    assert w.block_tokens == page
    assert w.num_blocks * page == wl.make_workload(name).num_blocks * 16
    _check_tables(w.block_table, w.context_lens, w.num_blocks, page, w.free_list, w.free_count)


def test_page_sizes_other_than_8_16_32_are_refused():
    with pytest.raises(ValueError):
        wl.make_prefill_workload("prefill8x2k", block_tokens=12)
    with pytest.raises(ValueError):
        wl.make_workload("llama1b", block_tokens=64)


@pytest.mark.parametrize("name", ["prefill8x2k", "chunked32x512"])
def test_prefill_workload_first_layers_only(name):
    """layers=k keeps the prompts, chunks and cached contexts, the first k
    layers' tables and a pool scaled by k / n_layers (rounded up), and the
    free list still serves every page the chunks open (the one-layer case is
    the small-footprint profile of a workload)."""
    full = wl.make_prefill_workload(name)
    for k in (1, 3):
        w = wl.make_prefill_workload(name, layers=k)
        assert w.n_layers == k
        assert w.num_blocks == -(-full.num_blocks * k // full.n_layers)
        assert np.array_equal(w.context_lens, full.context_lens)
        assert np.array_equal(w.chunk_lens, full.chunk_lens)
        _check_tables(w.block_table, w.context_lens, w.num_blocks, 16, w.free_list, w.free_count)
        opened = ((w.context_lens + w.chunk_lens + 15) // 16 - (w.context_lens + 15) // 16).sum() * k
        assert w.free_count >= opened
    with pytest.raises(ValueError):
        wl.make_prefill_workload(name, layers=full.n_layers + 1)
