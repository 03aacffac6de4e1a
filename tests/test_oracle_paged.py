"""Pins for the oracle's paged-KV row gather (CPU only).

The page-table reading (segment b owns table entries
[page_indptr[b], page_indptr[b+1]); row i is slot i % page_size of page
page_indices[page_indptr[b] + i // page_size]; a segment of n pages has
(n - 1) * page_size + last_page_len[b] rows, n rows when page_size is 1) is
checked against the pages' own call, a small table worked out by hand, and
invariants that a swapped quotient/remainder, a dropped offset or a wrong
length rule would break.
"""
import numpy as np

from mla_decode_attention_split_gb300 import synth


def _labelled_pool(num_pages, page_size):
    # row value = 10 * page + slot, so every gathered row names where it came from
    return (10 * np.arange(num_pages)[:, None] + np.arange(page_size)[None, :]).astype(np.int64)


def test_page_size_one_with_identity_indices_is_the_contiguous_cache(oracle_mod):
    # kernelbot-amd-mixed-mla-753817, the paged call: page_size 1,
    # kv_indices = arange(total_kv), kv_last_page_len = the segment lengths,
    # and the row indptr reused as the page indptr
    lens = [3, 0, 5, 1]
    kv_indptr = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    rng = np.random.default_rng(1)
    flat = rng.integers(0, 256, size=(int(kv_indptr[-1]), 4)).astype(np.uint8)
    rows, kvp = oracle_mod.paged_rows(flat[:, None, :], kv_indptr, np.arange(kv_indptr[-1]), np.array(lens), 1)
    assert np.array_equal(rows, flat)
    assert np.array_equal(kvp, kv_indptr)


def test_hand_worked_table(oracle_mod):
    # page_size 3, five pages; rows worked out by hand from the reading above:
    #   segment 0: pages [4, 1], last 2  -> 40 41 42 10 11
    #   segment 1: pages [0],    last 1  -> 0
    #   segment 2: no pages              -> (empty)
    #   segment 3: pages [2, 2, 3], last 3 -> 20 21 22 20 21 22 30 31 32
    pool = _labelled_pool(5, 3)
    rows, kvp = oracle_mod.paged_rows(pool, [0, 2, 3, 3, 6], [4, 1, 0, 2, 2, 3], [2, 1, 3, 3], 3)
    assert rows.tolist() == [40, 41, 42, 10, 11, 0, 20, 21, 22, 20, 21, 22, 30, 31, 32]
    assert kvp.tolist() == [0, 5, 6, 6, 15]


def test_consecutive_pages_are_a_slice_of_the_flat_pool(oracle_mod):
    # pages i, i+1, ... in order are rows i*ps ... of the flattened pool
    ps, num_pages = 7, 9
    pool = np.arange(num_pages * ps * 2).reshape(num_pages, ps, 2)
    flat = pool.reshape(-1, 2)
    rows, kvp = oracle_mod.paged_rows(pool, [0, 3, 9], [2, 3, 4, 0, 1, 2, 3, 4, 5], [5, 7], ps)
    assert np.array_equal(rows[: kvp[1]], flat[2 * ps: 2 * ps + 2 * ps + 5])
    assert np.array_equal(rows[kvp[1]:], flat[0: 6 * ps])


def test_relabelling_the_pool_leaves_the_rows_unchanged(oracle_mod):
    rng = np.random.default_rng(4)
    ps, num_pages = 4, 11
    pool = rng.integers(0, 1000, size=(num_pages, ps, 3))
    pip = np.array([0, 4, 4, 7, 11])
    idx = rng.permutation(num_pages)
    last = np.array([1, 2, 4, 3])
    rows, kvp = oracle_mod.paged_rows(pool, pip, idx, last, ps)
    perm = rng.permutation(num_pages)  # new id of old page j is perm[j]
    pool2 = np.empty_like(pool)
    pool2[perm] = pool
    rows2, kvp2 = oracle_mod.paged_rows(pool2, pip, perm[idx], last, ps)
    assert np.array_equal(rows, rows2) and np.array_equal(kvp, kvp2)
    assert kvp.tolist() == [0, 13, 13, 25, 40]  # (4-1)*4+1, empty, (3-1)*4+4, (4-1)*4+3


def test_generated_page_tables_follow_the_reading(oracle_mod):
    lens = [1, 63, 64, 65, 0, 300]
    for ps in (1, 7, 16, 64):
        w = synth.Workload("paged", len(lens), 1, 0, synth.BF16, synth.FP8_E4M3, seed=3)
        inp = synth.make_paged_inputs(w, "cpu", kv_lens=lens, page_size=ps, spare_pages=5)
        rows, kvp = oracle_mod.paged_rows(inp.kv_pages.numpy(), inp.page_indptr.numpy(), inp.page_indices.numpy(),
                                          inp.last_page_len.numpy(), ps)
        assert np.diff(kvp).tolist() == lens
        assert rows.shape == (sum(lens), synth.D_QK)
        # every pool page is used at most once
        idx = inp.page_indices.numpy()
        assert len(set(idx.tolist())) == idx.size
    inp = synth.make_paged_inputs(w, "cpu", kv_lens=lens, page_size=1, lengths_as_last=True)
    assert inp.last_page_len.tolist() == lens
