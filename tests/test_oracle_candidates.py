"""Pins of the oracle's wide top-k candidate selection and its exact merge.

The candidate selector of the DFlash2 drafter takes up to 16 lm_head
candidates per block position on the GPU (lucebox commit list, "candidate
selector head"), and the two-GPU drafter splits the vocabulary and joins the
halves with an exact top-16 merge (ninfer-tp2 v0.4.0 notes).  Each check
compares the oracle with something it does not compute: numpy's lexsort,
Python's own sort, a hand-derived case, or the exactness property of the
merge (the union of the shards' top-k lists holds the row's top-k).
"""
import numpy as np
import pytest

import oracle
import workloads as W


def lexsort_ids(row, K):
    """numpy's stable lexsort on (id, -value): value descending, id ascending.
    -0.0 and +0.0 compare equal in both keys, so they tie."""
    ids = np.arange(row.size)
    neg = -row.astype(np.float64)
    neg[neg == 0] = 0.0
    return np.lexsort((ids, neg))[:K]


@pytest.mark.parametrize("K", [1, 8, 9, 11, 13, 15, 16])
def test_candidates_match_lexsort_on_wide_rows(K):
    rows = W.make_candidate_logits(4, 20011, seed=7)
    ids, vals, bad = oracle.candidates_topk(rows, K)
    assert bad == 0
    for t in range(rows.shape[0]):
        want = lexsort_ids(rows[t], K)
        assert list(ids[t]) == list(want)
        assert np.array_equal(vals[t], rows[t][want])


def test_candidates_full_vocabulary_width():
    rows = W.make_candidate_logits(2, W.CANDIDATES_N, seed=3)
    ids, vals, _ = oracle.candidates_topk(rows, 16)
    for t in range(2):
        assert list(ids[t]) == list(lexsort_ids(rows[t], 16))
        # the 16th value bounds every unselected entry; ties there go to lower ids
        rest = np.setdiff1d(np.arange(rows.shape[1]), ids[t])
        assert rows[t][rest].max() <= vals[t][-1]
        tied = rest[rows[t][rest] == vals[t][-1]]
        assert tied.size == 0 or tied.min() > ids[t][vals[t] == vals[t][-1]].max()


def test_candidates_python_sort_with_signed_zeros():
    row = np.array([0.0, -0.0, 1.0, -0.0, 0.0, 1.0, -1.0] * 5, np.float32)
    ids, _, _ = oracle.candidates_topk(row[None, :], 16)
    want = sorted(range(row.size), key=lambda i: (-float(row[i]) + 0.0, i))[:16]
    assert list(ids[0]) == want


def test_merge_hand_derived_case():
    # shard A holds ids 0..3, shard B ids 4..7; each list is its shard's top-3
    # A values [5, 1, 5, 2] -> (5,0) (5,2) (2,3);  B [5, 7, 0, 5] -> (7,5) (5,4) (5,7)
    ids = np.array([[[0, 2, 3], [5, 4, 7]]], np.int32)
    vals = np.array([[[5, 5, 2], [7, 5, 5]]], np.float32)
    out_i, out_v, bad = oracle.merge_topk(ids, vals, 3)
    assert bad == 0
    assert list(out_i[0]) == [5, 0, 2]
    assert list(out_v[0]) == [7, 5, 5]


@pytest.mark.parametrize("n_shards", [2, 3, 7])
@pytest.mark.parametrize("K", [1, 9, 16])
def test_merge_of_shard_lists_is_the_row_topk(n_shards, K):
    rows = W.make_candidate_logits(4, 5003, seed=11)
    T, N = rows.shape
    cuts = np.linspace(0, N, n_shards + 1).astype(int)
    li = np.empty((T, n_shards, K), np.int32)
    lv = np.empty((T, n_shards, K), np.float32)
    for s in range(n_shards):
        a, b = cuts[s], cuts[s + 1]
        si, sv, _ = oracle.candidates_topk(np.ascontiguousarray(rows[:, a:b]), K)
        li[:, s] = si + a
        lv[:, s] = sv
    mi, mv, bad = oracle.merge_topk(li, lv, K)
    wi, wv, _ = oracle.candidates_topk(rows, K)
    assert bad == 0
    assert np.array_equal(mi, wi) and np.array_equal(mv, wv)


def test_merge_ignores_list_and_entry_order():
    rows = W.make_candidate_logits(2, 4096, seed=5)
    K = 16
    li = np.empty((2, 4, K), np.int32)
    lv = np.empty((2, 4, K), np.float32)
    for s in range(4):
        si, sv, _ = oracle.candidates_topk(np.ascontiguousarray(rows[:, s * 1024:(s + 1) * 1024]), K)
        li[:, s], lv[:, s] = si + s * 1024, sv
    a_i, a_v, _ = oracle.merge_topk(li, lv, K)
    rng = np.random.default_rng(0)
    flat_i, flat_v = li.reshape(2, -1), lv.reshape(2, -1)
    for t in range(2):
        p = rng.permutation(flat_i.shape[1])
        flat_i[t], flat_v[t] = flat_i[t][p], flat_v[t][p]
    b_i, b_v, _ = oracle.merge_topk(flat_i.reshape(2, 4, K), flat_v.reshape(2, 4, K), K)
    assert np.array_equal(a_i, b_i) and np.array_equal(a_v, b_v)


def test_nonfinite_rows_and_lists_get_sentinels():
    rows = W.make_candidate_logits(3, 3000, seed=2)
    rows[1, 2999] = np.nan
    rows[2, 0] = -np.inf
    ids, vals, bad = oracle.candidates_topk(rows, 16)
    assert bad == 2
    assert ids[0, 0] >= 0
    for t in (1, 2):
        assert (ids[t] == -1).all() and (vals[t] == 0).all()
    li = np.stack([ids, ids], axis=1)
    lv = np.stack([vals, vals], axis=1)
    mi, mv, mbad = oracle.merge_topk(li, lv, 16)
    assert mbad == 2 and (mi[1:] == -1).all() and (mv[1:] == 0).all()
