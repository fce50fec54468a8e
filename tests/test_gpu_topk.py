"""Wide-row top-k candidates and the exact merge on the GPU against the
oracle: ids bit-exact in rank order, values bit-exact (the row's own fp32
entries, -0.0 included), status bits as the oracle's non-finite count."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import gpu_env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    moe, dev = gpu_env()
    return moe, dev


def gpu_candidates(env, rows, k, ld=None):
    import torch
    moe, dev = env
    T, N = rows.shape
    ld = N + (-N) % 4 if ld is None else ld
    buf = np.full((T, ld), 1e30, np.float32)  # padding past N must never be read
    buf[:, :N] = rows
    L = torch.from_numpy(buf).to(dev)
    ids = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    vals = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
    ws_bytes = moe.moe_topk_workspace_bytes(T, N)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    moe.moe_topk_candidates(L, T, ld, N, k, ids, vals, ws, ws_bytes)
    return ids.cpu().numpy(), vals.cpu().numpy(), moe.moe_read_status(ws)


def gpu_merge(env, li, lv):
    import torch
    moe, dev = env
    T, n_lists, k = li.shape
    ids = torch.from_numpy(np.ascontiguousarray(li, np.int32)).to(dev)
    vals = torch.from_numpy(np.ascontiguousarray(lv, np.float32)).to(dev)
    oi = torch.full((T, k), -7, dtype=torch.int32, device=dev)
    ov = torch.full((T, k), -7.0, dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    moe.moe_topk_merge(ids, vals, T, n_lists, k, oi, ov, ws, 256)
    return oi.cpu().numpy(), ov.cpu().numpy(), moe.moe_read_status(ws)


def same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32),
                          np.asarray(b, np.float32).view(np.uint32))


def check(env, rows, k, ld=None):
    ids, vals, status = gpu_candidates(env, rows, k, ld)
    rid, rv, bad = oracle.candidates_topk(rows, k)
    assert np.array_equal(ids, rid), np.argwhere(ids != rid)[:5]
    assert same_bits(vals, rv)
    assert status == (env[0].DEV_NONFINITE if bad else 0)
    return ids, vals


# widths around the 1024-column warp chunks and the 8-warp CTA, ragged tails
@pytest.mark.parametrize("N", [16, 100, 1023, 1024, 1025, 8191, 8192, 8193, 20011, 65536 + 12])
@pytest.mark.parametrize("k", [1, 8, 9, 13, 16])
def test_candidates_match_oracle(env, N, k):
    rows = W.make_candidate_logits(3, N, seed=N % 97 + k)
    check(env, rows, k)


def test_candidates_full_vocabulary(env):
    rows = W.make_candidate_logits(W.CANDIDATES_T, W.CANDIDATES_N, seed=0)
    check(env, rows, W.CANDIDATES_K)


@pytest.mark.parametrize("k", [2, 11, 15])
def test_candidates_row_stride(env, k):
    rows = W.make_candidate_logits(5, 9000, seed=4)
    check(env, rows, k, ld=9000 + 44)


def test_candidates_ties_and_signed_zeros(env):
    N = 5000
    rows = np.zeros((4, N), np.float32)
    rows[1, 1::3] = -0.0          # -0 and +0 tie: ids 0..15 in order
    rows[2] = -1.0
    rows[2, 4000:] = -0.0         # the best are -0.0 entries, lowest ids first
    rows[3] = W.int_uniform(N, W.stream_key(9, "misc"), -1, 1).astype(np.float32)
    ids, vals = check(env, rows, 16)
    assert list(ids[1]) == list(range(16))
    assert list(ids[2]) == list(range(4000, 4016))
    assert (np.signbit(vals[2])).all()


def test_candidates_nonfinite_rows(env):
    rows = W.make_candidate_logits(4, 17000, seed=5)
    rows[1, 16999] = np.nan
    rows[2, 8192] = np.inf
    rows[3, 0] = -np.inf
    ids, vals = check(env, rows, 16)
    assert (ids[1:] == -1).all() and (vals[1:] == 0).all() and (ids[0] >= 0).all()


@pytest.mark.parametrize("n_shards", [2, 5])
@pytest.mark.parametrize("k", [4, 16])
def test_shard_merge_equals_the_whole_row(env, n_shards, k):
    rows = W.make_candidate_logits(W.CANDIDATES_T, 40000, seed=6)
    T, N = rows.shape
    cuts = [int(c) // 4 * 4 for c in np.linspace(0, N, n_shards + 1)]
    cuts[-1] = N
    li = np.empty((T, n_shards, k), np.int32)
    lv = np.empty((T, n_shards, k), np.float32)
    for s in range(n_shards):
        a, b = cuts[s], cuts[s + 1]
        si, sv, st = gpu_candidates(env, np.ascontiguousarray(rows[:, a:b]), k)
        assert st == 0
        li[:, s], lv[:, s] = si + a, sv
    mi, mv, st = gpu_merge(env, li, lv)
    wi, wv, _ = oracle.candidates_topk(rows, k)
    assert st == 0
    assert np.array_equal(mi, wi) and same_bits(mv, wv)


def test_merge_many_unsorted_lists(env):
    # 300 lists per row (more than one per thread of the merging CTA), each
    # a shard's top-9 in shuffled order
    T, n_lists, k, width = 3, 300, 9, 64
    rows = W.make_candidate_logits(T, n_lists * width, seed=8)
    li = np.empty((T, n_lists, k), np.int32)
    lv = np.empty((T, n_lists, k), np.float32)
    rng = np.random.default_rng(1)
    for s in range(n_lists):
        si, sv, _ = oracle.candidates_topk(np.ascontiguousarray(rows[:, s * width:(s + 1) * width]), k)
        p = rng.permutation(k)
        li[:, s], lv[:, s] = (si + s * width)[:, p], sv[:, p]
    mi, mv, st = gpu_merge(env, li, lv)
    ri, rv, _ = oracle.merge_topk(li, lv, k)
    assert st == 0
    assert np.array_equal(mi, ri) and same_bits(mv, rv)


def test_merge_sentinel_rows(env):
    rows = W.make_candidate_logits(3, 3000, seed=2)
    rows[1, 5] = np.nan
    ids, vals, _ = oracle.candidates_topk(rows, 16)
    li = np.stack([ids, ids + 0], axis=1)
    li[:, 1] = np.where(li[:, 1] >= 0, li[:, 1] + 3000, -1)
    lv = np.stack([vals, vals], axis=1)
    mi, mv, st = gpu_merge(env, li, lv)
    ri, rv, bad = oracle.merge_topk(li, lv, 16)
    assert bad == 1 and st == env[0].DEV_NONFINITE
    assert np.array_equal(mi, ri) and same_bits(mv, rv)


def test_candidates_widest_row(env):
    # the largest N the call takes (2^24 columns, one 64 MB row) and a ragged
    # width just below it
    for N in (1 << 24, (1 << 24) - 3):
        rows = W.make_candidate_logits(1, N, seed=12)
        check(env, rows, 16)


@pytest.mark.parametrize("n_lists,k", [(65536, 1), (4096, 16)])
def test_merge_most_lists(env, n_lists, k):
    # the largest list count the merge takes, and 4096 lists of 16: lists
    # of random distinct ids with values from a tie-heavy integer draw
    T = 2
    rng = np.random.default_rng(n_lists + k)
    ids = np.stack([rng.permutation(n_lists * k * 4)[: n_lists * k] for _ in range(T)])
    vals = rng.integers(-50, 50, size=(T, n_lists * k)).astype(np.float32)
    li = ids.reshape(T, n_lists, k).astype(np.int32)
    lv = vals.reshape(T, n_lists, k)
    mi, mv, st = gpu_merge(env, li, lv)
    ri, rv, bad = oracle.merge_topk(li, lv, k)
    assert st == 0 and bad == 0
    assert np.array_equal(mi, ri) and same_bits(mv, rv)
