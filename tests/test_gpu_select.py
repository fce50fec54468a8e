"""A2 selector on the GPU against the oracle: bit-exact ids and order on the
same fp32 logits, softmax weights within 1e-6, sigmoid gate within 1e-6."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import WEIGHT_ABS, gpu_env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch
    moe, dev = gpu_env()
    ws = torch.zeros(1 << 12, dtype=torch.uint8, device=dev)
    return moe, dev, ws


def run_select(env, logits, gate=None, ld=256):
    import torch
    moe, dev, ws = env
    T = logits.shape[0]
    buf = np.zeros((T, ld), np.float32)
    buf[:, :256] = logits
    L = torch.from_numpy(buf).to(dev)
    g = None if gate is None else torch.from_numpy(np.ascontiguousarray(gate, np.float32)).to(dev)
    ids = torch.full((T, 8), -7, dtype=torch.int32, device=dev)
    w = torch.full((T, 8), -7.0, dtype=torch.float32, device=dev)
    sg = None if gate is None else torch.empty(T, dtype=torch.float32, device=dev)
    moe.moe_clear_status(ws)
    moe.moe_select_top8(L, T, ld, 256, g, ids, w, sg, ws, ws.numel())
    status = moe.moe_read_status(ws)
    return ids.cpu().numpy(), w.cpu().numpy(), (None if sg is None else sg.cpu().numpy()), status


def check(env, logits, gate=None, ld=256):
    ids, w, sg, status = run_select(env, logits, gate, ld)
    rid, rw, rsg, bad = oracle.select_topk(logits, gate, K=8)
    assert np.array_equal(ids, rid), np.argwhere(ids != rid)[:5]
    assert np.abs(w - rw).max() <= WEIGHT_ABS
    if gate is not None:
        assert np.abs(sg - rsg).max() <= WEIGHT_ABS
    assert status == (moe_nonfinite(env) if bad else 0)
    return ids, w


def moe_nonfinite(env):
    return env[0].DEV_NONFINITE


@pytest.mark.parametrize("T", W.SELECTOR_T)
def test_selector_config(env, T):
    logits = W.make_selector_logits(T)
    gate = W.normal(T, W.stream_key(T, "misc")).astype(np.float32) * 2
    check(env, logits, gate)


def test_selector_T1_both_kinds(env):
    rows = W.make_selector_logits(2)
    check(env, rows[0:1])
    check(env, rows[1:2])


def test_selector_sweep_1_to_64_and_ragged(env):
    for T in range(1, 65):
        logits = W.make_selector_logits(T, seed=1000 + T)
        check(env, logits)
    for T in (127, 129, 1000, 4097):
        check(env, W.make_selector_logits(T, seed=T))


def test_selector_strided_rows(env):
    check(env, W.make_selector_logits(33, seed=5), ld=260)


def test_selector_golden_tie_rows(env):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "select_ties.txt")
    rows, wants = [], []
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            _, vals, want = [p.strip() for p in line.split("|")]
            row = np.full(256, -1e30, np.float32)
            row[:16] = [float(v) for v in vals.split()]
            rows.append(row)
            wants.append([int(v) for v in want.split()])
    ids, _ = check(env, np.stack(rows))
    assert ids.tolist() == wants


def test_selector_ties_signed_zeros_and_all_equal(env):
    T = 8
    logits = np.zeros((T, 256), np.float32)
    signs = W.int_uniform(T * 256, W.stream_key(9, "misc"), 0, 1).reshape(T, 256)
    logits[signs == 1] = -0.0
    logits[3] = 2.5
    logits[4] = -1.0
    logits[5, 250:] = 1.0   # six high ids, then ties at 0 broken by low ids
    logits[6, ::2] = 3.0    # 128 tied leaders
    logits[7, 8] = np.float32(1e-45)  # smallest subnormal beats +-0
    ids, _ = check(env, logits)
    assert ids[0].tolist() == list(range(8))
    assert ids[5].tolist() == [250, 251, 252, 253, 254, 255, 0, 1]
    assert ids[6].tolist() == [0, 2, 4, 6, 8, 10, 12, 14]
    assert ids[7].tolist() == [8, 0, 1, 2, 3, 4, 5, 6]


def test_selector_nonfinite_rows(env):
    logits = W.make_selector_logits(6, seed=3)
    logits[1, 100] = np.nan
    logits[4, 0] = np.inf
    ids, w, _, status = run_select(env, logits)
    assert status & env[0].DEV_NONFINITE
    assert (ids[[1, 4]] == -1).all() and (w[[1, 4]] == 0).all()
    rid, rw, _, bad = oracle.select_topk(logits, K=8)
    assert bad == 2
    assert np.array_equal(ids, rid)
