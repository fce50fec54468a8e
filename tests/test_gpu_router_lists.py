"""A1 router logits and A3 expert lists on the GPU against the oracle."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import LOGIT_REL, bf16_f64, gpu_env, to_dev, workload, workload_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return gpu_env()


@pytest.mark.parametrize("name,T", [("pr1", 4), ("pr1", 37), ("pr1", 200), ("decode", 1),
                                    ("decode", 32), ("decode", 129), ("decode", 2048)])
def test_router_logits(env, name, T):
    import torch
    moe, dev = env
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    x, _ = W.make_x(dims, T, seed=50 + T)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    logits = torch.empty((T, 256), dtype=torch.float32, device=dev)
    gate = torch.empty(T, dtype=torch.float32, device=dev)
    moe.moe_router_logits(d, moe.weights_struct(wd), to_dev(x, dev), T, logits, gate)
    torch.cuda.synchronize()
    rl, rg = oracle.router_logits(x, w["w_router"], w["w_gate"])
    xn = np.linalg.norm(bf16_f64(x), axis=1)
    wn = np.linalg.norm(bf16_f64(w["w_router"]), axis=1)
    tol = LOGIT_REL * xn[:, None] * wn[None, :]
    assert (np.abs(logits.cpu().numpy() - rl) <= tol).all()
    gn = np.linalg.norm(bf16_f64(w["w_gate"]))
    assert (np.abs(gate.cpu().numpy() - rg) <= LOGIT_REL * xn * gn).all()


def _ids(T, seed, hot=None):
    ids = np.stack([W.permutation(256, W.stream_key(seed, "misc", t))[:8] for t in range(T)])
    if hot is not None:
        ids[: T // 3, 0] = hot
        for t in range(T // 3):  # keep ids distinct within a token
            row = ids[t]
            dup = np.where(row[1:] == hot)[0]
            if len(dup):
                row[1 + dup[0]] = next(e for e in range(256) if e not in row)
    return ids.astype(np.int32)


@pytest.mark.parametrize("T", [1, 7, 32, 64, 2048, 2049, 4097])
def test_expert_lists_exact(env, T):
    import torch
    moe, dev = env
    ids = _ids(T, seed=T, hot=17 if T > 3 else None)
    if T > 5:
        ids[5] = -1  # a sentinel (non-finite) token is skipped
    ws = torch.zeros(1 << 14, dtype=torch.uint8, device=dev)
    counts = torch.full((256,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((257,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * 8,), -1, dtype=torch.int32, device=dev)
    moe.moe_build_expert_lists(to_dev(ids, dev), T, 256, counts, offsets, perm, ws, ws.numel())
    assert moe.moe_read_status(ws) == 0
    rc, ro, rp = oracle.expert_lists(ids, 256)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy()[: ro[256]], rp)


def test_expert_lists_flag_out_of_range_ids(env):
    import torch
    moe, dev = env
    ids = _ids(4, seed=1)
    ids[2, 3] = 300
    ws = torch.zeros(1 << 14, dtype=torch.uint8, device=dev)
    c = torch.empty(256, dtype=torch.int32, device=dev)
    o = torch.empty(257, dtype=torch.int32, device=dev)
    p = torch.empty(32, dtype=torch.int32, device=dev)
    moe.moe_build_expert_lists(to_dev(ids, dev), 4, 256, c, o, p, ws, ws.numel())
    assert moe.moe_read_status(ws) & moe.DEV_BAD_EXPERT
    assert int(o[256]) == 31


@pytest.mark.parametrize("T", [3, 256, 257, 3000])
def test_expert_lists_repeated_expert_in_a_token(env, T):
    """Caller ids may name one expert in several slots of a token: each such
    entry keeps its own place, in (t, j) order, as the oracle's sort gives.
    Ids drawn from 12 experts repeat often; T crosses the kernel's 256-token
    chunks."""
    import torch
    moe, dev = env
    r = W.uniform(T * 8, W.stream_key(T, "misc"))
    ids = np.minimum((r * 12).astype(np.int32), 11).reshape(T, 8)
    ids[0] = 4  # all eight slots of token 0 name expert 4
    ws = torch.zeros(1 << 14, dtype=torch.uint8, device=dev)
    counts = torch.full((256,), -1, dtype=torch.int32, device=dev)
    offsets = torch.full((257,), -1, dtype=torch.int32, device=dev)
    perm = torch.full((T * 8,), -1, dtype=torch.int32, device=dev)
    moe.moe_build_expert_lists(to_dev(ids, dev), T, 256, counts, offsets, perm, ws, ws.numel())
    assert moe.moe_read_status(ws) == 0
    rc, ro, rp = oracle.expert_lists(ids, 256)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(perm.cpu().numpy(), rp)
