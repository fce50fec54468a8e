"""A4/A5/A6 expert outputs (moe_expert_swiglu_w8) and A7 combine on the GPU
against the oracle's per-slot outputs."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import (assert_out_close, assert_slots_close, gpu_env, ncpu, to_dev, workload,
                  workload_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return gpu_env()


def run_experts(moe, dev, name, T, seed):
    import torch
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    x, _ = W.make_x(dims, T, seed=seed)
    logits, gate = oracle.router_logits(x, w["w_router"], w["w_gate"])
    ids, wts, sg, _ = oracle.select_topk(logits, gate, K=8)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    wsb = moe.moe_workspace_bytes(d, T)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    y = torch.full((T, 9, dims.H), np.nan, dtype=torch.float32, device=dev)
    moe.moe_expert_swiglu_w8(d, moe.weights_struct(wd), to_dev(x, dev), T, to_dev(ids, dev), y,
                             ws, wsb)
    assert moe.moe_read_status(ws) == 0
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=logits, route_gate=gate,
                               nthreads=ncpu(), want=("out", "y"))
    return dims, x, ids, wts, sg, y.cpu().numpy(), ref


@pytest.mark.parametrize("name,T,seed", [("pr1", 4, 0), ("pr1", 21, 3), ("decode", 1, 1),
                                         ("decode", 32, 2)])
def test_expert_slots_match_oracle(env, name, T, seed):
    moe, dev = env
    dims, x, ids, wts, sg, y, ref = run_experts(moe, dev, name, T, seed)
    assert_slots_close(y, ref["y"], ids, "%s T=%d" % (name, T))


@pytest.mark.parametrize("name,T,seed", [("decode", 65, 65), ("pr1", 200, 4),
                                         ("prefill", 2048, 3)])
def test_expert_slots_tensor_core_route(env, name, T, seed):
    """From T = 65 the call runs the tcgen05 grouped GEMMs (its down kernel
    storing each slot's output): every slot of every token against the
    oracle, and the rows of slots with no expert left as they were."""
    moe, dev = env
    dims, x, ids, wts, sg, y, ref = run_experts(moe, dev, name, T, seed)
    assert_slots_close(y, ref["y"], ids, "%s T=%d" % (name, T))
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    assert moe.moe_block_kernel_name(d, T, 0) == "router_tc"  # the same T takes that route


def test_expert_slots_tensor_core_route_bad_ids(env):
    """Slots naming no expert (-1) keep their rows; an id >= E is skipped and
    flagged."""
    import torch
    moe, dev = env
    dims, w = workload("pr1")
    wd = workload_dev("pr1", dev)
    T = 80
    x, _ = W.make_x(dims, T, 21)
    logits, gate = oracle.router_logits(x, w["w_router"], w["w_gate"])
    ids, _, _, _ = oracle.select_topk(logits, gate, K=8)
    ids = ids.copy()
    ids[3, 5] = -1
    ids[7, :] = -1
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    wsb = moe.moe_workspace_bytes(d, T)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    y = torch.full((T, 9, dims.H), np.nan, dtype=torch.float32, device=dev)
    moe.moe_expert_swiglu_w8(d, moe.weights_struct(wd), to_dev(x, dev), T, to_dev(ids, dev), y,
                             ws, wsb)
    assert moe.moe_read_status(ws) == 0
    yh = y.cpu().numpy()
    assert np.isnan(yh[3, 5]).all() and np.isnan(yh[7, :8]).all()
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=logits, route_gate=gate,
                               nthreads=ncpu(), want=("y",))
    # a slot's output depends only on its token and expert: the oracle's
    # slots (routed on the unmodified ids) serve every slot that kept its id
    assert_slots_close(yh, ref["y"], ids, "pr1 T=80 with -1 ids")
    ids[9, 2] = 300
    y.fill_(np.nan)
    moe.moe_expert_swiglu_w8(d, moe.weights_struct(wd), to_dev(x, dev), T, to_dev(ids, dev), y,
                             ws, wsb)
    assert moe.moe_read_status(ws) & moe.DEV_BAD_EXPERT
    assert np.isnan(y[9, 2].cpu().numpy()).all()


@pytest.mark.parametrize("T", [20, 80])
def test_expert_slots_repeated_expert_in_a_token(env, T):
    """Caller ids that name one expert in two slots of a token (both routes):
    the repeated slot holds that expert's output for the token, which is the
    oracle's output for the slot it was copied from."""
    import torch
    moe, dev = env
    dims, w = workload("pr1")
    wd = workload_dev("pr1", dev)
    x, _ = W.make_x(dims, T, 30 + T)
    logits, gate = oracle.router_logits(x, w["w_router"], w["w_gate"])
    ids, _, _, _ = oracle.select_topk(logits, gate, K=8)
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=logits, route_gate=gate,
                               nthreads=ncpu(), want=("y",))
    dup = ids.copy()
    src = np.zeros((T, 8), np.int32) + np.arange(8)
    for t in range(0, T, 3):
        dup[t, 7] = dup[t, 2]
        src[t, 7] = 2
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    wsb = moe.moe_workspace_bytes(d, T)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    y = torch.full((T, 9, dims.H), np.nan, dtype=torch.float32, device=dev)
    moe.moe_expert_swiglu_w8(d, moe.weights_struct(wd), to_dev(x, dev), T, to_dev(dup, dev), y,
                             ws, wsb)
    assert moe.moe_read_status(ws) == 0
    want = np.concatenate([np.take_along_axis(ref["y"][:, :8], src[..., None], axis=1),
                           ref["y"][:, 8:]], axis=1)
    assert_slots_close(y.cpu().numpy(), want, dup, "pr1 T=%d repeated experts" % T)


def test_combine_matches_oracle(env):
    import torch
    moe, dev = env
    T, H = 16, 512
    y = W.normal(T * 9 * H, W.stream_key(1, "misc")).reshape(T, 9, H).astype(np.float32) * 50
    logits = W.make_selector_logits(T, seed=2)
    _, wts, _, _ = oracle.select_topk(logits, K=8)
    sg = W.uniform(T, W.stream_key(2, "misc"))
    wts32, sg32 = wts.astype(np.float32), sg.astype(np.float32)
    out = torch.empty((T, H), dtype=torch.int16, device=dev)
    d = moe.Dims.make(H, 128, 128)
    moe.moe_combine(d, T, to_dev(y, dev), to_dev(wts32, dev), to_dev(sg32, dev), out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    for t in range(T):
        _, ob = oracle.combine(y[t, :8].astype(np.float64), wts32[t].astype(np.float64),
                               y[t, 8].astype(np.float64), float(sg32[t]))
        assert_out_close(got[t], ob, "t=%d" % t)
    # a zero weight skips its slot even when the slot holds NaN
    y[3, 2] = np.nan
    wts32[3, 2] = 0.0
    moe.moe_combine(d, T, to_dev(y, dev), to_dev(wts32, dev), to_dev(sg32, dev), out)
    torch.cuda.synchronize()
    assert np.isfinite(W.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16)[3])).all()
