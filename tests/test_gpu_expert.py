"""A4/A5/A6 expert outputs (moe_expert_swiglu_w8) and A7 combine on the GPU
against the oracle's per-slot outputs."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import assert_f32_close, assert_out_close, gpu_env, ncpu, to_dev, workload, workload_dev

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
    for t in range(T):
        for j in range(9):
            assert_f32_close(y[t, j], ref["y"][t, j], "t=%d slot=%d" % (t, j))


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
