"""moe_block_forward_residual: the block, the residual add in its combine
epilogue and the next layer's RMS-normed input (lucebox commit list, the
fused residual add + RMS norm + weight multiply), against the oracle's
oracle_add_rmsnorm fed with the oracle's unrounded block output.

Bars: resid_out and x_next meet the block's two bars against the oracle
(their error is the block's error); x_next is also within one bf16 ulp of
the oracle's norm of the GPU's own resid_out (the norm kernel alone: fp32
against fp64, so a rounding may flip, and nothing more)."""
import numpy as np
import pytest

import oracle
import workloads as W
from util import assert_out_close, bf16_f64, bits, gpu_env, ncpu, to_dev, workload, workload_dev

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module")
def env():
    return gpu_env()


def residual_inputs(dims, T, seed):
    resid = W.bf16_normal((T, dims.H), W.stream_key(seed, "misc", 7), 4.0)
    gamma = W.bf16_normal((dims.H,), W.stream_key(seed, "misc", 8), 1.0)
    return resid, gamma


def run(moe, dev, dims, wd, x, resid, gamma, in_place=False):
    import torch
    T = x.shape[0]
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    wsb = moe.moe_workspace_bytes(d, T)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    r_in = to_dev(resid, dev)
    r_out = r_in if in_place else torch.full_like(r_in, -1)
    x_next = torch.full((T, dims.H), -1, dtype=torch.int16, device=dev)
    moe.moe_block_forward_residual(d, moe.weights_struct(wd), to_dev(x, dev), T, r_in,
                                   to_dev(gamma, dev), EPS, r_out, x_next, ws, wsb)
    assert moe.moe_read_status(ws) == 0
    # the routing the GPU took, for the oracle
    lg = torch.empty((T, 256), dtype=torch.float32, device=dev)
    gl = torch.empty((T,), dtype=torch.float32, device=dev)
    out = torch.empty((T, dims.H), dtype=torch.int16, device=dev)
    moe.moe_block_forward(d, moe.weights_struct(wd), to_dev(x, dev), T, out, None, None, lg, gl,
                          ws, wsb)
    torch.cuda.synchronize()
    return bits(r_out), bits(x_next), lg.cpu().numpy(), gl.cpu().numpy()


def ulp_distance(a, b):
    def line(v):
        v = v.astype(np.int32)
        return np.where(v & 0x8000, 0x8000 - v, v)
    return np.abs(line(a) - line(b))


def check(moe, dev, dims, w, wd, x, seed, what, tokens=None):
    resid, gamma = residual_inputs(dims, x.shape[0], seed)
    r_out, x_next, lg, gl = run(moe, dev, dims, wd, x, resid, gamma)
    ref = oracle.block_forward(dims.as_dict(), w, x, tokens=tokens, route_logits=lg,
                               route_gate=gl, nthreads=ncpu(), want=("out_f64",))
    rows = np.arange(x.shape[0]) if tokens is None else tokens
    r_ref, x_ref = oracle.add_rmsnorm(resid[rows], ref["out_f64"][rows], gamma, EPS)
    assert_out_close(r_out[rows], r_ref, what + " resid_out")
    assert_out_close(x_next[rows], x_ref, what + " x_next")
    # the norm kernel alone: the oracle's norm of the GPU's own residual sum
    _, x_own = oracle.add_rmsnorm(r_out[rows], np.zeros((len(rows), dims.H)), gamma, EPS)
    u = ulp_distance(x_next[rows], x_own)
    assert u.max() <= 1, "%s: x_next %d ulp from the norm of its own resid_out" % (what, u.max())
    assert (u > 0).mean() < 1e-2
    return r_out, x_next, resid, gamma


@pytest.mark.parametrize("name,T,seed", [("pr1", 4, 1), ("decode", 1, 2), ("verify", 32, 3),
                                         ("decode", 100, 4)])
def test_residual_matches_oracle(env, name, T, seed):
    moe, dev = env
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    if name == "verify":
        x = W.workload_inputs("verify")[2]
    else:
        x, _ = W.make_x(dims, T, 60 + seed)
    check(moe, dev, dims, w, wd, x, seed, "%s T=%d" % (name, T))


def test_residual_weight_streaming_route(env):
    """H = 640 (not a multiple of 512) runs the separate weight-streaming
    kernels at decode sizes; their combine adds the residual too."""
    import torch
    moe, dev = env
    dims = W.Dims(H=640, I=384, Is=384)
    w = W.make_weights(dims, 21)
    wd = {k: to_dev(v, dev) for k, v in w.items()}
    x, _ = W.make_x(dims, 5, 22)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    assert moe.moe_block_kernel_name(d, 5, 0) == "router_gemv"
    check(moe, dev, dims, w, wd, x, 5, "H640 T=5")


def test_residual_prefill_sampled(env):
    moe, dev = env
    dims, w, x, _ = W.workload_inputs("prefill")
    toks = np.sort(W.permutation(x.shape[0], W.stream_key(9, "misc"))[:40]).astype(np.int32)
    check(moe, dev, dims, w, workload_dev("prefill", dev), x, 6, "prefill T=2048",
          tokens=toks)


@pytest.mark.parametrize("name,T", [("verify", 32), ("decode", 100)])
def test_residual_in_place_and_batch_width(env, name, T):
    """resid_out written over resid_in gives the same result: the same bits
    on the fused route (deterministic), and within the block's bars on the
    tcgen05 route, whose fp32 atomics may order a sum differently from run
    to run; on the fused route a token's x_next does not depend on the
    batch it rides in."""
    moe, dev = env
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    x, _ = W.make_x(dims, T, 80 + T)
    resid, gamma = residual_inputs(dims, T, 11)
    r1, x1, _, _ = run(moe, dev, dims, wd, x, resid, gamma)
    r2, x2, _, _ = run(moe, dev, dims, wd, x, resid, gamma, in_place=True)
    if T > 64:
        assert_out_close(r2, r1, "in place, tcgen05 route")
        assert_out_close(x2, x1, "in place, tcgen05 route")
        return
    assert np.array_equal(r1, r2)
    assert np.array_equal(x1, x2)
    if T <= 64:
        for t in (0, T - 1):
            r3, x3, _, _ = run(moe, dev, dims, wd, x[t:t + 1], resid[t:t + 1], gamma)
            assert np.array_equal(r3[0], r1[t]) and np.array_equal(x3[0], x1[t])
