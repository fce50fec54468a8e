"""The decode-size routes agree: the fused persistent kernel (default for
T <= 64) and the separate weight-streaming kernels (forced with
MOE_DECODE_ROUTE=gemv in a child process) both meet the block tolerance
against the oracle on the same inputs, and route identically."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads as W
from util import assert_out_close, bits, gpu_env, ncpu, to_dev, workload, workload_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np, torch
sys.path.insert(0, %(root)r); sys.path.insert(0, %(tests)r)
import sparse_moe_decode_gb300 as moe, workloads as W
from util import to_dev, bits, workload, workload_dev
dev = torch.device('cuda:0')
dims, w = workload(%(name)r); wd = workload_dev(%(name)r, dev)
x, _ = W.make_x(dims, %(T)d, %(seed)d)
blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=%(T)d, device=dev)
d = blk.dims
assert moe.moe_block_kernel_name(d, %(T)d, 0) == 'router_gemv'
out = torch.empty((%(T)d, dims.H), dtype=torch.int16, device=dev)
ids = torch.empty((%(T)d, 8), dtype=torch.int32, device=dev)
blk.forward(to_dev(x, dev), out=out, ids=ids); torch.cuda.synchronize()
assert blk.status() == 0
np.savez(%(path)r, out=bits(out), ids=ids.cpu().numpy())
"""


@pytest.mark.parametrize("name,T,seed", [("pr1", 4, 0), ("decode", 1, 1), ("decode", 32, 9)])
def test_fused_and_gemv_routes_agree(name, T, seed, tmp_path):
    import torch
    moe, dev = gpu_env()
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    x, _ = W.make_x(dims, T, seed)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    assert moe.moe_block_kernel_name(d, T, 0) == "decode_fused"
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T, device=dev)
    out = torch.empty((T, dims.H), dtype=torch.int16, device=dev)
    ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
    lg = torch.empty((T, 256), dtype=torch.float32, device=dev)
    gl = torch.empty((T,), dtype=torch.float32, device=dev)
    blk.forward(to_dev(x, dev), out=out, ids=ids, logits=lg, gate_logit=gl)
    torch.cuda.synchronize()
    assert blk.status() == 0
    path = str(tmp_path / "gemv.npz")
    env = dict(os.environ, MOE_DECODE_ROUTE="gemv")
    code = CHILD % {"root": ROOT, "tests": os.path.join(ROOT, "tests"), "name": name, "T": T,
                    "seed": seed, "path": path}
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    g = np.load(path)
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=lg.cpu().numpy(),
                               route_gate=gl.cpu().numpy(), nthreads=ncpu())
    fused = bits(out)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(g["ids"], ref["ids"])
    assert_out_close(fused, ref["out"], "fused")
    assert_out_close(g["out"], ref["out"], "gemv")
