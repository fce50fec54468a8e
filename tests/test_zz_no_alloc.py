"""The entry point that allocates nothing (moe_block_forward_noalloc).

It serves callers that cannot call cudaMalloc where they run the block (a
plugin in a runtime that owns all device memory, a process with a fixed
device-memory budget, a latency-critical path that cannot take cudaMalloc's
implicit synchronisation): its scratch is a fixed 4 MiB device array inside
the library.  This file is named to be collected last, so that its checks
run after the other tests in the same process; one more check starts a fresh
interpreter, whose first call looks up the array's address on a clean
context.
"""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

import workloads as W
from util import assert_out_close, bits, gpu_env, to_dev, workload, workload_dev

pytestmark = pytest.mark.gpu


def _existing(moe, dev, dims, wd, x):
    import torch
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=x.shape[0], device=dev)
    out = torch.empty((x.shape[0], dims.H), dtype=torch.int16, device=dev)
    blk.forward(to_dev(x, dev), out=out)
    torch.cuda.synchronize()
    return bits(out)


@pytest.mark.parametrize("name,T", [("pr1", 4), ("decode", 1), ("verify", 32)])
def test_noalloc_matches_existing_entry_on_two_calls(name, T):
    import torch
    moe, dev = gpu_env()
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    ws = moe.weights_struct(wd)
    L = moe.lib()
    for call, seed in enumerate((11, 12)):  # two calls in a row share the array
        x, _ = W.make_x(dims, T, seed)
        want = _existing(moe, dev, dims, wd, x)
        xd = to_dev(x, dev)
        out = torch.full((T, dims.H), -1, dtype=torch.int16, device=dev)
        st = L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(ws), xd.data_ptr(), T,
                                         out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == moe.MOE_OK, st
        torch.cuda.synchronize()
        got = bits(out)
        assert_out_close(got, want, "%s call %d" % (name, call))
        assert np.array_equal(got, want)  # same kernels, same order: same bits


def test_noalloc_rejects_sizes_beyond_its_array():
    moe, dev = gpu_env()
    dims, _ = workload("decode")
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    assert moe.moe_workspace_bytes(d, 2048) > (4 << 20)
    w = moe.Weights(*([1 << 20] * 10))
    L = moe.lib()
    st = L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(w), 1 << 20, 2048, 1 << 20,
                                     None)
    assert st == moe.MOE_ERR_WORKSPACE
    assert L.moe_block_forward_noalloc(None, ctypes.byref(w), 1 << 20, 4, 1 << 20,
                                       None) == moe.MOE_ERR_INVALID_ARG


@pytest.mark.parametrize("T,ok", [(38, True), (39, False)])
def test_noalloc_size_limit_at_decode_dims(T, ok):
    """At H = 2048, I = Is = 512 the 4 MiB array holds the workspace of up to
    38 tokens: T = 38 runs and matches the ordinary entry, T = 39 is refused
    before anything is enqueued."""
    import torch
    moe, dev = gpu_env()
    dims, w = workload("decode")
    wd = workload_dev("decode", dev)
    d = moe.Dims.make(dims.H, dims.I, dims.Is)
    ws = moe.weights_struct(wd)
    x, _ = W.make_x(dims, T, 40 + T)
    xd = to_dev(x, dev)
    out = torch.full((T, dims.H), -1, dtype=torch.int16, device=dev)
    st = moe.lib().moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(ws), xd.data_ptr(), T,
                                             out.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    if ok:
        assert st == moe.MOE_OK, st
        assert np.array_equal(bits(out), _existing(moe, dev, dims, wd, x))
    else:
        assert st == moe.MOE_ERR_WORKSPACE, st
        assert (bits(out) == 0xFFFF).all()  # nothing was written


_FRESH = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import oracle, workloads as W
import sparse_moe_decode_gb300 as moe
from util import assert_out_close, bits, to_dev, workload, workload_dev
dev = torch.device("cuda:0")
dims, w = workload("pr1")
wd = workload_dev("pr1", dev)
x, _ = W.make_x(dims, 4, 13)
d = moe.Dims.make(dims.H, dims.I, dims.Is)
ws = moe.weights_struct(wd)
out = torch.full((4, dims.H), -1, dtype=torch.int16, device=dev)
st = moe.lib().moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(ws),
                                         to_dev(x, dev).data_ptr(), 4, out.data_ptr(), None)
torch.cuda.synchronize()
assert st == moe.MOE_OK, st
ref = oracle.block_forward(dims.as_dict(), w, x, want=("out",))
assert_out_close(bits(out), ref["out"], "fresh process")
print("fresh ok")
"""


def test_noalloc_first_call_in_a_fresh_process():
    """A new interpreter's first call (the array's address looked up on a
    clean context) against the oracle."""
    gpu_env()  # builds the library
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "fresh ok" in r.stdout
