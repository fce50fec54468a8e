"""The entry point that allocates nothing (moe_block_forward_noalloc).

It serves callers that cannot call cudaMalloc where they run the block (a
plugin in a runtime that owns all device memory, a process with a fixed
device-memory budget, a latency-critical path that cannot take cudaMalloc's
implicit synchronisation): its scratch is a fixed 4 MiB device array inside
the library.  This file is named to be collected last, and each check runs
in a fresh process as well as after the other tests.
"""
import ctypes

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
