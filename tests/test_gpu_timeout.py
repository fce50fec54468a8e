"""Bounded waits on the GPU.  With a wait budget of 1 ns every pipeline wait
that does not succeed at once gives up: the kernels must set MOE_DEV_TIMEOUT
in the status word, let the work already in flight finish (copies landing,
MMAs completing before tensor memory is freed), return, and leave the CUDA
context usable.  Runs in a child process because the budget is read once per
process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import torch
import sparse_moe_decode_gb300 as moe
import workloads as W
from util import to_dev, workload, workload_dev
dev = torch.device("cuda:0")
res = []
for name, T in (("verify", 32), ("prefill", 256)):
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    x, _ = W.make_x(dims, T, 5)
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T, device=dev)
    blk.forward(to_dev(x, dev))
    torch.cuda.synchronize()
    res.append(blk.status())
y = torch.ones(1 << 20, device=dev).sum().item()  # the context still computes
print("RESULT", res[0], res[1], int(y))
"""


def test_wait_budget_expiry_sets_timeout_and_keeps_context():
    import __graft_entry__ as g
    g.build()
    import sparse_moe_decode_gb300 as moe
    env = dict(os.environ, MOE_WAIT_BUDGET_NS="1")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT")][-1].split()
    st_verify, st_prefill, y = int(line[1]), int(line[2]), int(line[3])
    timeout_bit = moe.DEV_TIMEOUT
    assert st_verify & timeout_bit, st_verify
    assert st_prefill & timeout_bit, st_prefill
    assert y == 1 << 20
