"""The parity tests can fail: four test-only builds of the library, each
compiled with MOE_SABOTAGE = n (never the product library), plant one known
mistake in the GPU path, and the block parity check must reject every one of
them on every route it touches, while the product library passes the same
check in the same harness.

  1  the 8th selected id moves to the next expert not already chosen
  2  the softmax weights of ranks 7 and 8 trade places, their ids do not
  3  the shared expert's sigmoid gate is dropped
  4  gate|up weights are dequantised with the next group's scale

Arms 1 and 2 are the pages' own two sabotage arms for the bit-identity gate
(ninfer-windows PR #8, the test paragraph); 3 and 4 cover the shared gate and
the group-wise scales.  Each build runs in its own interpreter, on PR1
dimensions at T = 4 (fused kernel, one-warp lists), T = 32 (fused kernel,
selection shared by the grid) and T = 100 (tcgen05 route).
"""
import json
import os
import subprocess
import sys

import pytest

from util import gpu_env

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = (4, 32, 100)

_RUN = r"""
import json, sys
root, lib_path = sys.argv[1], sys.argv[2]
sys.path[:0] = [root, root + "/tests"]
import torch
import sparse_moe_decode_gb300 as moe
moe.LIB_PATH = lib_path
import workloads as W
from test_gpu_block import check_block
from util import workload
dev = torch.device("cuda:0")
dims, _ = workload("pr1")
res = {}
for T in (%s):
    x, _ = W.make_x(dims, T, 500 + T)
    try:
        check_block(moe, dev, "pr1", x)
        res[T] = "pass"
    except AssertionError as e:
        res[T] = "fail: " + (str(e).splitlines() or ["assertion"])[0][:120]
torch.cuda.synchronize()
assert moe.lib()._name == lib_path
print("RESULT " + json.dumps(res))
""" % ", ".join(str(t) for t in CASES)


def _run(lib_path):
    r = subprocess.run([sys.executable, "-c", _RUN, ROOT, lib_path], capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    return {int(k): v for k, v in json.loads(line[7:]).items()}


def test_product_library_passes_the_harness():
    moe, _ = gpu_env()
    res = _run(moe.LIB_PATH)
    assert all(v == "pass" for v in res.values()), res


@pytest.mark.parametrize("arm", [1, 2, 3, 4])
def test_sabotage_arm_is_caught(arm):
    gpu_env()
    from sparse_moe_decode_gb300 import build
    lib_path = build.build_variant("sabotage%d" % arm, {"MOE_SABOTAGE": arm})
    res = _run(lib_path)
    caught = {T: v for T, v in res.items() if v.startswith("fail")}
    print("arm %d:" % arm, res)
    assert set(caught) == set(CASES), "arm %d not caught at %s" % (
        arm, sorted(set(CASES) - set(caught)))
