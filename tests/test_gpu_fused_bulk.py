"""The fused decode kernel's bulk-copy path: the producer fetches each
gate|up unit with tensor-map copies, and with four bulk copies (two 16 KB row
blocks, two blocks of group scales) when the maps cannot be encoded.  A
test-only build (MOE_FUSED_BULK_COPIES = 1, never the product library)
forces that path; it must pass the same block parity checks as the product
library, on the fused kernel's item-mode and row-owner down phases and both
selection modes, in its own interpreter."""
import json
import os
import subprocess
import sys

import pytest

from util import gpu_env

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

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
res = {}
for name, T in (("pr1", 4), ("pr1", 32), ("decode", 1), ("decode", 20), ("decode", 40)):
    dims, _ = workload(name)
    x, _ = W.make_x(dims, T, 700 + T)
    try:
        check_block(moe, dev, name, x, n_sample=16, seed=T)
        res["%s T=%d" % (name, T)] = "pass"
    except AssertionError as e:
        res["%s T=%d" % (name, T)] = "fail: " + (str(e).splitlines() or ["assertion"])[0][:120]
torch.cuda.synchronize()
assert moe.lib()._name == lib_path
print("RESULT " + json.dumps(res))
"""


def test_bulk_copy_path_passes_block_parity():
    gpu_env()
    from sparse_moe_decode_gb300 import build
    lib_path = build.build_variant("fusedbulk", {"MOE_FUSED_BULK_COPIES": 1})
    r = subprocess.run([sys.executable, "-c", _RUN, ROOT, lib_path], capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    res = json.loads(line[7:])
    print(res)
    assert all(v == "pass" for v in res.values()), res
