"""The C-ABI library loads and exports what include/moe_gb300.h declares;
host-side argument checks reject bad calls before any device work (no GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__ as g
    g.build()
    import sparse_moe_decode_gb300 as m
    return m


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_router_logits", "moe_select_top8", "moe_expert_swiglu_w8", "moe_combine",
              "moe_block_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(moe):
    L = moe.lib()
    for n in declared_functions():
        assert hasattr(L, n), n
    assert set(declared_functions()) == set(moe.EXPORTS)
    assert L.moe_abi_version() == 1


def test_library_is_built_for_sm_103a(moe):
    from sparse_moe_decode_gb300 import build
    assert "arch=compute_103a,code=sm_103a" in build.ARCH
    assert os.path.exists(moe.LIB_PATH)


def test_workspace_bytes_and_unsupported_dims(moe):
    d = moe.Dims.make(2048, 512, 512)
    small, big = moe.moe_workspace_bytes(d, 1), moe.moe_workspace_bytes(d, 2048)
    assert 0 < small < big
    assert moe.moe_workspace_bytes(d, 65537) == 0
    for bad in (moe.Dims.make(2048, 512, 512, num_experts=128),
                moe.Dims.make(2048, 512, 512, top_k=4),
                moe.Dims.make(2000, 512, 512),
                moe.Dims.make(2048, 500, 512),
                moe.Dims.make(2048, 512, 100),
                moe.Dims.make(2048, 512, 512, group=64)):
        assert moe.moe_workspace_bytes(bad, 4) == 0


def test_host_checks_reject_before_touching_the_device(moe):
    L = moe.lib()
    d = moe.Dims.make(512, 128, 128)
    w = moe.Weights()
    # null weights
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), 4096, 4, 4096, None, None,
                             None, None, 256, 1 << 30, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    fake = 1 << 20  # aligned fake addresses are never dereferenced on these paths
    w = moe.Weights(*([fake] * 10))
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), fake, 4, fake, None, None, None,
                             None, fake, 16, None)
    assert st == moe.MOE_ERR_WORKSPACE
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), fake, -1, fake, None, None, None,
                             None, fake, 1 << 30, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), fake, 70000, fake, None, None,
                             None, None, fake, 1 << 40, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), fake + 8, 4, fake, None, None,
                             None, None, fake, 1 << 30, None)
    assert st == moe.MOE_ERR_INVALID_ARG  # misaligned x
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), fake, 4, fake, None, None, None,
                             None, fake + 16, 1 << 30, None)
    assert st == moe.MOE_ERR_INVALID_ARG  # workspace not 256-aligned
    # T == 0 is a no-op
    st = L.moe_block_forward(ctypes.byref(d), ctypes.byref(w), None, 0, None, None, None, None,
                             None, fake, 1 << 30, None)
    assert st == moe.MOE_OK
    # selector: E must be 256, ld >= E
    assert L.moe_select_top8(fake, 4, 256, 128, None, fake, fake, None, fake, 256,
                             None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_select_top8(fake, 4, 100, 256, None, fake, fake, None, fake, 256,
                             None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_select_top8(fake, 4, 256, 256, None, fake, fake, None, fake, 16,
                             None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_combine(ctypes.byref(d), 4, None, fake, None, fake,
                         None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_status_string(moe.MOE_ERR_WORKSPACE) == b"workspace too small"


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "moe_oracle" not in src, fn


def test_topk_host_checks(moe):
    L = moe.lib()
    fake = 1 << 20  # aligned fake addresses are never dereferenced on these paths
    ws = moe.moe_topk_workspace_bytes(8, 151936)
    assert ws == 256 + ((8 * 149 * 16 * 8 + 255) // 256) * 256  # a run per 1024 columns
    assert moe.moe_topk_workspace_bytes(8, (1 << 24) + 1) == 0
    assert moe.moe_topk_workspace_bytes(-1, 100) == 0

    def cand(T=8, ld=151936, N=151936, k=16, ws_bytes=ws, logits=fake):
        return L.moe_topk_candidates(logits, T, ld, N, k, fake, fake, fake, ws_bytes, None)

    assert cand(T=0) == moe.MOE_OK
    assert cand(k=0) == moe.MOE_ERR_INVALID_ARG
    assert cand(k=17) == moe.MOE_ERR_UNSUPPORTED
    assert cand(N=10, ld=12, k=11) == moe.MOE_ERR_INVALID_ARG
    assert cand(ld=151932) == moe.MOE_ERR_INVALID_ARG
    assert cand(ld=151937) == moe.MOE_ERR_INVALID_ARG  # ld not a multiple of 4
    assert cand(logits=fake + 4) == moe.MOE_ERR_INVALID_ARG
    assert cand(ws_bytes=ws - 1) == moe.MOE_ERR_WORKSPACE
    assert cand(N=(1 << 24) + 4, ld=(1 << 24) + 4) == moe.MOE_ERR_UNSUPPORTED

    def merge(T=8, n_lists=2, k=16, ws_bytes=256):
        return L.moe_topk_merge(fake, fake, T, n_lists, k, fake, fake, fake, ws_bytes, None)

    assert merge(T=0) == moe.MOE_OK
    assert merge(n_lists=0) == moe.MOE_ERR_INVALID_ARG
    assert merge(k=17) == moe.MOE_ERR_UNSUPPORTED
    assert merge(n_lists=65537) == moe.MOE_ERR_UNSUPPORTED
    assert merge(ws_bytes=255) == moe.MOE_ERR_WORKSPACE


def test_noalloc_limit_and_host_checks(moe):
    """The no-allocation entry's 4 MiB array admits the workspace of T <= 38
    at H = 2048, I = Is = 512 (and T <= 247 at H = 512, I = Is = 128), and
    every rejection happens on the host before any device call."""
    L = moe.lib()
    lim = 4 << 20
    d = moe.Dims.make(2048, 512, 512)
    assert moe.moe_workspace_bytes(d, 38) <= lim < moe.moe_workspace_bytes(d, 39)
    d1 = moe.Dims.make(512, 128, 128)
    assert moe.moe_workspace_bytes(d1, 247) <= lim < moe.moe_workspace_bytes(d1, 248)
    fake = 1 << 20
    w = moe.Weights(*([fake] * 10))
    assert L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(w), fake, 39, fake,
                                       None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(w), None, 4, fake,
                                       None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(w), fake + 2, 4, fake,
                                       None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_block_forward_noalloc(ctypes.byref(d), ctypes.byref(moe.Weights()), fake, 4,
                                       fake, None) == moe.MOE_ERR_INVALID_ARG
    bad = moe.Dims.make(2048, 512, 512, top_k=4)
    assert L.moe_block_forward_noalloc(ctypes.byref(bad), ctypes.byref(w), fake, 4, fake,
                                       None) == moe.MOE_ERR_UNSUPPORTED


def test_residual_entry_host_checks(moe):
    """moe_block_forward_residual rejects bad eps and overlapping buffers on
    the host, before anything is enqueued."""
    L = moe.lib()
    d = moe.Dims.make(512, 128, 128)
    fake = 1 << 20
    w = moe.Weights(*([fake] * 10))
    T, row = 4, 512 * 2
    ws = fake * 64
    wsb = moe.moe_workspace_bytes(d, T)

    def call(r_in, r_out, x_next, eps=1e-6, x=fake):
        return L.moe_block_forward_residual(ctypes.byref(d), ctypes.byref(w), x, T, r_in, fake,
                                            eps, r_out, x_next, ws, wsb, None)

    a, b, c = fake * 2, fake * 4, fake * 6
    assert call(a, b, c, eps=-1.0) == moe.MOE_ERR_INVALID_ARG
    assert call(a, b, c, eps=float("nan")) == moe.MOE_ERR_INVALID_ARG
    assert call(a, b, b + row) == moe.MOE_ERR_INVALID_ARG       # x_next inside resid_out
    assert call(a, b, a) == moe.MOE_ERR_INVALID_ARG             # x_next over resid_in
    assert call(a, a + row, c) == moe.MOE_ERR_INVALID_ARG       # residuals partly overlap
    assert call(None, b, c) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_block_forward_residual(ctypes.byref(d), ctypes.byref(w), fake, T, a, fake,
                                        1e-6, b, c, ws, 16, None) == moe.MOE_ERR_WORKSPACE
