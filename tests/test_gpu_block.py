"""moe_block_forward (A1..A7) on the GPU against the oracle.

Routing: the oracle selects on the GPU's own fp32 logits, so ids and order
must match bit for bit; against the oracle's own fp64-derived logits, a token
may differ only where the oracle's ranking has a near tie.  Output: the bf16
tolerance of the block.  The T sweep checks a seeded sample of tokens; the
prefill workload (T = 2048) is checked on every token.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from util import (assert_out_close, bf16_f64, bits, gpu_env, ncpu, near_tie, to_dev, workload,
                  workload_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    return gpu_env()


def forward(moe, dev, name, x, T_max=None):
    import torch
    dims, w = workload(name)
    wd = workload_dev(name, dev)
    T = x.shape[0]
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T_max or T, device=dev)
    o = {
        "out": torch.empty((T, dims.H), dtype=torch.int16, device=dev),
        "ids": torch.empty((T, 8), dtype=torch.int32, device=dev),
        "weights": torch.empty((T, 8), dtype=torch.float32, device=dev),
        "logits": torch.empty((T, 256), dtype=torch.float32, device=dev),
        "gate": torch.empty((T,), dtype=torch.float32, device=dev),
    }
    blk.forward(to_dev(x, dev), out=o["out"], ids=o["ids"], weights=o["weights"],
                logits=o["logits"], gate_logit=o["gate"])
    torch.cuda.synchronize()
    # status words 5..7: where a timed-out wait gave up (site, detail, CTA)
    assert blk.status() == 0, "wait gave up: site %d detail %d cta %d" % tuple(
        blk.workspace[20:32].view(torch.int32).tolist())
    res = {k: (bits(v) if k == "out" else v.cpu().numpy()) for k, v in o.items()}
    return dims, w, res, blk


def sample_tokens(T, n, seed):
    if T <= n:
        return None
    s = np.sort(W.permutation(T, W.stream_key(seed, "misc"))[: n - 2])
    return np.unique(np.concatenate([[0, T - 1], s])).astype(np.int32)


def check_block(moe, dev, name, x, n_sample=64, seed=0):
    dims, w, g, _ = forward(moe, dev, name, x)
    T = x.shape[0]
    toks = sample_tokens(T, n_sample, seed)
    rows = np.arange(T) if toks is None else toks
    ref = oracle.block_forward(dims.as_dict(), w, x, tokens=toks, route_logits=g["logits"],
                               route_gate=g["gate"], nthreads=ncpu(),
                               want=("out", "out_f64"))
    assert np.array_equal(g["ids"][rows], ref["ids"][rows])
    assert np.abs(g["weights"][rows] - ref["weights"][rows]).max() <= 1e-6
    assert_out_close(g["out"][rows], ref["out"][rows], name)
    # the GPU's logits against the oracle's fp64-derived fp32 logits
    xn = np.linalg.norm(W.bf16_bits_to_f32(x[rows]).astype(np.float64), axis=1)
    wn = np.linalg.norm(W.bf16_bits_to_f32(w["w_router"]).astype(np.float64), axis=1)
    assert (np.abs(g["logits"][rows] - ref["logits"][rows]) <=
            1e-5 * xn[:, None] * wn[None, :]).all()
    # routing on the oracle's own logits: any difference needs a near tie there
    own_ids, _, _, _ = oracle.select_topk(ref["logits"][rows], K=8)
    for i, t in enumerate(rows):
        if not np.array_equal(own_ids[i], g["ids"][t]):
            assert near_tie(ref["logits"][t]), "token %d routes differently without a tie" % t
    return dims, w, g


def test_block_pr1(env):
    moe, dev = env
    dims, w = workload("pr1")
    x, _ = W.make_x(dims, 4, 0)
    check_block(moe, dev, "pr1", x)


def test_block_pr1_ragged_T(env):
    moe, dev = env
    dims, w = workload("pr1")
    for T in (1, 3, 9, 12, 13, 33, 64, 65):
        x, _ = W.make_x(dims, T, 7 + T)
        check_block(moe, dev, "pr1", x)


def test_block_decode_T1(env):
    moe, dev = env
    dims, w, x, _ = W.workload_inputs("decode")
    check_block(moe, dev, "decode", x)


def test_block_verify_T32_skewed(env):
    moe, dev = env
    dims, w, x, info = W.workload_inputs("verify")
    _, _, g = check_block(moe, dev, "verify", x)
    assert (g["ids"][info["skewed"], 0] == info["e_star"]).all()
    assert len(np.unique(g["ids"])) > 100  # many distinct experts are active


@pytest.mark.parametrize("T", [2, 12, 13, 19, 20, 24, 25, 46, 47, 64, 65, 100, 768, 4097])
def test_block_decode_dims_T_sweep(env, T):
    moe, dev = env
    dims, _ = workload("decode")
    x, _ = W.make_x(dims, T, 100 + T)
    check_block(moe, dev, "decode", x, n_sample=48, seed=T)


def test_block_prefill_T2048_every_token(env):
    moe, dev = env
    dims, w, x, _ = W.workload_inputs("prefill")
    _, _, g = check_block(moe, dev, "prefill", x, n_sample=x.shape[0], seed=3)
    counts = np.bincount(g["ids"].ravel(), minlength=256)
    assert counts.min() > 0  # uniform routing touches every expert


def _bf16_ulp(b):
    """Spacing of bf16 values at each value (bits), from its magnitude up."""
    m = (b.astype(np.int32) & 0x7FFF)
    m = np.minimum(m, 0x7F7F)
    return (W.bf16_bits_to_f32((m + 1).astype(np.uint16)).astype(np.float64) -
            W.bf16_bits_to_f32(m.astype(np.uint16)).astype(np.float64))


def _order_bound(moe, dev, x, g):
    """Per output element, how far two fp32 summation orders of the block's
    nine terms (w_j y_j, then sg y_s) may land apart before the bf16
    rounding: each order is within 8 * 2^-24 * sum|terms| of the exact sum
    (terms from the oracle's per-slot outputs on the GPU's routing)."""
    dims, w = workload("prefill")
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=g["logits"],
                               route_gate=g["gate"], nthreads=ncpu(), want=("y",))
    terms = np.abs(ref["y"][:, :8] * ref["weights"][:, :, None]).sum(axis=1)
    terms += np.abs(ref["y"][:, 8] * ref["sgate"][:, None])
    return 16.0 * 2.0 ** -24 * terms


def _check_reordered(a_bits, b_bits, bound, what, capsys):
    """a and b differ at most by the summation-order bound plus one bf16 ulp
    of the larger of the two (its rounding); the counts are printed."""
    da = np.abs(bf16_f64(a_bits) - bf16_f64(b_bits))
    ulp = np.maximum(_bf16_ulp(a_bits), _bf16_ulp(b_bits))
    n_diff = int((da > 0).sum())
    in_ulps = da / ulp
    with capsys.disabled():
        print("\n  %s: %d of %d outputs differ, max %.0f ulp, max |diff| / bound %.3g" %
              (what, n_diff, da.size, in_ulps.max(), (np.maximum(da - ulp, 0) / bound).max()))
    assert (da <= bound + ulp).all(), what


def test_block_tensor_core_route_run_to_run(env, capsys):
    """The tcgen05 route adds the routed terms with fp32 atomics in the order
    they arrive, so runs of the prefill workload may differ by a reordered
    fp32 sum of nine terms (at most 16 * 2^-24 * sum|terms|) plus one bf16
    ulp of rounding; routing and logits do not differ at all."""
    moe, dev = env
    dims, w, x, _ = W.workload_inputs("prefill")
    runs = [forward(moe, dev, "prefill", x)[2] for _ in range(3)]
    bound = _order_bound(moe, dev, x, runs[0])
    for r in runs[1:]:
        assert np.array_equal(r["ids"], runs[0]["ids"])
        assert np.array_equal(r["logits"], runs[0]["logits"])
        _check_reordered(r["out"], runs[0]["out"], bound, "tcgen05 route run-to-run", capsys)


def test_block_batch_width_invariance_tensor_core_route(env, capsys):
    """Tokens 0..64 of the prefill workload as a T = 65 batch against the
    same tokens inside the T = 2048 batch (both on the tcgen05 route):
    identical routing and logits, outputs within the summation-order bound
    of the run-to-run test."""
    moe, dev = env
    dims, w, x, _ = W.workload_inputs("prefill")
    full = forward(moe, dev, "prefill", x)[2]
    part = forward(moe, dev, "prefill", x[:65])[2]
    assert np.array_equal(part["logits"], full["logits"][:65])
    assert np.array_equal(part["ids"], full["ids"][:65])
    assert np.array_equal(part["weights"], full["weights"][:65])
    g65 = {k: v[:65] for k, v in full.items()}
    bound = _order_bound(moe, dev, x[:65], g65)
    _check_reordered(part["out"], full["out"][:65], bound, "tcgen05 route T=65 vs T=2048",
                     capsys)


def test_block_batch_width_invariance_decode_route(env):
    """A token's output bits do not depend on the batch it rides in."""
    moe, dev = env
    dims, _ = workload("decode")
    x, _ = W.make_x(dims, 32, 77)
    _, _, full, _ = forward(moe, dev, "decode", x)
    for t in (0, 13, 31):
        _, _, one, _ = forward(moe, dev, "decode", x[t:t + 1])
        assert np.array_equal(one["out"][0], full["out"][t])
        assert np.array_equal(one["ids"][0], full["ids"][t])


def test_block_host_entry_matches_device_entry(env):
    import torch
    moe, dev = env
    dims, _ = workload("pr1")
    x, _ = W.make_x(dims, 6, 5)
    _, _, g, blk = forward(moe, dev, "pr1", x)
    out = np.zeros((6, dims.H), np.uint16)
    moe.moe_block_forward_host(blk.dims, blk.w, np.ascontiguousarray(x), 6, out, blk.workspace,
                               blk.ws_bytes)
    assert np.array_equal(out, g["out"])


def test_block_nonfinite_input_sets_status_and_keeps_shared(env):
    import torch
    moe, dev = env
    dims, w = workload("pr1")
    x, _ = W.make_x(dims, 3, 9)
    x[1, 5] = 0x7FC0  # NaN activation -> NaN logits for token 1
    wd = workload_dev("pr1", dev)
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=3, device=dev)
    ids = torch.empty((3, 8), dtype=torch.int32, device=dev)
    out = torch.empty((3, dims.H), dtype=torch.int16, device=dev)
    lg = torch.empty((3, 256), dtype=torch.float32, device=dev)
    gl = torch.empty((3,), dtype=torch.float32, device=dev)
    blk.forward(to_dev(x, dev), out=out, ids=ids, logits=lg, gate_logit=gl)
    assert blk.status() & moe.DEV_NONFINITE
    assert (ids[1].cpu().numpy() == -1).all() and (ids[0].cpu().numpy() >= 0).all()
    # the finite tokens are computed as usual, the other one gets only the
    # shared expert (whose gate is finite here only if its logit is)
    ref = oracle.block_forward(dims.as_dict(), w, x, tokens=np.array([0, 2], np.int32),
                               route_logits=lg.cpu().numpy(), route_gate=gl.cpu().numpy(),
                               nthreads=ncpu(), want=("out",))
    assert np.array_equal(ids.cpu().numpy()[[0, 2]], ref["ids"][[0, 2]])
    assert_out_close(bits(out)[[0, 2]], ref["out"][[0, 2]], "pr1")
    blk.clear_status()
    assert blk.status() == 0


@pytest.mark.parametrize("T", [200])
def test_block_prefill_route_rows_odd_multiple_of_128(env, T):
    """Prefill route with H, I, Is odd multiples of 128 (row chunks that cover
    half a warp), every token checked against the oracle."""
    import torch
    moe, dev = env
    dims = W.Dims(H=640, I=384, Is=384)
    w = W.make_weights(dims, 11)
    x, _ = W.make_x(dims, T, 12)
    wd = {k: to_dev(v, dev) for k, v in w.items()}
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T, device=dev)
    out = torch.empty((T, dims.H), dtype=torch.int16, device=dev)
    logits = torch.empty((T, 256), dtype=torch.float32, device=dev)
    gate = torch.empty((T,), dtype=torch.float32, device=dev)
    ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
    blk.forward(to_dev(x, dev), out=out, ids=ids, logits=logits, gate_logit=gate)
    torch.cuda.synchronize()
    assert blk.status() == 0
    ref = oracle.block_forward(dims.as_dict(), w, x, route_logits=logits.cpu().numpy(),
                               route_gate=gate.cpu().numpy(), nthreads=ncpu(),
                               want=("out", "out_f64"))
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    assert_out_close(bits(out), ref["out"], "H640 prefill route")


@pytest.mark.parametrize("T", [4, 32])
def test_block_fused_wide_h_takes_bf16_down(env, T):
    """Activations scaled by 2^8 scale h by 2^16, so some |h| >= 2^15 (the
    oracle's max |h| for these inputs is about 1.1e4): the fused kernel's
    down projection must then run on the bf16 h (its fp16 copies would
    overflow) and still match the oracle; unscaled, it takes the fp16
    copies.  The flag is the fifth word of the workspace."""
    import torch
    moe, dev = env
    dims, _ = workload("decode")
    x, _ = W.make_x(dims, T, 300 + T)
    for scale, wide in ((1.0, 0), (256.0, 1)):
        xs = W.f32_to_bf16_bits(W.bf16_bits_to_f32(x) * np.float32(scale))
        _, _, _, blk = forward(moe, dev, "decode", xs)
        assert int(blk.workspace[16:20].view(torch.int32).item()) == wide
        check_block(moe, dev, "decode", xs)


def _check_custom(moe, dev, dims, w, x, n_sample=None, seed=0, what=""):
    """Block forward at any dims against the oracle on the GPU's routing
    (every token, or a seeded sample of n_sample tokens)."""
    import torch
    T = x.shape[0]
    wd = {k: to_dev(v, dev) for k, v in w.items()}
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T, device=dev)
    out = torch.empty((T, dims.H), dtype=torch.int16, device=dev)
    logits = torch.empty((T, 256), dtype=torch.float32, device=dev)
    gate = torch.empty((T,), dtype=torch.float32, device=dev) if dims.Is else None
    ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
    blk.forward(to_dev(x, dev), out=out, ids=ids, logits=logits, gate_logit=gate)
    torch.cuda.synchronize()
    assert blk.status() == 0
    toks = None if n_sample is None else sample_tokens(T, n_sample, seed)
    rows = np.arange(T) if toks is None else toks
    ref = oracle.block_forward(dims.as_dict(), w, x, tokens=toks, route_logits=logits.cpu().numpy(),
                               route_gate=None if gate is None else gate.cpu().numpy(),
                               nthreads=ncpu(), want=("out",))
    assert np.array_equal(ids.cpu().numpy()[rows], ref["ids"][rows])
    assert_out_close(bits(out)[rows], ref["out"][rows], what)
    return bits(out), ids.cpu().numpy()


@pytest.mark.parametrize("T", [4, 33, 100])
def test_block_without_shared_expert(env, T):
    """shared_inter = 0: no gate row, no shared term, on every route."""
    moe, dev = env
    dims = W.Dims(H=512, I=128, Is=0)
    w = W.make_weights(dims, 31)
    x, _ = W.make_x(dims, T, 32 + T)
    _check_custom(moe, dev, dims, w, x, what="Is=0 T=%d" % T)


@pytest.mark.parametrize("T", [8, 40, 100])
def test_block_expert_and_shared_sizes_differ(env, T):
    """I = 256, Is = 128 (the fused kernel's stages hold the larger size)."""
    moe, dev = env
    dims = W.Dims(H=1024, I=256, Is=128)
    w = W.make_weights(dims, 41)
    x, _ = W.make_x(dims, T, 42 + T)
    _check_custom(moe, dev, dims, w, x, what="I=256 Is=128 T=%d" % T)


@pytest.mark.parametrize("T", [1, 12, 33, 100])
def test_block_all_zero_input(env, T):
    """x = 0: every logit is 0, so the total order picks experts 0..7 (the
    lower id wins a tie), the softmax weights are all 1/8, and the output is
    exactly zero on every route."""
    import torch
    moe, dev = env
    dims, _ = workload("pr1")
    wd = workload_dev("pr1", dev)
    x = np.zeros((T, dims.H), np.uint16)
    blk = moe.MoEBlock(dims.H, dims.I, dims.Is, wd, T_max=T, device=dev)
    out = torch.full((T, dims.H), -1, dtype=torch.int16, device=dev)
    ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
    wts = torch.empty((T, 8), dtype=torch.float32, device=dev)
    blk.forward(to_dev(x, dev), out=out, ids=ids, weights=wts)
    torch.cuda.synchronize()
    assert blk.status() == 0
    assert (ids.cpu().numpy() == np.arange(8)).all()
    assert (wts.cpu().numpy() == np.float32(0.125)).all()
    o = bits(out)
    assert ((o == 0) | (o == 0x8000)).all()  # +0 or -0


def test_block_largest_T(env):
    """T = 65536, the largest supported batch (tcgen05 route, PR1 dims), on a
    seeded sample of tokens including the first and the last."""
    moe, dev = env
    dims, w = workload("pr1")
    T = 65536
    x, _ = W.make_x(dims, T, 65)
    _check_custom(moe, dev, dims, w, x, n_sample=24, seed=5, what="T=65536")
