"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks one oracle step against something the oracle does not
compute: a brute-force sort, a hand-derived fixture, a closed form, an
invariant, or an independent library routine.  Each is chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a wrong scale group, a swapped gate/up half) fails it.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(vals):
    return W.f32_to_bf16_bits(np.asarray(vals, np.float32))


def f(b):
    return W.bf16_bits_to_f32(b).astype(np.float64)


# ------------------------------------------------------------ selection

def brute_sort_ids(row, K):
    """Full sort of (value, id) with Python's own sort: value desc, id asc."""
    keyed = sorted(range(len(row)), key=lambda e: (-float(row[e]) if row[e] != 0 else 0.0, e))
    return keyed[:K]


def argmax_passes(row, K):
    """K linear passes, each taking the best remaining candidate."""
    taken, out = set(), []
    for _ in range(K):
        best = None
        for e, v in enumerate(row):
            if e in taken:
                continue
            if best is None or v > row[best] or (v == row[best] and e < best):
                best = e
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("kind", ["normal", "ties"])
def test_select_matches_bruteforce_E256(kind):
    rows = []
    for t in range(24):
        k = W.stream_key(100 + t, "misc")
        if kind == "normal":
            rows.append(W.normal(256, k).astype(np.float32))
        else:
            rows.append(W.int_uniform(256, k, -4, 4).astype(np.float32))
    logits = np.stack(rows)
    ids, w, _, bad = oracle.select_topk(logits, K=8)
    assert bad == 0
    for t, row in enumerate(logits):
        assert list(ids[t]) == brute_sort_ids(list(row), 8)
        assert list(ids[t]) == argmax_passes(list(row), 8)


@pytest.mark.parametrize("K", [1, 2, 3, 4, 8])
def test_select_every_arrangement_of_a_tied_multiset(K):
    base = [3.0, 3.0, 1.0, 1.0, 0.0, 0.0, -1.0, 2.0]
    perms = np.array(sorted(set(itertools.permutations(base))), np.float32)
    assert len(perms) == 5040
    ids, _, _, _ = oracle.select_topk(perms, K=K)
    for t, row in enumerate(perms):
        assert list(ids[t]) == argmax_passes(list(row), K)


def test_select_E10_all_permutations_distinct_K3():
    vals = np.arange(10, dtype=np.float32)
    rows = np.array([p for i, p in enumerate(itertools.permutations(vals)) if i % 97 == 0],
                    np.float32)
    ids, _, _, _ = oracle.select_topk(rows, K=3)
    for t, row in enumerate(rows):
        assert list(ids[t]) == brute_sort_ids(list(row), 3)


def _golden_select():
    cases = []
    with open(os.path.join(GOLDEN, "select_ties.txt")) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            name, vals, want = [p.strip() for p in line.split("|")]
            cases.append((name, np.array([float(v) for v in vals.split()], np.float32),
                          [int(v) for v in want.split()]))
    return cases


@pytest.mark.parametrize("name,row,want", _golden_select(),
                         ids=[c[0] for c in _golden_select()])
def test_select_golden_fixture(name, row, want):
    ids, w, _, _ = oracle.select_topk(row[None, :], K=8)
    assert list(ids[0]) == want


def test_select_nonfinite_rows_get_sentinel():
    logits = np.zeros((4, 256), np.float32)
    logits[1, 17] = np.nan
    logits[2, 200] = np.inf
    logits[3, 0] = -np.inf
    ids, w, _, bad = oracle.select_topk(logits, K=8)
    assert bad == 3
    assert list(ids[0]) == list(range(8))
    for t in (1, 2, 3):
        assert (ids[t] == -1).all() and (w[t] == 0).all()


# --------------------------------------------------------------- softmax

def test_softmax_invariants():
    logits = np.stack([W.normal(256, W.stream_key(7, "misc", t)).astype(np.float32) * 3
                       for t in range(64)])
    ids, w, _, _ = oracle.select_topk(logits, K=8)
    assert np.all(np.abs(w.sum(1) - 1) <= 1e-12)
    assert np.all(w > 0) and np.all(w <= 1)
    assert np.all(np.diff(w, axis=1) <= 0)  # non-increasing along rank order


def test_softmax_closed_forms():
    # all 8 selected tied -> 1/8 each
    _, w, _, _ = oracle.select_topk(np.zeros((1, 256), np.float32), K=8)
    assert np.allclose(w, 1 / 8, rtol=0, atol=1e-15)
    # one leader a, seven at b: w0 = 1 / (1 + 7 e^(b-a))
    row = np.full(256, -10.0, np.float32)
    row[5] = 2.0
    row[100:107] = 0.5
    ids, w, _, _ = oracle.select_topk(row[None], K=8)
    assert list(ids[0]) == [5] + list(range(100, 107))
    r = math.exp(0.5 - 2.0)
    assert abs(w[0, 0] - 1 / (1 + 7 * r)) < 1e-15
    assert np.allclose(w[0, 1:], r / (1 + 7 * r), rtol=0, atol=1e-15)
    # the 9th candidate never enters the softmax
    row[50] = 0.25
    _, w2, _, _ = oracle.select_topk(row[None], K=8)
    assert np.array_equal(w, w2)
    # two plateaus golden row: weights e^(v-9) / (2 + 4e^-4 + 2e^-9)
    row = np.array([5, 5, 5, 5, 9, 9] + [0] * 10, np.float32)
    _, w, _, _ = oracle.select_topk(row[None], K=8)
    Z = 2 + 4 * math.exp(-4) + 2 * math.exp(-9)
    want = [1 / Z] * 2 + [math.exp(-4) / Z] * 4 + [math.exp(-9) / Z] * 2
    assert np.allclose(w[0], want, rtol=1e-14, atol=0)


def test_sigmoid_gate_closed_forms():
    g = np.array([0.0, math.log(3.0), -math.log(3.0), 20.0], np.float32)
    _, _, sg, _ = oracle.select_topk(np.zeros((4, 256), np.float32), g, K=8)
    assert sg[0] == 0.5
    assert abs(sg[1] - 0.75) < 1e-7 and abs(sg[2] - 0.25) < 1e-7  # fp32 ln 3
    assert abs(sg[1] + sg[2] - 1) < 1e-15
    assert 1 - sg[3] < 3e-9


# ----------------------------------------------------------------- bf16

def test_bf16_rounding_ties_to_even_and_direct():
    cases = {
        1.0: 0x3F80,
        1 + 2 ** -8: 0x3F80,             # tie -> even (down)
        1 + 3 * 2 ** -8: 0x3F82,         # tie -> even (up)
        1 + 2 ** -8 + 2 ** -40: 0x3F81,  # just above the tie: up (direct, not via fp32)
        -(1 + 2 ** -7): 0xBF81,
        2.0 ** -133: 0x0001,             # smallest subnormal
        2.0 ** -134: 0x0000,             # tie with zero -> even (zero)
        3 * 2.0 ** -134: 0x0002,         # tie between 1 and 2 quanta -> even
        (2 - 2 ** -8) * 2.0 ** 127: 0x7F80,  # rounds past the max -> inf
        (2 - 2 ** -7) * 2.0 ** 127: 0x7F7F,  # the max itself
        -0.0: 0x8000,
    }
    for v, want in cases.items():
        assert oracle.lib().oracle_f64_to_bf16(v) == want, (v, hex(want))
    assert oracle.lib().oracle_f64_to_bf16(float("nan")) == 0x7FC0
    assert oracle.lib().oracle_f64_to_bf16(float("-inf")) == 0xFF80


def test_bf16_rounding_agrees_with_torch_on_fp32_values():
    torch = pytest.importorskip("torch")
    v = (W.normal(200000, W.stream_key(3, "misc")) *
         np.exp(W.normal(200000, W.stream_key(4, "misc")) * 8)).astype(np.float32)
    ours = oracle.f64_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.bf16_to_f64(ours)
    assert np.array_equal(back, W.bf16_bits_to_f32(ours).astype(np.float64))


# ---------------------------------------------------------------- router

def _rand_bf16(shape, seed, std=1.0):
    return W.bf16_normal(shape, W.stream_key(seed, "misc"), std)


def test_router_one_hot_is_column_lookup():
    H, E = 64, 256
    wr = _rand_bf16((E, H), 1, 0.02)
    wg = _rand_bf16((H,), 2, 0.02)
    x = np.zeros((3, H), np.uint16)
    x[0, 5] = bf16([1.0])[0]
    x[1, 63] = bf16([1.0])[0]
    x[2, 0] = bf16([2.0])[0]
    x[2, 9] = bf16([-3.0])[0]
    logits, gate = oracle.router_logits(x, wr, wg)
    assert np.array_equal(logits[0], f(wr[:, 5]).astype(np.float32))
    assert np.array_equal(logits[1], f(wr[:, 63]).astype(np.float32))
    assert np.array_equal(logits[2], (2 * f(wr[:, 0]) - 3 * f(wr[:, 9])).astype(np.float32))
    assert gate[0] == np.float32(f(wg[5:6])[0]) and gate[1] == np.float32(f(wg[63:64])[0])


def test_router_scales_exactly_by_powers_of_two():
    H, E = 256, 256
    wr = _rand_bf16((E, H), 3, 0.02)
    x = _rand_bf16((4, H), 4)
    x2 = bf16(f(x) * 2)
    l1, _ = oracle.router_logits(x, wr)
    l2, _ = oracle.router_logits(x2, wr)
    assert np.array_equal(l2, 2 * l1)


# -------------------------------------------------- groupwise int8 GEMV

def test_w8_gemv_one_hot_reads_q_times_its_group_scale():
    R, C, G = 24, 512, 128
    q = W.int8_uniform(R * C, W.stream_key(5, "misc")).reshape(R, C)
    s = W.bf16_normal((R, C // G), W.stream_key(6, "misc"), 0.01, True)
    for k in (0, 1, G - 1, G, 2 * G + 17, C - 1):
        v = np.zeros(C, np.uint16)
        v[k] = bf16([1.0])[0]
        out = oracle.w8_gemv(q, s, v, G)
        want = q[:, k].astype(np.float64) * f(s[:, k // G])
        assert np.array_equal(out, want), k


def test_w8_gemv_all_ones_sums_v_and_zero_scale_masks_group():
    R, C, G = 8, 384, 128
    v = _rand_bf16((C,), 7)
    q = np.ones((R, C), np.int8)
    s = bf16(np.ones((R, C // G)))
    out = oracle.w8_gemv(q, s, v, G)
    assert np.allclose(out, f(v).sum(), rtol=1e-15, atol=1e-12)
    q = W.int8_uniform(R * C, W.stream_key(8, "misc")).reshape(R, C)
    s = W.bf16_normal((R, C // G), W.stream_key(9, "misc"), 0.01, True)
    s[:, 1] = 0
    v2 = v.copy()
    v2[G:2 * G] = _rand_bf16((G,), 10)
    assert np.array_equal(oracle.w8_gemv(q, s, v, G), oracle.w8_gemv(q, s, v2, G))
    v3 = v.copy()
    v3[0] = bf16([5.0])[0]
    assert not np.array_equal(oracle.w8_gemv(q, s, v, G), oracle.w8_gemv(q, s, v3, G))


def test_w8_gemv_is_bilinear_in_scale_and_input():
    R, C, G = 16, 256, 128
    q = W.int8_uniform(R * C, W.stream_key(11, "misc")).reshape(R, C)
    s = W.bf16_normal((R, C // G), W.stream_key(12, "misc"), 0.01, True)
    v = _rand_bf16((C,), 13)
    base = oracle.w8_gemv(q, s, v, G)
    assert np.array_equal(oracle.w8_gemv(q, bf16(f(s) * 4), v, G), 4 * base)
    assert np.array_equal(oracle.w8_gemv(q, s, bf16(-f(v)), G), -base)
    assert np.array_equal(oracle.w8_gemv(-q, s, v, G), -base)


# --------------------------------------------------------------- SwiGLU

def test_swiglu_closed_forms_and_gate_up_order():
    I = 4
    c = math.log(3.0)
    # gate half = [0, c, 2, -1], up half = [7, 1, 0, 2]
    a = np.array([0.0, c, 2.0, -1.0, 7.0, 1.0, 0.0, 2.0])
    h, hb = oracle.swiglu(a)
    assert h[0] == 0.0                              # silu(0) = 0
    assert abs(h[1] - c * 0.75) < 1e-15             # sigmoid(ln 3) = 3/4
    assert h[2] == 0.0                              # up = 0
    assert abs(h[3] - 2 * (-1) / (1 + math.e)) < 1e-15
    assert np.array_equal(hb, oracle.f64_to_bf16(h))
    # swapped halves would give silu(up) * gate: must differ
    h_sw, _ = oracle.swiglu(np.concatenate([a[I:], a[:I]]))
    assert not np.allclose(h, h_sw)


# --------------------------------------------------------------- combine

def test_combine_linearity_and_special_cases():
    K, H = 8, 64
    y1 = W.normal(K * H, W.stream_key(14, "misc")).reshape(K, H)
    y2 = W.normal(K * H, W.stream_key(15, "misc")).reshape(K, H)
    ys = W.normal(H, W.stream_key(16, "misc"))
    w = np.sort(W.uniform(K, W.stream_key(17, "misc")))[::-1]
    w = w / w.sum()
    o1, _ = oracle.combine(y1, w, ys, 0.3)
    o2, _ = oracle.combine(y2, w, ys, 0.3)
    o12, _ = oracle.combine(2 * y1 - 3 * y2, w, -ys, 0.3)
    assert np.allclose(o12, 2 * o1 - 3 * o2, rtol=1e-12, atol=1e-12)
    # all slots equal -> y * sum(w) + sg * ys = y + sg * ys
    same = np.tile(y1[0], (K, 1))
    o, ob = oracle.combine(same, w, ys, 0.3)
    assert np.allclose(o, y1[0] + 0.3 * ys, rtol=1e-14, atol=1e-14)
    assert np.array_equal(ob, oracle.f64_to_bf16(o))
    # one-hot weight picks its slot; no shared expert
    e3 = np.zeros(K)
    e3[3] = 1
    o, _ = oracle.combine(y1, e3, None, 0.0)
    assert np.array_equal(o, y1[3])


# ---------------------------------------------------------- expert lists

def test_expert_lists_against_python_sort():
    T, K, E = 37, 8, 256
    ids = np.stack([W.permutation(E, W.stream_key(18, "misc", t))[:K] for t in range(T)]
                   ).astype(np.int32)
    ids[5] = np.arange(100, 108)  # several tokens on the same experts
    ids[6] = np.arange(100, 108)[::-1]
    counts, offsets, perm = oracle.expert_lists(ids, E)
    entries = sorted(range(T * K), key=lambda i: (ids.flat[i], i // K, i % K))
    assert list(perm) == entries
    assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    ids[2] = -1
    counts, offsets, perm = oracle.expert_lists(ids, E)
    assert offsets[E] == (T - 1) * K and all(i // K != 2 for i in perm)


# ----------------------------------------------------------- the block

def _tiny_block(seed=0, T=5, H=256, I=128, Is=128, E=16):
    d = {"H": H, "E": E, "K": 8, "I": I, "Is": Is, "G": 128}
    dims = W.Dims(H=H, I=I, Is=Is, E=E)
    w = W.make_weights(dims, seed)
    x, _ = W.make_x(dims, T, seed)
    return d, w, x


def test_block_wiring_expert_scale_ladder():
    """All experts share q and s except the down scale of expert e, which is
    (e+1) times a base: then y_e = (e+1) * y_base and the output must be
    sum_j w_j (id_j + 1) y_base + sigmoid(g) y_shared, exactly in fp64."""
    d, w, x = _tiny_block()
    E, H, I = d["E"], d["H"], d["I"]
    w["w13_q"] = np.repeat(w["w13_q"][:1], E, 0)
    w["w13_s"] = np.repeat(w["w13_s"][:1], E, 0)
    w["w2_q"] = np.repeat(w["w2_q"][:1], E, 0)
    base_s = bf16(np.full((H, I // 128), 2.0 ** -7))
    w["w2_s"] = np.stack([bf16(f(base_s) * (e + 1)) for e in range(E)])
    r = oracle.block_forward(d, w, x, want=("out", "y"))
    for t in range(x.shape[0]):
        a = oracle.w8_gemv(w["w13_q"][0], w["w13_s"][0], x[t])
        _, hb = oracle.swiglu(a)
        y_base = oracle.w8_gemv(w["w2_q"][0], base_s, hb)
        a_s = oracle.w8_gemv(w["ws13_q"], w["ws13_s"], x[t])
        _, hs = oracle.swiglu(a_s)
        ys = oracle.w8_gemv(w["ws2_q"], w["ws2_s"], hs)
        scale = float(np.sum(r["weights"][t] * (r["ids"][t] + 1)))
        want = scale * y_base + r["sgate"][t] * ys
        assert np.allclose(r["out_f64"][t], want, rtol=1e-12, atol=1e-9 * np.abs(want).max())
        assert np.array_equal(r["y"][t, 8], ys)


def test_block_routes_on_supplied_logits_and_gate():
    d, w, x = _tiny_block(seed=1)
    T, E = x.shape[0], d["E"]
    rl = np.tile(np.arange(E, dtype=np.float32), (T, 1))  # ids 15..8 every token
    rg = np.zeros(T, np.float32)
    r = oracle.block_forward(d, w, x, route_logits=rl, route_gate=rg,
                             want=("out", "y"))
    assert (r["ids"] == np.arange(E - 1, E - 9, -1)).all()
    assert (r["sgate"] == 0.5).all()
    ids, wts, _, _ = oracle.select_topk(rl, K=8)
    assert np.array_equal(r["weights"], wts)
    # own logits are still reported and equal the router step's output
    own, gate = oracle.router_logits(x, w["w_router"], w["w_gate"])
    assert np.array_equal(r["logits"], own) and np.array_equal(r["gate_logit"], gate)


def test_block_tokens_are_independent_and_subset_matches():
    d, w, x = _tiny_block(seed=2, T=7)
    full = oracle.block_forward(d, w, x, want=("out",))
    sub = oracle.block_forward(d, w, x, tokens=[6, 2], nthreads=2, want=("out",))
    for t in (2, 6):
        assert np.array_equal(full["out"][t], sub["out"][t])
    alone = oracle.block_forward(d, w, x[2:3], want=("out",))
    assert np.array_equal(alone["out"][0], full["out"][2])


def test_block_nonfinite_row_keeps_only_the_shared_expert():
    d, w, x = _tiny_block(seed=3, T=2)
    rl, rg = oracle.router_logits(x, w["w_router"], w["w_gate"])
    rl[1, 3] = np.nan
    r = oracle.block_forward(d, w, x, route_logits=rl, route_gate=rg, want=("out", "y"))
    assert r["bad"] == 1 and (r["ids"][1] == -1).all()
    assert np.allclose(r["out_f64"][1], r["sgate"][1] * r["y"][1, 8], rtol=1e-15, atol=0)


def test_block_without_shared_expert():
    d, w, x = _tiny_block(seed=4, T=3, Is=0)
    r = oracle.block_forward(d, w, x, want=("out", "y"))
    for t in range(3):
        o, _ = oracle.combine(r["y"][t, :8], r["weights"][t], None, 0.0)
        assert np.array_equal(o, r["out_f64"][t])


def test_workload_skew_gives_shared_top1():
    dims, w, x, info = W.workload_inputs("verify")
    logits, _ = oracle.router_logits(x[info["skewed"]], w["w_router"])
    ids, _, _, _ = oracle.select_topk(logits, K=8)
    assert len(info["skewed"]) == 10
    assert (ids[:, 0] == info["e_star"]).all()
