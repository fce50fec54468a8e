"""Benchmark of the GB300 sparse-MoE block (one JSON line on rank 0).

Metric: MoE-block tokens/s at the serving configurations T = 1 (decode),
T = 32 (speculative verify, 8 sequences x 4 draft tokens) and T = 2048
(prefill chunk); H = 2048, 256 experts top-8, I = Is = 512, int8 group-128
weights with bf16 scales, bf16 activations.  The headline `value` is the
workload named by --workload (default: verify T=32); the other two are in
`workloads`.

Timing protocol:
  * weights and inputs are resident in HBM before timing starts;
  * L2 stays cold across steps: R rotating weight banks (each a relabelled
    copy of the seeded weights with its experts permuted, so the same math
    reads different memory) and R distinct inputs; the bytes one lap of the
    banks touches exceed L2 (129 MB) many times over;
  * each step is one CUDA-graph replay of moe_block_forward; W warm-up steps,
    then exactly K timed steps between CUDA events, barrier + synchronize on
    both sides, max over ranks; an event after every step gives the median
    and minimum step time beside the mean, and five replays on an idle
    device give the single-call latency (`workloads`);
  * a second timed pass runs the profiled entry point (events between the
    block's kernels) to give the dominant kernel's average duration;
  * e2e: moe_block_forward_host with pinned host x/out, copies inside;
  * cpu_baseline: the fp64 oracle on this host's cores, on a bounded sample.
Multi-GPU: replicas only (the block has no exchange step); each rank runs
the same workload on its own GPU and `value` sums the ranks' tokens.
Unless --only is given, `workloads` also times a stack of eight decoder-layer
blocks at T = 1 in one CUDA graph (moe_block_forward_residual: the block, the
residual add and the next layer's RMS norm; per-layer time, L2-cold) and the
wide-row top-16 candidate selector (T = 8 and 64 rows of a 151,936-wide
vocabulary, L2-cold).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

WORKLOAD_T = {"decode": 1, "verify": 32, "prefill": 2048}
LABEL = {"decode": "decode_T1", "verify": "verify_T32", "prefill": "prefill_T2048"}


def read_peak_gbs(torch, dev, gib: float = 2.0, reps: int = 5):
    """Self-measured read-only HBM bandwidth: a reduction over a buffer far
    larger than L2, best of reps, CUDA events (a measurement aid, not the
    hot path)."""
    n = int(gib * (1 << 30)) // 4
    buf = torch.ones(n, dtype=torch.float32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = None
    for _ in range(reps + 1):
        e0.record()
        buf.sum()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    del buf
    torch.cuda.empty_cache()
    return n * 4 / (best * 1e-3) / 1e9


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "src": "fallback"}


# --------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------- workloads

def algorithmic_bytes(d: W.Dims, T: int, n_active: int):
    """Bytes the method must touch: each distinct routed expert's int8
    weights + scales once, the shared expert, router + gate rows, x in, out."""
    return ((n_active + (1 if d.Is else 0)) * d.expert_bytes + d.router_bytes +
            2 * 2 * T * d.H)


def gateup_bytes(d: W.Dims, T: int, n_active: int):
    H, I, Is, G = d.H, d.I, d.Is, d.G
    per = 2 * I * H + 2 * 2 * I * (H // G)
    sh = 2 * Is * H + 2 * 2 * Is * (H // G) if Is else 0
    return n_active * per + sh + 2 * T * H + 2 * (T * 8 * I + T * Is)


def down_bytes(d: W.Dims, T: int, n_active: int):
    """Down projection + combine: each routed expert's down weights + scales
    once, the shared expert's, the h rows in, the bf16 output out."""
    H, I, Is, G = d.H, d.I, d.Is, d.G
    per = H * I + 2 * H * (I // G)
    sh = H * Is + 2 * H * (Is // G) if Is else 0
    return n_active * per + sh + 2 * (T * 8 * I + T * Is) + 2 * T * H


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# one ncu capture of each kernel (summaries under profiles/), valid only while
# the kernel's sources hash to the value recorded with the capture.
MEASURED_TRAFFIC = {
    "decode_fused": {"bytes": 529.7e6, "workload": "verify_T32",
                     "sources": ["decode_fused.cu", "common.cuh", "select.cuh", "sm100_ptx.cuh"],
                     "sha256_16": "9f47c0b17b71b145",
                     "profile": "profiles/decode_fused_verify_T32.md"},
    "gateup_swiglu_tc": {"bytes": 645.6e6, "workload": "prefill_T2048",
                         "sources": ["tc_expert.cu", "common.cuh", "sm100_ptx.cuh"],
                         "sha256_16": "fb7eb20b93e03113",
                         "profile": "profiles/split_kernels_prefill_T2048.md"},
    "down_combine_tc": {"bytes": 312.8e6, "workload": "prefill_T2048",
                        "sources": ["tc_expert.cu", "common.cuh", "sm100_ptx.cuh"],
                        "sha256_16": "fb7eb20b93e03113",
                        "profile": "profiles/split_kernels_prefill_T2048.md"},
}


# The candidate selector's first kernel, captured at 64 rows (the runs it
# writes stay in L2; the merge kernel reads them there): DRAM bytes per row.
CANDIDATES_TRAFFIC = {"bytes_per_row": 38.93e6 / 64, "rows_captured": 64,
                      "sources": ["topk.cu", "common.cuh"], "sha256_16": "382c56906eaa3e6e",
                      "profile": "profiles/topk_chunk_candidates_T64.md"}


def candidates_traffic(T: int):
    """DRAM bytes of one candidate-selection call of T rows, from the capture
    at 64 rows scaled by rows (each row is read once), or None when the
    kernel's sources changed since."""
    m = CANDIDATES_TRAFFIC
    h = hashlib.sha256()
    for f in m["sources"]:
        with open(os.path.join(HERE, "sparse_moe_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return m["bytes_per_row"] * T if h.hexdigest()[:16] == m["sha256_16"] else None


def measured_traffic(kname: str, workload: str):
    """The captured traffic of kname on this workload, or None when there is
    no capture or the kernel's sources changed since it was taken."""
    m = MEASURED_TRAFFIC.get(kname)
    if not m or m["workload"] != workload:
        return None
    h = hashlib.sha256()
    for f in m["sources"]:
        with open(os.path.join(HERE, "sparse_moe_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return m["bytes"] if h.hexdigest()[:16] == m["sha256_16"] else None


def kernel_bytes(kname: str, d: W.Dims, T: int, n_active: int):
    """Algorithmic bytes of one launch of a block kernel, None for kernels
    that run the whole block (the block's bytes apply)."""
    if kname in ("gateup_swiglu", "gateup_swiglu_tc"):
        return gateup_bytes(d, T, n_active)
    if kname in ("down", "down_combine_tc"):
        return down_bytes(d, T, n_active)
    return None


def algorithmic_flops(d: W.Dims, T: int):
    H, I, Is = d.H, d.I, d.Is
    return 2 * T * (8 * 3 * I * H + 3 * Is * H + 256 * H + H)


class Bench:
    def __init__(self, name, moe, torch, dev, banks, seed_base=0):
        self.name = name
        self.moe, self.torch, self.dev = moe, torch, dev
        wl = W.WORKLOADS[name]
        self.d = wl.dims
        self.T = T = WORKLOAD_T[name]
        self.R = banks
        host_w = W.make_weights(self.d, wl.seed)
        self.host_w = host_w
        base = {k: self._up(v) for k, v in host_w.items()}
        # R banks: bank r relabels experts by a seeded permutation
        self.banks, self.keep = [], []
        for r in range(banks):
            perm = torch.from_numpy(W.expert_permutation(256, wl.seed, r)).to(dev)
            w = dict(base)
            if r > 0:
                for k in ("w_router", "w13_q", "w13_s", "w2_q", "w2_s"):
                    w[k] = base[k].index_select(0, perm).contiguous()
            self.keep.append(w)
            self.banks.append(moe.weights_struct(w))
        # R inputs
        self.x_host, self.x = [], []
        for r in range(banks):
            x, _ = W.make_x(self.d, T, wl.seed * 1000 + r, wl.skew_tokens, host_w["w_router"])
            self.x_host.append(x)
            self.x.append(self._up(x))
        self.dims = moe.Dims.make(self.d.H, self.d.I, self.d.Is)
        self.ws_bytes = moe.moe_workspace_bytes(self.dims, T)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.out = torch.empty((T, self.d.H), dtype=torch.int16, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.nk = moe.moe_block_kernel_count(self.dims, T)
        self.kernel_names = [moe.moe_block_kernel_name(self.dims, T, i) for i in range(self.nk)]
        # routing of each input (bank 0 computes the same ids up to relabelling)
        ids = torch.empty((T, 8), dtype=torch.int32, device=dev)
        self.n_active = []
        self.per_expert = []  # (min, max) tokens per expert over the 256 experts
        for r in range(banks):
            moe.moe_block_forward(self.dims, self.banks[0], self.x[r], T, self.out, ids, None,
                                  None, None, self.ws, self.ws_bytes)
            h = ids.cpu().numpy().ravel()
            self.n_active.append(len(np.unique(h[h >= 0])))
            cnt = np.bincount(h[h >= 0], minlength=256)
            self.per_expert.append((int(cnt.min()), int(cnt.max())))
        torch.cuda.synchronize()
        assert moe.moe_read_status(self.ws) == 0

    def _up(self, a):
        if a is None:
            return None
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return self.torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def step(self, r, events=None):
        if events is None:
            self.moe.moe_block_forward(self.dims, self.banks[r], self.x[r], self.T, self.out, None,
                                       None, None, None, self.ws, self.ws_bytes, self.stream)
        else:
            self.moe.moe_block_forward_profiled(self.dims, self.banks[r], self.x[r], self.T,
                                                self.out, self.ws, self.ws_bytes, events,
                                                self.stream)

    def graphs(self):
        torch = self.torch
        gs = []
        with torch.cuda.stream(self.stream):
            for r in range(self.R):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    self.step(r)
                gs.append(g)
        self.plain = gs

    def run(self, steps, warmup, barrier, clocks_index):
        torch = self.torch
        self.graphs()
        s = self.stream
        with torch.cuda.stream(s):  # replays launch on the current stream
            for i in range(warmup):
                self.plain[i % self.R].replay()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(self.nk + 1)]
                  for _ in range(steps)]
        with Clocks(clocks_index) as clk:
            torch.cuda.synchronize()
            barrier()
            step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
            t_wall = time.perf_counter()
            with torch.cuda.stream(s):
                e0.record(s)
                for i in range(steps):
                    self.plain[i % self.R].replay()
                    step_ev[i].record(s)
                e1.record(s)
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - t_wall
            barrier()
            ms = e0.elapsed_time(e1) / steps
            per_step = [e0.elapsed_time(step_ev[0])] + [
                step_ev[i - 1].elapsed_time(step_ev[i]) for i in range(1, steps)]
            # single-call latency: one replay on an idle device, five times,
            # each of a bank replayed longest ago (the timed loop's last step
            # used bank (steps - 1) % R, so bank (steps + i) % R was last read
            # at least R - 5 steps ago, and L2 holds none of its bytes)
            single = []
            for i in range(5):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                with torch.cuda.stream(s):
                    a.record(s)
                    self.plain[(steps + i) % self.R].replay()
                    b.record(s)
                torch.cuda.synchronize()
                single.append(a.elapsed_time(b))
            self.step_stats = {"ms_median": float(statistics.median(per_step)),
                               "ms_min": float(min(per_step)),
                               "single_call_ms_median": float(statistics.median(single))}
            # profiled pass: the same K steps through the profiled entry point,
            # events between kernels; a bounded sleep kernel first lets the host
            # enqueue every step so kernels run back to back on the device
            with torch.cuda.stream(s):
                for ev in events:
                    for e in ev:
                        e.record(s)  # creates the event handles
                torch.cuda.synchronize()
                torch.cuda._sleep(50_000_000)
                for i in range(steps):
                    self.step(i % self.R, events[i])
            torch.cuda.synchronize()
        per_kernel = np.zeros(self.nk)
        for ev in events:
            for k in range(self.nk):
                per_kernel[k] += ev[k].elapsed_time(ev[k + 1])
        per_kernel /= max(1, steps)
        assert self.moe.moe_read_status(self.ws) == 0
        return ms, t_wall, per_kernel, clk.summary()

    def e2e(self, steps, warmup):
        """Whole call through the host entry point: H2D of x, block, D2H."""
        torch = self.torch
        xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in self.x_host]
        oh = torch.empty((self.T, self.d.H), dtype=torch.int16).pin_memory()
        for i in range(warmup):
            self.moe.moe_block_forward_host(self.dims, self.banks[i % self.R], xh[i % self.R],
                                            self.T, oh, self.ws, self.ws_bytes, self.stream)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for i in range(steps):
            self.moe.moe_block_forward_host(self.dims, self.banks[i % self.R], xh[i % self.R],
                                            self.T, oh, self.ws, self.ws_bytes, self.stream)
        t = time.perf_counter() - t
        return t / steps, 2 * self.T * self.d.H, 2 * self.T * self.d.H


def bench_layers(moe, torch, dev, T: int, n_layers: int, steps: int, warmup: int,
                 barrier=lambda: None, max_all=lambda v: v):
    """A stack of decoder-layer blocks at decode size, as a serving loop runs
    them: each layer is moe_block_forward_residual (the block, the residual
    added in its combine, the next layer's RMS-normed input) on its own
    weight bank (an expert-permuted copy of the seeded weights), x and the
    residual carried in place from layer to layer, all layers captured in
    one CUDA graph.  Two such stacks on distinct banks alternate between
    replays, so L2 holds none of a replay's weights.  The same stacks of
    plain moe_block_forward calls are timed beside them."""
    name = "decode"
    wl = W.WORKLOADS[name]
    d = wl.dims
    host_w = W.make_weights(d, wl.seed)
    base = {k: (torch.from_numpy(np.ascontiguousarray(v.view(np.int16) if v.dtype == np.uint16
                                                      else v)).to(dev) if v is not None else None)
            for k, v in host_w.items()}
    keep, banks = [], []
    for r in range(2 * n_layers):
        perm = torch.from_numpy(W.expert_permutation(256, wl.seed, 100 + r)).to(dev)
        w = dict(base)
        for k in ("w_router", "w13_q", "w13_s", "w2_q", "w2_s"):
            w[k] = base[k].index_select(0, perm).contiguous()
        keep.append(w)
        banks.append(moe.weights_struct(w))
    dims = moe.Dims.make(d.H, d.I, d.Is)
    wsb = moe.moe_workspace_bytes(dims, T)
    ws = torch.zeros(wsb, dtype=torch.uint8, device=dev)
    x0 = torch.from_numpy(W.make_x(d, T, 4242)[0].view(np.int16)).to(dev)
    r0 = torch.from_numpy(W.bf16_normal((T, d.H), W.stream_key(4243, "misc"), 4.0)
                          .view(np.int16)).to(dev)
    gammas = [torch.from_numpy(W.bf16_normal((d.H,), W.stream_key(4244, "misc", l), 1.0)
                               .view(np.int16)).to(dev) for l in range(n_layers)]
    x = x0.clone()
    resid = r0.clone()
    out = torch.empty_like(x0)
    s = torch.cuda.Stream(device=dev)

    def stack(k, residual):
        for l in range(n_layers):
            wb = banks[k * n_layers + l]
            if residual:
                moe.moe_block_forward_residual(dims, wb, x, T, resid, gammas[l], 1e-6, resid, x,
                                               ws, wsb, s)
            else:
                moe.moe_block_forward(dims, wb, x, T, out, None, None, None, None, ws, wsb, s)

    res = {}
    for residual in (True, False):
        with torch.cuda.stream(s):
            for k in range(2):  # eager pass first (checks the calls)
                stack(k, residual)
            graphs = []
            for k in range(2):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    stack(k, residual)
                graphs.append(g)
            for i in range(warmup):
                graphs[i % 2].replay()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            for i in range(steps):
                graphs[i % 2].replay()
            e1.record(s)
        torch.cuda.synchronize()
        barrier()
        us = max_all(e0.elapsed_time(e1) * 1e3 / (steps * n_layers))
        res["us_per_layer" if residual else "us_per_layer_block_only"] = us
    assert moe.moe_read_status(ws) == 0
    res.update({"T": T, "layers": n_layers, "kernels_per_layer": 2,
                "tokens_per_s_per_layer": T / (res["us_per_layer"] * 1e-6),
                "l2": "cold: two stacks of %d layers on distinct weight banks alternate" %
                      n_layers})
    return res


def bench_candidates(moe, torch, dev, T: int, steps: int, warmup: int, peak_gbs: float,
                     barrier=lambda: None, max_all=lambda v: v, world: int = 1):
    """Wide-row top-16 candidates (the drafter's lm_head candidate selector):
    T rows of the 151,936-wide vocabulary.  R rotating input buffers, more
    than twice L2 in all, captured as R calls in one CUDA graph; per-call
    time = replay time / R."""
    N, k = W.CANDIDATES_N, W.CANDIDATES_K
    row_bytes = N * 4
    R = max(8, -(-300_000_000 // (T * row_bytes)))
    bufs = [torch.from_numpy(W.make_candidate_logits(T, N, seed=500 + r)).to(dev)
            for r in range(min(R, 4))]
    bufs += [bufs[r % len(bufs)].clone() for r in range(len(bufs), R)]
    ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    vals = torch.empty((T, k), dtype=torch.float32, device=dev)
    ws_bytes = moe.moe_topk_workspace_bytes(T, N)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(s):
        for r in range(R):  # eager pass: checks the calls before capture
            moe.moe_topk_candidates(bufs[r], T, N, N, k, ids, vals, ws, ws_bytes, s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for r in range(R):
                moe.moe_topk_candidates(bufs[r], T, N, N, k, ids, vals, ws, ws_bytes, s)
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        for _ in range(steps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    barrier()
    assert moe.moe_read_status(ws) == 0
    us = max_all(e0.elapsed_time(e1) * 1e3 / (steps * R))
    nbytes = T * row_bytes + T * k * 8
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"rows_per_s": world * T / (us * 1e-6), "us_per_call": us, "T": T, "N": N, "k": k,
            "algorithmic_bytes": nbytes, "achieved_gbs": gbs, "frac_hbm_measured": gbs / peak_gbs,
            "kernels_per_call": 2, "l2": "cold: %d rotating inputs of %.1f MB" % (R, T * row_bytes / 1e6)}


def candidates_main(args, rank: int):
    """--workload candidates: the top-16 candidate selector alone (replicas
    on several GPUs, like the block)."""
    import torch
    import __graft_entry__ as g
    g.build()
    import sparse_moe_decode_gb300 as moe
    world = int(os.environ.get("WORLD_SIZE", "1"))
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    barrier, max_all = collectives(dist, dev)
    pk = peaks()
    r = bench_candidates(moe, torch, dev, args.cand_T, args.steps, args.warmup, pk["hbm_gbs"],
                         barrier, max_all, world)
    if rank == 0:
        cb = oracle_candidates(args.cand_T, budget_s=args.cpu_budget)
        print(json.dumps({"metric": "candidate_rows_per_s", "value": r["rows_per_s"],
                          "unit": "rows/s", "n_gpus": world, "steps": args.steps,
                          "scaling": "weak",
                          "warmup": args.warmup, "ms_per_step": r["us_per_call"] * 1e-3,
                          "higher_is_better": True, "dtype": "f32", "data": "synthetic",
                          "config": {"workload": "candidates_T%d_N%d_k%d" % (
                              r["T"], r["N"], r["k"]), "l2": r["l2"]},
                          "roofline": {"bound": "hbm", "kernel": "topk_chunk + topk_merge",
                                       "achieved": r["achieved_gbs"], "peak": pk["hbm_gbs"],
                                       "unit": "GB/s", "frac": r["frac_hbm_measured"],
                                       "traffic": candidates_traffic(r["T"]),
                                       "traffic_src": "ncu capture at 64 rows, scaled by rows",
                                       "peak_src": pk["src"]},
                          "cpu_baseline": cb, "candidates": r}))


def _oracle_inputs(name: str, n: int):
    wl = W.WORKLOADS[name]
    w = W.make_weights(wl.dims, wl.seed)
    T = WORKLOAD_T[name]
    x, _ = W.make_x(wl.dims, max(n, T), wl.seed * 1000, wl.skew_tokens if n <= T else 0,
                    w["w_router"])
    return wl.dims, w, x


def oracle_steps(name: str, steps: int, warmup: int, budget_s: float | None = None,
                 threads: int | None = None):
    """The oracle as it stands on this host's cores (all of them, or
    `threads`).  One step = `cores` tokens of the workload's recipe through
    A1..A7 (fp64, one token per thread at a time).  With a budget, the
    number of steps is cut to fit it."""
    import oracle
    cores = threads or os.cpu_count() or 1
    dims, w, x = _oracle_inputs(name, cores)
    toks = np.arange(cores, dtype=np.int32)

    def one():
        oracle.block_forward(dims.as_dict(), w, x, tokens=toks, nthreads=cores)

    for _ in range(warmup):
        one()
    t0 = time.perf_counter()
    done = 0
    while done < steps:
        one()
        done += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    T = WORKLOAD_T[name]
    return {"value": done * cores / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d steps x %d tokens drawn like the %s batch (T=%d) through the fp64 "
                      "oracle, %d threads, %.1f s" % (done, cores, LABEL[name], T, cores, dt)}


def oracle_candidates(T: int, budget_s: float = 10.0):
    """The oracle's top-16 selection (a full sort of each row) on rows of the
    candidate workload, one row at a time, until the budget is spent."""
    import oracle
    rows = W.make_candidate_logits(min(T, 4), W.CANDIDATES_N, seed=500)
    oracle.candidates_topk(rows[:1], W.CANDIDATES_K)  # builds and loads the library
    t0 = time.perf_counter()
    done = 0
    while done < 1000:
        oracle.candidates_topk(rows[done % rows.shape[0]][None, :], W.CANDIDATES_K)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": "%d rows of %d fp32 logits, top-%d by a full qsort in the fp64 oracle "
                      "library, 1 thread, %.1f s" % (done, W.CANDIDATES_N, W.CANDIDATES_K, dt)}


def cpu_baseline(name: str, budget_s: float = 10.0):
    """The oracle on all host cores, with its one-thread figure beside it."""
    cb = oracle_steps(name, steps=1000, warmup=1, budget_s=budget_s)
    one = oracle_steps(name, steps=1000, warmup=0, budget_s=budget_s / 2, threads=1)
    cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1,
                           "sample": one["sample"]}
    return cb


def collectives(dist, device):
    """The replicas' timing collectives for any backend (NCCL on GPUs, gloo in
    the CPU tests): a barrier, and the maximum of a float over the ranks."""

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_all(v):
        if dist is None:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    return barrier, max_all


def whole_job_tokens_per_s(world: int, T: int, ms_max: float) -> float:
    """Every rank runs T tokens per step; the job's step time is the slowest
    rank's, so the whole job moves world * T tokens per ms_max."""
    return world * T / (ms_max * 1e-3)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_T) + ["candidates"], default="verify",
                    help="'candidates': only the top-16 candidate selector, one JSON line")
    ap.add_argument("--cand-T", type=int, default=W.CANDIDATES_T,
                    help="rows of the candidate selector for --workload candidates")
    ap.add_argument("--only", action="store_true", help="time only --workload")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--banks", type=int, default=0,
                    help="weight banks (default 16 for T <= 32, else 2); fewer keep a "
                         "profiler capture small, and a bench line taken with them says so")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.workload == "candidates":
        if args.impl == "reference":
            if rank == 0:
                cb = oracle_candidates(args.cand_T, budget_s=max(args.cpu_budget, 1.0))
                print(json.dumps({
                    "impl": "reference", "metric": "candidate_rows_per_s", "value": cb["value"],
                    "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
                    "warmup": args.warmup, "ms_per_step": 1e3 / cb["value"],
                    "higher_is_better": True, "dtype": "f64", "data": "synthetic",
                    "config": {"workload": "candidates_T%d_N%d_k%d" % (
                        args.cand_T, W.CANDIDATES_N, W.CANDIDATES_K)},
                    "cpu_baseline": cb,
                    "e2e": {"value": cb["value"], "unit": "rows/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}))
            return
        return candidates_main(args, rank)

    if args.impl == "reference":
        # the oracle is the reference arm: rank 0 only, host cores
        if rank != 0:
            return
        cb = oracle_steps(args.workload, args.steps, args.warmup, budget_s=240.0)
        T = WORKLOAD_T[args.workload]
        line = {"impl": "reference", "metric": "moe_block_tokens_per_s", "value": cb["value"],
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * (os.cpu_count() or 1) / cb["value"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": LABEL[args.workload], "T": T,
                                                "H": 2048, "I": 512, "Is": 512, "E": 256,
                                                "K": 8, "G": 128},
                "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    import __graft_entry__ as g
    g.build()
    import sparse_moe_decode_gb300 as moe

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    barrier, max_all = collectives(dist, dev)

    pk = peaks()
    read_gbs = read_peak_gbs(torch, dev) if world == 1 or rank == 0 else None
    order = [args.workload] + ([] if args.only else
                               [n for n in ("decode", "verify", "prefill") if n != args.workload])
    results = {}
    head = None
    for name in order:
        T = WORKLOAD_T[name]
        banks = args.banks if args.banks > 0 else (16 if T <= 32 else 2)
        b = Bench(name, moe, torch, dev, banks)
        ms, wall, per_kernel, clk = b.run(args.steps, args.warmup, barrier, local)
        ms = max_all(ms)
        d = b.d
        n_act = float(np.mean(b.n_active))
        bytes_step = algorithmic_bytes(d, T, n_act)
        gbs = bytes_step / (ms * 1e-3) / 1e9
        flops = algorithmic_flops(d, T)
        tfs = flops / (ms * 1e-3) / 1e12
        t_hbm = bytes_step / (pk["hbm_gbs"] * 1e9)
        t_tc = flops / (pk["bf16_tflops"] * 1e12)
        k_dom = int(np.argmax(per_kernel))
        r = {
            "tokens_per_s": whole_job_tokens_per_s(world, T, ms), "ms_per_step": ms,
            "T": T, "n_active_experts": n_act, "algorithmic_bytes": bytes_step,
            "achieved_gbs": gbs, "frac_hbm_measured": gbs / pk["hbm_gbs"],
            "frac_hbm_8000": gbs / 8000.0, "tflops": tfs,
            "frac_bf16_peak": tfs / pk["bf16_tflops"],
            "frac_bf16_peak_sustained": (tfs / pk["bf16_tflops_sustained"]
                                         if pk.get("bf16_tflops_sustained") else None),
            "frac_hbm_read_self": gbs / read_gbs if read_gbs else None,
            "tokens_per_expert_min_max": [min(a for a, _ in b.per_expert),
                                          max(c for _, c in b.per_expert)],
            "frac_roofline_time": max(t_hbm, t_tc) / (ms * 1e-3),
            "kernels_ms": {n: float(v) for n, v in zip(b.kernel_names, per_kernel)},
            "dominant_kernel": b.kernel_names[k_dom], "wall_s": wall, "clocks": clk,
            "banks": banks, **b.step_stats,
        }
        if name == args.workload:
            kb = kernel_bytes(b.kernel_names[k_dom], d, T, n_act)
            r["_kernel"] = (b.kernel_names[k_dom], per_kernel[k_dom], kb)
            e2e_s, bi, bo = b.e2e(args.steps, args.warmup)
            e2e_s = max_all(e2e_s)
            r["e2e"] = {"value": whole_job_tokens_per_s(world, T, e2e_s * 1e3),
                        "unit": "tokens/s", "h2d_bytes_per_step": bi,
                        "d2h_bytes_per_step": bo}
            r["gpu_launches"] = args.steps * b.nk
            head = r
        results[LABEL[name]] = r
        del b
        torch.cuda.empty_cache()

    if not args.only:
        results["decode_T1_layers8"] = bench_layers(moe, torch, dev, 1, 8, args.steps,
                                                    args.warmup, barrier, max_all)
        for Tc in (W.CANDIDATES_T, 64):
            results["candidates_T%d_N%d_k%d" % (Tc, W.CANDIDATES_N, W.CANDIDATES_K)] = \
                bench_candidates(moe, torch, dev, Tc, args.steps, args.warmup, pk["hbm_gbs"],
                                 barrier, max_all, world)
    if rank != 0:
        return
    kname, kms, kbytes = head.pop("_kernel")
    if kbytes is None:  # fall back to the block's bytes for another dominant kernel
        kbytes = head["algorithmic_bytes"]
    achieved = kbytes / (kms * 1e-3) / 1e9
    roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": pk["hbm_gbs"],
            "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
            "traffic": measured_traffic(kname, LABEL[args.workload]),
            "peak_src": pk["src"] + " (copy, burst)", "kernel_ms": kms,
            "read_peak_self_gbs": read_gbs,
            "algorithmic_bytes_per_launch": kbytes}
    cb = cpu_baseline(args.workload, budget_s=args.cpu_budget) if world == 1 or rank == 0 else None
    line = {
        "metric": "moe_block_tokens_per_s", "value": head["tokens_per_s"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8*bf16->f32", "data": "synthetic",
        "config": {"workload": LABEL[args.workload], "T": head["T"], "H": 2048, "I": 512,
                   "Is": 512, "E": 256, "K": 8, "G": 128, "parallelism": "replicas" if world > 1
                   else "single", "l2": "cold: %d rotating weight banks (expert-permuted copies) "
                   "and %d inputs, larger than L2" % (head["banks"], head["banks"])},
        "roofline": roof, "cpu_baseline": cb, "e2e": head.pop("e2e"),
        "gpu_launches": head.pop("gpu_launches"), "clocks": head["clocks"],
        "workloads": results,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
