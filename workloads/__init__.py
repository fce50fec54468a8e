"""Seeded synthetic inputs for the sparse-MoE block.

This module is the one piece both sides of every parity check consume: it
draws the input arrays (bf16 bit patterns as ``uint16``, int8 weights, fp32
logits) and holds none of the block's arithmetic.  The oracle and the CUDA
path each receive the same host arrays from here.

Generator: a counter-based splitmix64.  Output i of the stream with key k is
``mix(k + (i + 1) * 0x9E3779B97F4A7C15)`` where ``mix`` is the splitmix64
finaliser (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014).  Each tensor gets its own key from (seed, tag), so
a tensor's values do not depend on which other tensors were drawn.  Normals
are Box-Muller pairs over two uniforms in (0, 1); bf16 values are fp32
samples rounded to nearest, ties to even.

Workload recipes (shapes and distributions of the pages' model and of the
block's serving configurations):
  * weights: router W and shared gate W ~ bf16(N(0, 0.02)); expert and
    shared-expert int8 weights uniform in [-127, 127]; bf16 scales
    |N(0, 0.01)| per row per group of 128 along the reduction dimension;
  * activations x ~ bf16(N(0, 1));
  * the speculative-verify batch (T = 32 = 8 sequences x 4 draft tokens)
    pushes 10 of its 32 tokens towards one expert e* so that about 30 % of the
    tokens share their top-1 expert: x_t <- x_t + alpha * Wr[e*] / |Wr[e*]|,
    alpha = 6, before the bf16 rounding;
  * selector-only rows: even rows N(0, 1), odd rows integers in [-4, 4]
    (tie-heavy).
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# stream tags: fixed integers so keys never depend on Python's hash seed
TAGS = {"x": 1, "w_router": 2, "w_gate": 3, "w13_q": 4, "w13_s": 5, "w2_q": 6,
        "w2_s": 7, "ws13_q": 8, "ws13_s": 9, "ws2_q": 10, "ws2_s": 11,
        "skew": 12, "logits": 13, "perm": 14, "misc": 15}


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tag: str, sub: int = 0) -> np.uint64:
    base = np.array([(seed * 1000003 + TAGS[tag] * 7919 + sub) & (2**64 - 1)],
                    dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(_mix(base))[0]


def u64(n: int, key: np.uint64, offset: int = 0) -> np.ndarray:
    """n raw 64-bit outputs of the stream ``key`` starting at ``offset``."""
    out = np.empty(n, np.uint64)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            m = min(_CHUNK, n - s)
            c = np.arange(offset + s + 1, offset + s + m + 1, dtype=np.uint64)
            out[s:s + m] = _mix(key + c * GOLDEN)
    return out


def uniform(n: int, key, offset: int = 0) -> np.ndarray:
    """n doubles uniform in (0, 1) (53-bit, never 0 or 1)."""
    u = u64(n, key, offset)
    return ((u >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(n: int, key, offset: int = 0) -> np.ndarray:
    """n standard normals by Box-Muller over consecutive uniform pairs."""
    m = (n + 1) // 2
    u = uniform(2 * m, key, offset)
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    th = 2.0 * np.pi * u[1::2]
    z = np.empty(2 * m, np.float64)
    z[0::2] = r * np.cos(th)
    z[1::2] = r * np.sin(th)
    return z[:n]


# int8 value of each 16-bit draw: multiply-shift of [0, 65536) onto [0, 255)
_I8_LUT = ((np.arange(65536, dtype=np.uint32) * np.uint32(255)) >> np.uint32(16)
           ).astype(np.int16) - 127


def int8_uniform(n: int, key) -> np.ndarray:
    """n int8 uniform in [-127, 127]: four 16-bit draws per 64-bit output
    (draw i of output o is bits 16i..16i+15 of o), mapped by multiply-shift."""
    m = (n + 3) // 4
    out = np.empty(4 * m, np.int8)
    lut = _I8_LUT.astype(np.int8)

    def work(s):
        c = min(_CHUNK, m - s)
        u = u64(c, key, s).astype("<u8")
        out[4 * s:4 * (s + c)] = lut[u.view("<u2")]

    starts = list(range(0, m, _CHUNK))
    if len(starts) > 1:
        with concurrent.futures.ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    else:
        for s0 in starts:
            work(s0)
    return out[:n]


def int_uniform(n: int, key, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] (inclusive), by multiply-shift."""
    span = np.uint64(hi - lo + 1)
    u = u64(n, key) >> np.uint64(32)
    return ((u * span) >> np.uint64(32)).astype(np.int64) + lo


def permutation(n: int, key) -> np.ndarray:
    return np.argsort(uniform(n, key), kind="stable").astype(np.int64)


def f32_to_bf16_bits(v) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest, ties to even (finite)."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def bf16_normal(shape, key, std: float = 1.0, absolute: bool = False):
    z = normal(int(np.prod(shape)), key) * std
    if absolute:
        z = np.abs(z)
    return f32_to_bf16_bits(z.astype(np.float32)).reshape(shape)


# ------------------------------------------------------------- workloads

@dataclasses.dataclass(frozen=True)
class Dims:
    H: int
    I: int
    Is: int
    E: int = 256
    K: int = 8
    G: int = 128

    def as_dict(self):
        return dataclasses.asdict(self)

    @property
    def expert_bytes(self) -> int:
        """int8 weights + bf16 scales of one routed expert (gate|up and down)."""
        H, I, G = self.H, self.I, self.G
        return 2 * I * H + 2 * (2 * I * (H // G)) + H * I + 2 * (H * (I // G))

    @property
    def shared_bytes(self) -> int:
        H, I, G = self.H, self.Is, self.G
        return 2 * I * H + 2 * (2 * I * (H // G)) + H * I + 2 * (H * (I // G))

    @property
    def router_bytes(self) -> int:
        return 2 * self.E * self.H + (2 * self.H if self.Is else 0)


PR1 = Dims(H=512, I=128, Is=128)
FULL = Dims(H=2048, I=512, Is=512)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    T: int
    seed: int
    skew_tokens: int = 0


WORKLOADS = {
    "pr1": Workload("pr1", PR1, 4, 0),
    "decode": Workload("decode", FULL, 1, 1),
    "verify": Workload("verify", FULL, 32, 2, skew_tokens=10),
    "prefill": Workload("prefill", FULL, 2048, 3),
}

SELECTOR_T = (1, 4, 32, 64)


def make_weights(d: Dims, seed: int) -> dict:
    """All weights of one block as host arrays (uint16 = bf16 bits)."""
    E, H, I, Is, G = d.E, d.H, d.I, d.Is, d.G
    k = lambda tag: stream_key(seed, tag)
    w = {
        "w_router": bf16_normal((E, H), k("w_router"), 0.02),
        "w_gate": bf16_normal((H,), k("w_gate"), 0.02) if Is else None,
        "w13_q": int8_uniform(E * 2 * I * H, k("w13_q")).reshape(E, 2 * I, H),
        "w13_s": bf16_normal((E, 2 * I, H // G), k("w13_s"), 0.01, True),
        "w2_q": int8_uniform(E * H * I, k("w2_q")).reshape(E, H, I),
        "w2_s": bf16_normal((E, H, I // G), k("w2_s"), 0.01, True),
    }
    if Is:
        w.update({
            "ws13_q": int8_uniform(2 * Is * H, k("ws13_q")).reshape(2 * Is, H),
            "ws13_s": bf16_normal((2 * Is, H // G), k("ws13_s"), 0.01, True),
            "ws2_q": int8_uniform(H * Is, k("ws2_q")).reshape(H, Is),
            "ws2_s": bf16_normal((H, Is // G), k("ws2_s"), 0.01, True),
        })
    else:
        w.update({"ws13_q": None, "ws13_s": None, "ws2_q": None, "ws2_s": None})
    return w


def make_x(d: Dims, T: int, seed: int, skew_tokens: int = 0,
           w_router=None, alpha: float = 6.0):
    """Activations [T][H] (bf16 bits); optionally push ``skew_tokens`` tokens
    towards one expert.  Returns (x, info) with info = {"e_star", "skewed"}."""
    z = normal(T * d.H, stream_key(seed, "x")).reshape(T, d.H)
    info = {"e_star": None, "skewed": np.zeros(0, np.int64)}
    if skew_tokens:
        ks = stream_key(seed, "skew")
        e_star = int(int_uniform(1, ks, 0, d.E - 1)[0])
        toks = np.sort(permutation(T, stream_key(seed, "skew", 1))[:skew_tokens])
        wr = bf16_bits_to_f32(w_router[e_star]).astype(np.float64)
        z[toks] += alpha * wr / np.linalg.norm(wr)
        info = {"e_star": e_star, "skewed": toks}
    return f32_to_bf16_bits(z.astype(np.float32)), info


def make_selector_logits(T: int, E: int = 256, seed: int | None = None):
    """Selector-only rows: even t ~ N(0,1), odd t integers in [-4, 4]."""
    seed = T if seed is None else seed
    out = np.empty((T, E), np.float32)
    for t in range(T):
        k = stream_key(seed, "logits", t)
        if t % 2 == 0:
            out[t] = normal(E, k).astype(np.float32)
        else:
            out[t] = int_uniform(E, k, -4, 4).astype(np.float32)
    return out


# Candidate selection over a vocabulary: 8 block positions (a draft of 7
# tokens plus the anchor) against a 151,936-wide lm_head row.
CANDIDATES_T, CANDIDATES_N, CANDIDATES_K = 8, 151936, 16


def make_candidate_logits(T: int, N: int, seed: int):
    """Wide rows: even t ~ 3*N(0,1) (fp32), odd t integers in [-8, 8] (many
    ties, so the lower-id rule decides most places)."""
    out = np.empty((T, N), np.float32)
    for t in range(T):
        k = stream_key(seed, "logits", 1000 + t)
        if t % 2 == 0:
            out[t] = (3.0 * normal(N, k)).astype(np.float32)
        else:
            out[t] = int_uniform(N, k, -8, 8).astype(np.float32)
    return out


def workload_inputs(name: str, T: int | None = None, seed: int | None = None):
    """(dims, weights, x, info) of a named workload, T/seed overridable."""
    wl = WORKLOADS[name]
    T = wl.T if T is None else T
    seed = wl.seed if seed is None else seed
    w = make_weights(wl.dims, wl.seed)
    x, info = make_x(wl.dims, T, seed, wl.skew_tokens if T == wl.T else 0,
                     w["w_router"])
    return wl.dims, w, x, info


def expert_permutation(E: int, seed: int, bank: int) -> np.ndarray:
    """A seeded relabelling of the experts (bank 0 is the identity)."""
    if bank == 0:
        return np.arange(E, dtype=np.int64)
    return permutation(E, stream_key(seed, "perm", bank))
