"""Plain fp64 CPU oracle of the sparse-MoE block (ctypes wrapper).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product package ``sparse_moe_decode_gb300`` never imports it,
and the two share no code: the C source here (``moe_oracle.c``) is compiled by
gcc on its own, and the only thing both sides consume is the seeded input
arrays.

Arrays use numpy: bf16 values travel as ``uint16`` bit patterns, int8 weights
as ``int8``, logits as ``float32``, everything the oracle computes in fp64 as
``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_HDR = os.path.join(_HERE, "moe_oracle.h")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` with gcc into ``libmoe_oracle.so`` (in-tree)."""
    stale = force or not os.path.exists(_LIB) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if stale:
        tmp = _LIB + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            L.oracle_version.restype = i32
            L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f64.restype = ctypes.c_double
            L.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
            L.oracle_f64_to_bf16.restype = ctypes.c_uint16
            L.oracle_bf16_to_f64_array.argtypes = [i64, P, P]
            L.oracle_f64_to_bf16_array.argtypes = [i64, P, P]
            L.oracle_router_logits.argtypes = [i32, i32, i32, P, P, P, P, P]
            L.oracle_select_topk.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
            L.oracle_select_topk.restype = i32
            L.oracle_expert_lists.argtypes = [i32, i32, i32, P, P, P, P]
            L.oracle_merge_topk.argtypes = [i32, i32, i32, P, P, P, P]
            L.oracle_add_rmsnorm.argtypes = [i32, i32, P, P, P, ctypes.c_double, P, P]
            L.oracle_merge_topk.restype = i32
            L.oracle_w8_gemv.argtypes = [i32, i32, i32, P, P, P, P]
            L.oracle_swiglu.argtypes = [i32, P, P, P]
            L.oracle_combine.argtypes = [i32, i32, P, P, P, ctypes.c_double, P, P]
            L.oracle_block_forward.argtypes = [P, P, P, P, i32, P, P, P, P, P, P,
                                               P, P, P, P, P, i32]
            L.oracle_block_forward.restype = i32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ bf16

def bf16_to_f64(b) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, np.float64)
    lib().oracle_bf16_to_f64_array(b.size, _p(b), _p(out))
    return out


def f64_to_bf16(v) -> np.ndarray:
    v = _c(v, np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_f64_to_bf16_array(v.size, _p(v), _p(out))
    return out


# ------------------------------------------------------------- the steps

def router_logits(x, w_router, w_gate=None):
    """A1: fp32 logits [T][E] (fp64 dot, rounded once) and gate logit [T]."""
    x = _c(x, np.uint16)
    w_router = _c(w_router, np.uint16)
    T, H = x.shape
    E = w_router.shape[0]
    logits = np.empty((T, E), np.float32)
    gate = np.zeros(T, np.float32)
    wg = None if w_gate is None else _c(w_gate, np.uint16)
    lib().oracle_router_logits(T, H, E, _p(x), _p(w_router), _p(wg), _p(logits),
                               _p(gate))
    return logits, (gate if wg is not None else None)


def select_topk(logits, gate_logit=None, K: int = 8):
    """A2: ids [T][K] int32, softmax weights [T][K] fp64, sigmoid gate [T]."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    sg = np.empty(T, np.float64)
    g = None if gate_logit is None else _c(gate_logit, np.float32)
    bad = lib().oracle_select_topk(T, E, K, E, _p(logits), _p(g), _p(ids), _p(w),
                                   _p(sg))
    return ids, w, sg, bad


def add_rmsnorm(resid_in, block, gamma, eps: float):
    """Residual add then RMS norm times gamma: resid_out = bf16(resid_in +
    block) and x_next = bf16(resid_out / sqrt(mean(resid_out^2) + eps) *
    gamma), per token.  resid_in [T][H] and gamma [H] are bf16 bits, block
    [T][H] the block's unrounded fp64 output.  Returns (resid_out, x_next)."""
    resid_in = _c(resid_in, np.uint16)
    block = _c(block, np.float64)
    gamma = _c(gamma, np.uint16)
    T, H = resid_in.shape
    assert block.shape == (T, H) and gamma.shape == (H,)
    r_out = np.empty((T, H), np.uint16)
    x_next = np.empty((T, H), np.uint16)
    lib().oracle_add_rmsnorm(T, H, _p(resid_in), _p(block), _p(gamma), float(eps), _p(r_out),
                             _p(x_next))
    return r_out, x_next


def candidates_topk(logits, K: int):
    """Wide top-k candidates: ids [T][K] int32 in rank order and their fp32
    values [T][K] (the row's entries at those ids); a non-finite row gets
    ids -1 and values 0.  Returns (ids, values, bad)."""
    logits = _c(logits, np.float32)
    T, N = logits.shape
    ids, _, _, bad = select_topk(logits, K=K)
    vals = np.zeros((T, K), np.float32)
    ok = ids[:, 0] >= 0
    vals[ok] = np.take_along_axis(logits[ok], ids[ok].astype(np.int64), axis=1)
    return ids, vals, bad


def merge_topk(ids, values, K: int):
    """Exact merge: ids/values [T][n_lists][K] candidate lists -> the K best
    pairs of each row's union, ids [T][K] int32, values [T][K] fp32."""
    ids = _c(ids, np.int32)
    values = _c(values, np.float32)
    T, n_lists, k_in = ids.shape
    assert k_in == K and values.shape == ids.shape
    out_i = np.empty((T, K), np.int32)
    out_v = np.empty((T, K), np.float32)
    bad = lib().oracle_merge_topk(T, n_lists, K, _p(ids), _p(values), _p(out_i), _p(out_v))
    return out_i, out_v, bad


def expert_lists(ids, E: int):
    """A3: counts [E], offsets [E+1], perm [n] (entries t*K+j by (e, t, j))."""
    ids = _c(ids, np.int32)
    T, K = ids.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.full(T * K, -1, np.int32)
    lib().oracle_expert_lists(T, E, K, _p(ids), _p(counts), _p(offsets), _p(perm))
    return counts, offsets, perm[: int(offsets[E])]


def w8_gemv(q, s, v, G: int = 128):
    """out[r] = sum_k q[r,k] * s[r,k//G] * v[k] in fp64."""
    q = _c(q, np.int8)
    s = _c(s, np.uint16)
    v = _c(v, np.uint16)
    R, C = q.shape
    out = np.empty(R, np.float64)
    lib().oracle_w8_gemv(R, C, G, _p(q), _p(s), _p(v), _p(out))
    return out


def swiglu(a):
    """A4 activation of a stacked [gate; up] pre-activation of length 2I."""
    a = _c(a, np.float64)
    I = a.shape[0] // 2
    h = np.empty(I, np.float64)
    hb = np.empty(I, np.uint16)
    lib().oracle_swiglu(I, _p(a), _p(h), _p(hb))
    return h, hb


def combine(y, w, ys=None, sg: float = 0.0):
    """A7 for one token: y [K][H] fp64, w [K] -> (out fp64 [H], out bf16 [H])."""
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    K, H = y.shape
    ysa = None if ys is None else _c(ys, np.float64)
    out = np.empty(H, np.float64)
    ob = np.empty(H, np.uint16)
    lib().oracle_combine(H, K, _p(y), _p(w), _p(ysa), float(sg), _p(out), _p(ob))
    return out, ob


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "E", "K", "I", "Is", "G")]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "w_gate", "w13_q", "w13_s", "w2_q", "w2_s",
        "ws13_q", "ws13_s", "ws2_q", "ws2_s")]


_WKEYS = {"w_router": np.uint16, "w_gate": np.uint16, "w13_q": np.int8,
          "w13_s": np.uint16, "w2_q": np.int8, "w2_s": np.uint16,
          "ws13_q": np.int8, "ws13_s": np.uint16, "ws2_q": np.int8,
          "ws2_s": np.uint16}


def block_forward(dims: dict, weights: dict, x, tokens=None, route_logits=None,
                  route_gate=None, nthreads: int = 1, want=("out",)):
    """A1..A7 for the given tokens (all if None).

    ``dims`` holds H, E, K, I, Is, G; ``weights`` holds the numpy arrays named
    like the C-ABI weight struct.  Returns a dict with the requested outputs
    (``out`` bf16 bits, ``out_f64``, ``ids``, ``weights``, ``sgate``,
    ``logits``, ``gate_logit``, ``y``, ``h``) indexed by token, plus ``bad``.
    """
    x = _c(x, np.uint16)
    T, H = x.shape
    K, E, I, Is = dims["K"], dims["E"], dims["I"], dims.get("Is", 0)
    d = _Dims(T, H, E, K, I, Is, dims.get("G", 128))
    keep = {k: (None if weights.get(k) is None else _c(weights[k], dt))
            for k, dt in _WKEYS.items()}
    w = _Weights(*[None if keep[k] is None else keep[k].ctypes.data
                   for k in _WKEYS])
    tok = None if tokens is None else _c(tokens, np.int32)
    n_tok = T if tok is None else tok.size
    rl = None if route_logits is None else _c(route_logits, np.float32)
    rg = None if route_gate is None else _c(route_gate, np.float32)
    Imax = max(I, Is)
    bufs = {
        "out": np.zeros((T, H), np.uint16),
        "out_f64": np.zeros((T, H), np.float64),
        "ids": np.full((T, K), -1, np.int32),
        "weights": np.zeros((T, K), np.float64),
        "sgate": np.zeros(T, np.float64),
        "logits": np.zeros((T, E), np.float32),
        "gate_logit": np.zeros(T, np.float32),
        "y": np.zeros((T, K + 1, H), np.float64) if "y" in want else None,
        "h": np.zeros((T, K + 1, Imax), np.uint16) if "h" in want else None,
    }
    bad = lib().oracle_block_forward(
        ctypes.byref(d), ctypes.byref(w), _p(x), _p(tok), n_tok, _p(rl), _p(rg),
        _p(bufs["out"]), _p(bufs["out_f64"]), _p(bufs["ids"]), _p(bufs["weights"]),
        _p(bufs["sgate"]), _p(bufs["logits"]), _p(bufs["gate_logit"]),
        _p(bufs["y"]), _p(bufs["h"]), int(nthreads))
    if bad < 0:
        raise ValueError("oracle_block_forward rejected its arguments")
    res = {k: v for k, v in bufs.items() if v is not None}
    res["bad"] = bad
    return res
