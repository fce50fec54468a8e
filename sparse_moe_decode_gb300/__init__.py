"""GB300 (sm_103a) sparse-MoE block: thin ctypes binding of libmoe_gb300.so.

Every step of the block runs in the library's CUDA kernels; this module only
marshals arguments (device pointers, sizes, the caller's CUDA stream) to the
C ABI declared in ``include/moe_gb300.h`` and turns a non-OK status into an
exception.  PyTorch is used for device memory and streams only.

The entry points keep the C names: ``moe_router_logits``,
``moe_select_top8``, ``moe_build_expert_lists``, ``moe_expert_swiglu_w8``,
``moe_combine``, ``moe_block_forward``, ``moe_block_forward_host``,
``moe_workspace_bytes``, ``moe_read_status``, ``moe_clear_status``.  Array
arguments may be torch tensors (their ``data_ptr()`` is passed), raw integer
addresses, or None where the C argument is nullable.

There is no CPU fallback: if the library is missing, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "MoEError", "lib", "Dims", "weights_struct", "moe_router_logits",
    "moe_select_top8", "moe_build_expert_lists", "moe_expert_swiglu_w8",
    "moe_combine", "moe_block_forward", "moe_block_forward_host",
    "moe_workspace_bytes", "moe_read_status", "moe_clear_status", "MoEBlock",
    "DEV_NONFINITE", "DEV_BAD_EXPERT", "DEV_TIMEOUT", "EXPORTS",
    "moe_block_forward_profiled", "moe_block_kernel_count", "moe_block_kernel_name",
    "moe_block_forward_noalloc", "moe_topk_workspace_bytes", "moe_topk_candidates",
    "moe_topk_merge", "moe_block_forward_residual",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = range(5)
DEV_NONFINITE, DEV_BAD_EXPERT, DEV_TIMEOUT = 0x1, 0x2, 0x4

# every symbol include/moe_gb300.h declares
EXPORTS = (
    "moe_workspace_bytes", "moe_router_logits", "moe_select_top8",
    "moe_build_expert_lists", "moe_expert_swiglu_w8", "moe_combine",
    "moe_block_forward", "moe_block_forward_host", "moe_read_status",
    "moe_clear_status", "moe_status_string", "moe_abi_version",
    "moe_block_forward_profiled", "moe_block_kernel_count", "moe_block_kernel_name",
    "moe_block_forward_noalloc", "moe_topk_workspace_bytes", "moe_topk_candidates",
    "moe_topk_merge", "moe_block_forward_residual",
)


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().moe_status_string(status).decode()
        super().__init__("%s: status %d (%s)" % (where, status, msg))


class Dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("expert_inter", ctypes.c_int32),
                ("shared_inter", ctypes.c_int32), ("group", ctypes.c_int32)]

    @classmethod
    def make(cls, hidden, expert_inter, shared_inter, num_experts=256, top_k=8, group=128):
        return cls(hidden, num_experts, top_k, expert_inter, shared_inter, group)


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_router", "w_shared_gate", "w13_q", "w13_s", "w2_q", "w2_s",
        "ws13_q", "ws13_s", "ws2_q", "ws2_s")]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libmoe_gb300.so is not built; run `python -c \"import "
                    "__graft_entry__ as g; g.build()\"` (no CPU fallback exists)")
            L = ctypes.CDLL(LIB_PATH)
            P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            DP = ctypes.POINTER(Dims)
            WP = ctypes.POINTER(Weights)
            sig = {
                "moe_workspace_bytes": (Z, [DP, I]),
                "moe_router_logits": (I, [DP, WP, P, I, P, P, P]),
                "moe_select_top8": (I, [P, I, I, I, P, P, P, P, P, Z, P]),
                "moe_build_expert_lists": (I, [P, I, I, P, P, P, P, Z, P]),
                "moe_expert_swiglu_w8": (I, [DP, WP, P, I, P, P, P, Z, P]),
                "moe_combine": (I, [DP, I, P, P, P, P, P]),
                "moe_block_forward": (I, [DP, WP, P, I, P, P, P, P, P, P, Z, P]),
                "moe_block_forward_host": (I, [DP, WP, P, I, P, P, Z, P]),
                "moe_read_status": (I, [P, P, ctypes.POINTER(ctypes.c_uint32)]),
                "moe_clear_status": (I, [P, P]),
                "moe_status_string": (ctypes.c_char_p, [I]),
                "moe_abi_version": (I, []),
                "moe_block_forward_profiled": (I, [DP, WP, P, I, P, P, Z,
                                                   ctypes.POINTER(P), I, P]),
                "moe_block_kernel_count": (I, [DP, I]),
                "moe_block_kernel_name": (ctypes.c_char_p, [DP, I, I]),
                "moe_block_forward_noalloc": (I, [DP, WP, P, I, P, P]),
                "moe_topk_workspace_bytes": (Z, [I, I]),
                "moe_topk_candidates": (I, [P, I, I, I, I, P, P, P, Z, P]),
                "moe_topk_merge": (I, [P, P, I, I, I, P, P, P, Z, P]),
                "moe_block_forward_residual": (I, [DP, WP, P, I, P, P, ctypes.c_float, P, P,
                                                   P, Z, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _a(v):
    """Address of a tensor / int / None as a ctypes argument."""
    if v is None:
        return None
    if isinstance(v, int):
        return v
    if hasattr(v, "data_ptr"):
        return v.data_ptr()
    if hasattr(v, "ctypes"):  # numpy array (host buffers)
        return v.ctypes.data
    raise TypeError("cannot pass %r as a pointer" % (type(v),))


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != MOE_OK:
        raise MoEError(st, where)


def weights_struct(w: dict) -> Weights:
    """A moe_weights struct from a dict of device tensors (or addresses).
    Keys follow the C struct; ``w_gate`` is accepted for ``w_shared_gate``."""
    gate = w.get("w_shared_gate", w.get("w_gate"))
    return Weights(_a(w.get("w_router")), _a(gate), _a(w.get("w13_q")), _a(w.get("w13_s")),
                   _a(w.get("w2_q")), _a(w.get("w2_s")), _a(w.get("ws13_q")),
                   _a(w.get("ws13_s")), _a(w.get("ws2_q")), _a(w.get("ws2_s")))


def moe_workspace_bytes(dims: Dims, T_max: int) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(dims), int(T_max)))


def moe_router_logits(dims, weights: Weights, x, T, logits, shared_gate_logit=None, stream=None):
    _check(lib().moe_router_logits(ctypes.byref(dims), ctypes.byref(weights), _a(x), int(T),
                                   _a(logits), _a(shared_gate_logit), _s(stream)),
           "moe_router_logits")


def moe_select_top8(logits, T, ld, E, shared_gate_logit, ids, weights, shared_gate,
                    workspace, ws_bytes, stream=None):
    _check(lib().moe_select_top8(_a(logits), int(T), int(ld), int(E), _a(shared_gate_logit),
                                 _a(ids), _a(weights), _a(shared_gate), _a(workspace),
                                 int(ws_bytes), _s(stream)), "moe_select_top8")


def moe_build_expert_lists(ids, T, E, counts, offsets, perm, workspace, ws_bytes, stream=None):
    _check(lib().moe_build_expert_lists(_a(ids), int(T), int(E), _a(counts), _a(offsets),
                                        _a(perm), _a(workspace), int(ws_bytes), _s(stream)),
           "moe_build_expert_lists")


def moe_expert_swiglu_w8(dims, weights: Weights, x, T, ids, y, workspace, ws_bytes, stream=None):
    _check(lib().moe_expert_swiglu_w8(ctypes.byref(dims), ctypes.byref(weights), _a(x), int(T),
                                      _a(ids), _a(y), _a(workspace), int(ws_bytes), _s(stream)),
           "moe_expert_swiglu_w8")


def moe_combine(dims, T, y, weights, shared_gate, out, stream=None):
    _check(lib().moe_combine(ctypes.byref(dims), int(T), _a(y), _a(weights), _a(shared_gate),
                             _a(out), _s(stream)), "moe_combine")


def moe_block_forward(dims, weights: Weights, x, T, out, ids_out=None, weights_out=None,
                      logits_out=None, gate_logit_out=None, workspace=None, ws_bytes=0,
                      stream=None):
    _check(lib().moe_block_forward(ctypes.byref(dims), ctypes.byref(weights), _a(x), int(T),
                                   _a(out), _a(ids_out), _a(weights_out), _a(logits_out),
                                   _a(gate_logit_out), _a(workspace), int(ws_bytes), _s(stream)),
           "moe_block_forward")


def moe_block_forward_residual(dims, weights: Weights, x, T, resid_in, gamma, eps, resid_out,
                               x_next, workspace, ws_bytes, stream=None):
    _check(lib().moe_block_forward_residual(ctypes.byref(dims), ctypes.byref(weights), _a(x),
                                            int(T), _a(resid_in), _a(gamma), float(eps),
                                            _a(resid_out), _a(x_next), _a(workspace),
                                            int(ws_bytes), _s(stream)),
           "moe_block_forward_residual")


def moe_block_forward_host(dims, weights: Weights, x_host, T, out_host, workspace, ws_bytes,
                           stream=None):
    _check(lib().moe_block_forward_host(ctypes.byref(dims), ctypes.byref(weights), _a(x_host),
                                        int(T), _a(out_host), _a(workspace), int(ws_bytes),
                                        _s(stream)), "moe_block_forward_host")


def moe_block_forward_profiled(dims, weights: Weights, x, T, out, workspace, ws_bytes, events,
                               stream=None):
    """``events``: torch.cuda.Event objects (timing enabled), at least
    1 + moe_block_kernel_count(dims, T) of them."""
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_block_forward_profiled(ctypes.byref(dims), ctypes.byref(weights), _a(x),
                                            int(T), _a(out), _a(workspace), int(ws_bytes), arr,
                                            len(events), _s(stream)),
           "moe_block_forward_profiled")


def moe_block_kernel_count(dims, T) -> int:
    return int(lib().moe_block_kernel_count(ctypes.byref(dims), int(T)))


def moe_block_kernel_name(dims, T, i) -> str:
    r = lib().moe_block_kernel_name(ctypes.byref(dims), int(T), int(i))
    return None if r is None else r.decode()


def moe_block_forward_noalloc(dims, weights: Weights, x, T, out, stream=None):
    """moe_block_forward with the library's fixed 4 MiB device scratch instead
    of a caller workspace (for callers that cannot allocate)."""
    _check(lib().moe_block_forward_noalloc(ctypes.byref(dims), ctypes.byref(weights), _a(x),
                                           int(T), _a(out), _s(stream)),
           "moe_block_forward_noalloc")


def moe_topk_workspace_bytes(T, N) -> int:
    return int(lib().moe_topk_workspace_bytes(int(T), int(N)))


def moe_topk_candidates(logits, T, ld, N, k, ids, values, workspace, ws_bytes, stream=None):
    _check(lib().moe_topk_candidates(_a(logits), int(T), int(ld), int(N), int(k), _a(ids),
                                     _a(values), _a(workspace), int(ws_bytes), _s(stream)),
           "moe_topk_candidates")


def moe_topk_merge(ids, values, T, n_lists, k, ids_out, values_out, workspace, ws_bytes,
                   stream=None):
    _check(lib().moe_topk_merge(_a(ids), _a(values), int(T), int(n_lists), int(k), _a(ids_out),
                                _a(values_out), _a(workspace), int(ws_bytes), _s(stream)),
           "moe_topk_merge")


def moe_read_status(workspace, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check(lib().moe_read_status(_a(workspace), _s(stream), ctypes.byref(bits)), "moe_read_status")
    return int(bits.value)


def moe_clear_status(workspace, stream=None):
    _check(lib().moe_clear_status(_a(workspace), _s(stream)), "moe_clear_status")


class MoEBlock:
    """Device-resident weights + a workspace sized for ``T_max`` tokens.

    ``weights`` is a dict of device tensors keyed like the C weight struct
    (bf16 tensors may be torch.bfloat16 or int16/uint16 views).  The block
    keeps references to them; ``forward(x)`` runs ``moe_block_forward`` on the
    current stream and returns the bf16 output tensor.
    """

    def __init__(self, hidden, expert_inter, shared_inter, weights: dict, T_max: int,
                 device="cuda"):
        import torch
        self.dims = Dims.make(hidden, expert_inter, shared_inter)
        self._keep = dict(weights)
        self.w = weights_struct(weights)
        self.ws_bytes = moe_workspace_bytes(self.dims, T_max)
        if self.ws_bytes == 0:
            raise MoEError(MOE_ERR_UNSUPPORTED, "moe_workspace_bytes")
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        self.T_max = T_max
        self.device = device

    def forward(self, x, out=None, ids=None, weights=None, logits=None, gate_logit=None,
                stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.dims.hidden), dtype=torch.bfloat16, device=x.device)
        moe_block_forward(self.dims, self.w, x, T, out, ids, weights, logits, gate_logit,
                          self.workspace, self.ws_bytes, stream)
        return out

    def status(self, stream=None) -> int:
        return moe_read_status(self.workspace, stream)

    def clear_status(self, stream=None):
        moe_clear_status(self.workspace, stream)
