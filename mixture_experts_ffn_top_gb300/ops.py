"""Python binding of libmoe_ffn.so (include/moe_ffn.h): argument marshalling only.

Every function here has the name of the C entry point it calls; tensors are
torch CUDA tensors (PyTorch provides device memory and streams), outputs are
allocated with torch when not given, and every step of the layer runs in the
library's CUDA kernels.  If the library is not built this module raises: there
is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ffn.so")
_lib = None

MOE_PATH_AUTO, MOE_PATH_MATVEC, MOE_PATH_TENSOR = 0, 1, 2
QK = 32

_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t

# name -> (restype, argtypes)
_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_abi_version": (_I, []),
    "moe_status_from_word": (_I, [_I]),
    "moe_weights_create": (_I, [ctypes.POINTER(_P), _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P]),
    "moe_weights_create_ex": (_I, [ctypes.POINTER(_P), _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P, _P]),
    "moe_weights_format": (_I, [_P]),
    "moe_weights_destroy": (_I, [_P]),
    "moe_weights_shape": (_I, [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "moe_weights_device_bytes": (_SZ, [_P]),
    "moe_weights_tensor_path": (_I, [_P]),
    "moe_ffn_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_workspace_init": (_I, [_P, _SZ, _P]),
    "moe_workspace_status": (_I, [_P, _I, _P]),
    "moe_router_topk": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_router_topk_noalloc": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_topk_from_logits": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_quantize_q8_1": (_I, [_P, _I64, _P, _P, _P]),
    "moe_bucket_workspace_size": (_SZ, [_I, _I, _I]),
    "moe_bucket": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_grouped_ffn_ex": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_expert_gate_up": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _P, _SZ, _P]),
    "moe_expert_down": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_debug_gate_up_block_dots": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_debug_down_block_dots": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_debug_bucket_barrier_timeout": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _SZ, _P]),
    "moe_debug_expert_wait_timeout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "moe_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_ffn_prefill": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _SZ, _P]),
    "moe_ffn_prefill_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_ffn_prefill_timed": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P, _P]),
    "moe_ffn_prefill_host": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_host_memory_addressable": (_I, [_P]),
    "moe_device_host_numa_node": (_I, [_P]),
    "moe_combine_residual": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_ffn_prefill_residual": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _SZ, _P]),
    "moe_combine_residual_rmsnorm": (_I, [_P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P]),
    "moe_rmsnorm": (_I, [_P, _P, ctypes.c_float, _I, _I, _P, _P]),
    "moe_ffn_prefill_stack_rmsnorm": (_I, [_P, _P, _P, _P, ctypes.c_float, _I, _P, _P, _I, _I, _I, _I, _P, _SZ, _P]),
    "moe_ffn_prefill_residual_rmsnorm": (_I, [_P, _P, _P, _P, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _I, _P,
                                               _SZ, _P]),
    "moe_workspace_views": (_I, [_P, _I, _I, _I, _I, _I, _I] + [ctypes.POINTER(_P)] * 10),
    "moe_ffn_prefill_stack": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _SZ, _P]),
}


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {moe_status_string(code)} ({code})")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m mixture_experts_ffn_top_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def moe_status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise MoeError(rc, where)


def _dev(t: torch.Tensor | None, dtype=None, name: str = "tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return _P(t.data_ptr())


def _stream(stream) -> _P:
    s = stream if stream is not None else torch.cuda.current_stream()
    return _P(s.cuda_stream)


# --------------------------------------------------------------- weights ---
WEIGHT_FORMATS = {"q8_0": 0, "q4_k": 1, "q3_k": 2}  # MOE_WFMT_*


class MoeWeights:
    """Library-owned expert weights (moe_weights_create / moe_weights_destroy)."""

    def __init__(self, gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor, E: int, D: int, F: int,
                 sh_gate: torch.Tensor | None = None, sh_up: torch.Tensor | None = None,
                 sh_down: torch.Tensor | None = None, Fs: int = 0, stream=None, wfmt: str = "q8_0"):
        self.handle = _P()
        self.E, self.D, self.F, self.Fs = E, D, F, Fs
        self.wfmt = wfmt
        if wfmt not in WEIGHT_FORMATS:
            raise ValueError(f"unknown weight format {wfmt!r}")
        rc = lib().moe_weights_create_ex(ctypes.byref(self.handle), WEIGHT_FORMATS[wfmt], E, D, F,
                                         _dev(gate, torch.uint8, "gate"), _dev(up, torch.uint8, "up"),
                                         _dev(down, torch.uint8, "down"), Fs, _dev(sh_gate, torch.uint8, "sh_gate"),
                                         _dev(sh_up, torch.uint8, "sh_up"), _dev(sh_down, torch.uint8, "sh_down"),
                                         _stream(stream))
        _check(rc, "moe_weights_create_ex")

    @property
    def device_bytes(self) -> int:
        return int(lib().moe_weights_device_bytes(self.handle))

    def close(self) -> None:
        if self.handle is not None and self.handle.value:
            lib().moe_weights_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_weights_tensor_path(w: MoeWeights) -> bool:
    return bool(lib().moe_weights_tensor_path(w.handle))


tensor_path_available = moe_weights_tensor_path


def moe_weights_create(E, D, F, gate, up, down, Fs=0, sh_gate=None, sh_up=None, sh_down=None, stream=None,
                       wfmt="q8_0"):
    return MoeWeights(gate, up, down, E, D, F, sh_gate, sh_up, sh_down, Fs, stream, wfmt)


def moe_weights_format(w: MoeWeights) -> str:
    code = int(lib().moe_weights_format(w.handle))
    return {v: k for k, v in WEIGHT_FORMATS.items()}[code]


def moe_weights_destroy(w: MoeWeights) -> None:
    w.close()


# ------------------------------------------------------------- workspace ---
def moe_ffn_workspace_size(N, D, E, F, top_k, Fs=0) -> int:
    n = int(lib().moe_ffn_workspace_size(N, D, E, F, top_k, Fs))
    if n == 0:
        raise MoeError(-2, "moe_ffn_workspace_size")
    return n


def new_workspace(N, D, E, F, top_k, Fs=0, device="cuda", stream=None) -> torch.Tensor:
    ws = torch.empty(moe_ffn_workspace_size(N, D, E, F, top_k, Fs), dtype=torch.uint8, device=device)
    moe_workspace_init(ws, stream)
    return ws


def moe_workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(lib().moe_workspace_init(_dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "moe_workspace_init")


def moe_workspace_status(ws: torch.Tensor, clear: bool = True, stream=None) -> int:
    """Device status word (MOE_DEV_* bits); synchronises the stream."""
    rc = lib().moe_workspace_status(_dev(ws, torch.uint8, "ws"), int(clear), _stream(stream))
    if rc < 0:
        raise MoeError(rc, "moe_workspace_status")
    return rc


# ------------------------------------------------------------------ steps ---
def moe_router_topk(hidden, routerW, shexp_gate, top_k, norm_topk_prob, ws, want_logits=False, stream=None):
    """-> dict(topk_idx, topk_w, shexp_scale, x_q, x_d, logits)."""
    N, D = hidden.shape
    E = routerW.shape[0]
    dev = hidden.device
    r = dict(topk_idx=torch.empty((N, top_k), dtype=torch.int32, device=dev),
             topk_w=torch.empty((N, top_k), dtype=torch.float32, device=dev),
             shexp_scale=torch.empty(N, dtype=torch.float32, device=dev) if shexp_gate is not None else None,
             x_q=torch.empty((N, D), dtype=torch.int8, device=dev),
             x_d=torch.empty((N, D // QK), dtype=torch.float32, device=dev),
             logits=torch.empty((N, E), dtype=torch.float32, device=dev) if want_logits else None)
    rc = lib().moe_router_topk(_dev(hidden, torch.float32, "hidden"), _dev(routerW, torch.float32, "routerW"),
                               _dev(shexp_gate, torch.float32, "shexp_gate"), N, D, E, top_k, int(norm_topk_prob),
                               _dev(r["topk_idx"]), _dev(r["topk_w"]), _dev(r["shexp_scale"]), _dev(r["x_q"]),
                               _dev(r["x_d"]), _dev(r["logits"]), _dev(ws, torch.uint8, "ws"), ws.numel(),
                               _stream(stream))
    _check(rc, "moe_router_topk")
    return r


def moe_router_topk_noalloc(hidden, routerW, shexp_gate, top_k, norm_topk_prob, want_logits=False, stream=None,
                            outputs=None):
    """moe_router_topk without a workspace (the library's fixed scratch); outputs as moe_router_topk
    (written into `outputs`, a dict of those tensors, when given)."""
    N, D = hidden.shape
    E = routerW.shape[0]
    dev = hidden.device
    r = outputs if outputs is not None else dict(topk_idx=torch.empty((N, top_k), dtype=torch.int32, device=dev),
             topk_w=torch.empty((N, top_k), dtype=torch.float32, device=dev),
             shexp_scale=torch.empty(N, dtype=torch.float32, device=dev) if shexp_gate is not None else None,
             x_q=torch.empty((N, D), dtype=torch.int8, device=dev),
             x_d=torch.empty((N, D // QK), dtype=torch.float32, device=dev),
             logits=torch.empty((N, E), dtype=torch.float32, device=dev) if want_logits else None)
    rc = lib().moe_router_topk_noalloc(_dev(hidden, torch.float32, "hidden"), _dev(routerW, torch.float32, "routerW"),
                                       _dev(shexp_gate, torch.float32, "shexp_gate"), N, D, E, top_k,
                                       int(norm_topk_prob), _dev(r["topk_idx"]), _dev(r["topk_w"]),
                                       _dev(r["shexp_scale"]), _dev(r["x_q"]), _dev(r["x_d"]), _dev(r["logits"]),
                                       _stream(stream))
    _check(rc, "moe_router_topk_noalloc")
    return r


def moe_topk_from_logits(logits, top_k, norm_topk_prob, stream=None):
    N, E = logits.shape
    idx = torch.empty((N, top_k), dtype=torch.int32, device=logits.device)
    w = torch.empty((N, top_k), dtype=torch.float32, device=logits.device)
    _check(lib().moe_topk_from_logits(_dev(logits, torch.float32, "logits"), N, E, top_k, int(norm_topk_prob),
                                      _dev(idx), _dev(w), _stream(stream)), "moe_topk_from_logits")
    return idx, w


def moe_quantize_q8_1(x, stream=None):
    assert x.numel() % QK == 0
    q = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    d = torch.empty(x.shape[:-1] + (x.shape[-1] // QK,), dtype=torch.float32, device=x.device)
    _check(lib().moe_quantize_q8_1(_dev(x, torch.float32, "x"), x.numel() // QK, _dev(q), _dev(d), _stream(stream)),
           "moe_quantize_q8_1")
    return q, d


def moe_bucket(topk_idx, E, ws, stream=None):
    N, k = topk_idx.shape
    dev = topk_idx.device
    es = torch.empty(E + 1, dtype=torch.int32, device=dev)
    ti = torch.empty(N * k, dtype=torch.int32, device=dev)
    tk = torch.empty(N * k, dtype=torch.int32, device=dev)
    _check(lib().moe_bucket(_dev(topk_idx, torch.int32, "topk_idx"), N, k, E, _dev(es), _dev(ti), _dev(tk),
                            _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)), "moe_bucket")
    return es, ti, tk


def moe_debug_bucket_barrier_timeout(topk_idx, E, limit_ms, ws, stream=None):
    """moe_bucket with a grid barrier that cannot complete (bounded by limit_ms); the outcome is
    read with moe_workspace_status."""
    N, k = topk_idx.shape
    dev = topk_idx.device
    es = torch.full((E + 1,), -7, dtype=torch.int32, device=dev)
    ti = torch.full((N * k,), -7, dtype=torch.int32, device=dev)
    tk = torch.full((N * k,), -7, dtype=torch.int32, device=dev)
    _check(lib().moe_debug_bucket_barrier_timeout(_dev(topk_idx, torch.int32, "topk_idx"), N, k, E, _dev(es),
                                                  _dev(ti), _dev(tk), int(limit_ms), _dev(ws, torch.uint8, "ws"),
                                                  ws.numel(), _stream(stream)), "moe_debug_bucket_barrier_timeout")
    return es, ti, tk


def moe_grouped_ffn(w: MoeWeights, x_q, x_d, expStart, expTokI, expTokK, top_k, ws, shexp_scale=None,
                    path=MOE_PATH_AUTO, stream=None):
    """-> (partials [N*top_k, D], shared_out [N, D] or None)."""
    N = x_q.shape[0]
    dev = x_q.device
    partials = torch.empty((N * top_k, w.D), dtype=torch.float32, device=dev)
    shared = torch.empty((N, w.D), dtype=torch.float32, device=dev) if shexp_scale is not None else None
    rc = lib().moe_grouped_ffn_ex(w.handle, _dev(x_q, torch.int8, "x_q"), _dev(x_d, torch.float32, "x_d"),
                                  _dev(expStart, torch.int32), _dev(expTokI, torch.int32), _dev(expTokK, torch.int32),
                                  N, top_k, _dev(shexp_scale, torch.float32), _dev(partials), _dev(shared), path,
                                  _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check(rc, "moe_grouped_ffn")
    return partials, shared


def moe_expert_gate_up(w: MoeWeights, x_q, x_d, expStart, expTokI, top_k, ws, path=MOE_PATH_AUTO, stream=None):
    N = x_q.shape[0]
    h_q = torch.zeros((N * top_k, w.F), dtype=torch.int8, device=x_q.device)
    h_d = torch.zeros((N * top_k, w.F // QK), dtype=torch.float32, device=x_q.device)
    rc = lib().moe_expert_gate_up(w.handle, _dev(x_q, torch.int8), _dev(x_d, torch.float32),
                                  _dev(expStart, torch.int32), _dev(expTokI, torch.int32), N, top_k, _dev(h_q),
                                  _dev(h_d), path, _dev(ws, torch.uint8), ws.numel(), _stream(stream))
    _check(rc, "moe_expert_gate_up")
    return h_q, h_d


def moe_expert_down(w: MoeWeights, h_q, h_d, expStart, expTokI, expTokK, N, top_k, ws, path=MOE_PATH_AUTO,
                    stream=None):
    partials = torch.zeros((N * top_k, w.D), dtype=torch.float32, device=h_q.device)
    rc = lib().moe_expert_down(w.handle, _dev(h_q, torch.int8), _dev(h_d, torch.float32),
                               _dev(expStart, torch.int32), _dev(expTokI, torch.int32), _dev(expTokK, torch.int32),
                               N, top_k, _dev(partials), path, _dev(ws, torch.uint8), ws.numel(), _stream(stream))
    _check(rc, "moe_expert_down")
    return partials


def moe_debug_gate_up_block_dots(w: MoeWeights, x_q, x_d, expStart, expTokI, top_k, block, ws,
                                 path=MOE_PATH_AUTO, stream=None):
    N = x_q.shape[0]
    dots = torch.zeros((N * top_k, 2, w.F), dtype=torch.int32, device=x_q.device)
    rc = lib().moe_debug_gate_up_block_dots(w.handle, _dev(x_q, torch.int8), _dev(x_d, torch.float32),
                                            _dev(expStart, torch.int32), _dev(expTokI, torch.int32), N, top_k, block,
                                            _dev(dots), path, _dev(ws, torch.uint8), ws.numel(), _stream(stream))
    _check(rc, "moe_debug_gate_up_block_dots")
    return dots


def moe_debug_down_block_dots(w: MoeWeights, h_q, h_d, expStart, expTokI, expTokK, N, top_k, block, ws,
                              path=MOE_PATH_AUTO, stream=None):
    """int32 dots of the down GEMM's block `block` for every CSR entry and output column:
    [N * top_k, D] (entries beyond expStart[E] stay zero)."""
    dots = torch.zeros((N * top_k, w.D), dtype=torch.int32, device=h_q.device)
    rc = lib().moe_debug_down_block_dots(w.handle, _dev(h_q, torch.int8), _dev(h_d, torch.float32),
                                         _dev(expStart, torch.int32), _dev(expTokI, torch.int32),
                                         _dev(expTokK, torch.int32), N, top_k, block, _dev(dots), path,
                                         _dev(ws, torch.uint8), ws.numel(), _stream(stream))
    _check(rc, "moe_debug_down_block_dots")
    return dots


def moe_debug_expert_wait_timeout(w: MoeWeights, x_q, x_d, expStart, expTokI, top_k, limit_ms, ws, stream=None):
    N = x_q.shape[0]
    rc = lib().moe_debug_expert_wait_timeout(w.handle, _dev(x_q, torch.int8), _dev(x_d, torch.float32),
                                             _dev(expStart, torch.int32), _dev(expTokI, torch.int32), N, top_k,
                                             int(limit_ms), _dev(ws, torch.uint8), ws.numel(), _stream(stream))
    _check(rc, "moe_debug_expert_wait_timeout")


def moe_combine(partials, topk_w, shared=None, out=None, stream=None):
    N, k = topk_w.shape
    D = partials.shape[1]
    if out is None:
        out = torch.empty((N, D), dtype=torch.float32, device=partials.device)
    _check(lib().moe_combine(_dev(partials, torch.float32, "partials"), _dev(topk_w, torch.float32, "topk_w"),
                             _dev(shared, torch.float32, "shared"), N, k, D, _dev(out, torch.float32, "out"),
                             _stream(stream)), "moe_combine")
    return out


def moe_combine_residual(partials, topk_w, shared, residual, out=None, stream=None):
    """moe_combine, then + residual (the per-layer combine's residual add).  out may be residual."""
    N, k = topk_w.shape
    D = partials.shape[1]
    if out is None:
        out = torch.empty((N, D), dtype=torch.float32, device=partials.device)
    _check(lib().moe_combine_residual(_dev(partials, torch.float32, "partials"), _dev(topk_w, torch.float32, "topk_w"),
                                      _dev(shared, torch.float32, "shared"), _dev(residual, torch.float32, "residual"),
                                      N, k, D, _dev(out, torch.float32, "out"), _stream(stream)), "moe_combine_residual")
    return out


def moe_combine_residual_rmsnorm(partials, topk_w, shared, residual, gamma, eps, out=None, normed=None,
                                 stream=None):
    """moe_combine_residual, then RMSNorm of each output row with weight gamma and eps (the next
    layer's input).  Returns (out, normed); out may be residual."""
    N, k = topk_w.shape
    D = partials.shape[1]
    if out is None:
        out = torch.empty((N, D), dtype=torch.float32, device=partials.device)
    if normed is None:
        normed = torch.empty((N, D), dtype=torch.float32, device=partials.device)
    _check(lib().moe_combine_residual_rmsnorm(_dev(partials, torch.float32, "partials"),
                                              _dev(topk_w, torch.float32, "topk_w"), _dev(shared, torch.float32, "shared"),
                                              _dev(residual, torch.float32, "residual"),
                                              _dev(gamma, torch.float32, "gamma"), float(eps), N, k, D,
                                              _dev(out, torch.float32, "out"), _dev(normed, torch.float32, "normed"),
                                              _stream(stream)), "moe_combine_residual_rmsnorm")
    return out, normed


def moe_rmsnorm(x, gamma, eps, normed=None, stream=None):
    """normed = RMSNorm(x) * gamma (rows of x, weight gamma [D], eps)."""
    N, D = x.shape
    if normed is None:
        normed = torch.empty((N, D), dtype=torch.float32, device=x.device)
    _check(lib().moe_rmsnorm(_dev(x, torch.float32, "x"), _dev(gamma, torch.float32, "gamma"), float(eps), N, D,
                             _dev(normed, torch.float32, "normed"), _stream(stream)), "moe_rmsnorm")
    return normed


def moe_ffn_prefill_stack_rmsnorm(weights, routerWs, shexp_gates, gammas, eps, hidden, top_k, norm_topk_prob, ws,
                                  normed=None, path=MOE_PATH_AUTO, stream=None):
    """Pre-norm layers in place: normed = RMSNorm_0(hidden); per layer l hidden += FFN_l(normed) and
    normed = RMSNorm_{l+1}(hidden) (gammas: n + 1 entries, the last may be None).  Returns
    (hidden, normed)."""
    n = len(weights)
    assert len(routerWs) == n and len(shexp_gates) == n and len(gammas) == n + 1
    N, D = hidden.shape
    if normed is None:
        normed = torch.empty((N, D), dtype=torch.float32, device=hidden.device)
    wh = (_P * n)(*[w.handle for w in weights])
    rw = (_P * n)(*[_dev(r, torch.float32, "routerW") for r in routerWs])
    sg = None
    if any(g is not None for g in shexp_gates):
        sg = (_P * n)(*[_dev(g, torch.float32) for g in shexp_gates])
    gm = (_P * (n + 1))(*[_dev(g, torch.float32) for g in gammas])
    rc = lib().moe_ffn_prefill_stack_rmsnorm(ctypes.cast(wh, _P), ctypes.cast(rw, _P),
                                             None if sg is None else ctypes.cast(sg, _P), ctypes.cast(gm, _P),
                                             float(eps), n, _dev(hidden, torch.float32, "hidden"),
                                             _dev(normed, torch.float32, "normed"), N, top_k, int(norm_topk_prob), path,
                                             _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check(rc, "moe_ffn_prefill_stack_rmsnorm")
    return hidden, normed


def moe_ffn_prefill_stack(weights, routerWs, shexp_gates, hidden, top_k, norm_topk_prob, ws, path=MOE_PATH_AUTO,
                          stream=None):
    """Layers applied in place, hidden <- hidden + FFN_l(hidden) for each layer l in order (weights,
    routerWs, shexp_gates: one entry per layer; shexp_gates entries may be None)."""
    n = len(weights)
    assert len(routerWs) == n and len(shexp_gates) == n
    N = hidden.shape[0]
    wh = (_P * n)(*[w.handle for w in weights])
    rw = (_P * n)(*[_dev(r, torch.float32, "routerW") for r in routerWs])
    sg = None
    if any(g is not None for g in shexp_gates):
        sg = (_P * n)(*[_dev(g, torch.float32) for g in shexp_gates])
    rc = lib().moe_ffn_prefill_stack(ctypes.cast(wh, _P), ctypes.cast(rw, _P), None if sg is None else ctypes.cast(sg, _P),
                                     n, _dev(hidden, torch.float32, "hidden"), N, top_k, int(norm_topk_prob), path,
                                     _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check(rc, "moe_ffn_prefill_stack")
    return hidden


def moe_ffn_prefill_residual(w: MoeWeights, hidden, routerW, shexp_gate, residual, top_k, norm_topk_prob, ws,
                             out=None, path=MOE_PATH_AUTO, stream=None):
    """The layer with the residual add fused into its combine: out = residual + FFN(hidden)."""
    N = hidden.shape[0]
    if out is None:
        out = torch.empty((N, w.D), dtype=torch.float32, device=hidden.device)
    rc = lib().moe_ffn_prefill_residual(w.handle, _dev(hidden, torch.float32, "hidden"),
                                        _dev(routerW, torch.float32, "routerW"), _dev(shexp_gate, torch.float32),
                                        _dev(residual, torch.float32, "residual"), N, top_k, int(norm_topk_prob),
                                        _dev(out, torch.float32, "out"), path, _dev(ws, torch.uint8, "ws"), ws.numel(),
                                        _stream(stream))
    _check(rc, "moe_ffn_prefill_residual")
    return out


def moe_ffn_prefill_residual_rmsnorm(w: MoeWeights, hidden, routerW, shexp_gate, residual, gamma, eps, top_k,
                                     norm_topk_prob, ws, out=None, normed=None, path=MOE_PATH_AUTO, stream=None):
    """The layer with the residual add and the next layer's RMSNorm fused into its combine:
    out = residual + FFN(hidden), normed = RMSNorm(out) * gamma.  Returns (out, normed)."""
    N = hidden.shape[0]
    if out is None:
        out = torch.empty((N, w.D), dtype=torch.float32, device=hidden.device)
    if normed is None:
        normed = torch.empty((N, w.D), dtype=torch.float32, device=hidden.device)
    rc = lib().moe_ffn_prefill_residual_rmsnorm(w.handle, _dev(hidden, torch.float32, "hidden"),
                                                _dev(routerW, torch.float32, "routerW"), _dev(shexp_gate, torch.float32),
                                                _dev(residual, torch.float32, "residual"),
                                                _dev(gamma, torch.float32, "gamma"), float(eps), N, top_k,
                                                int(norm_topk_prob), _dev(out, torch.float32, "out"),
                                                _dev(normed, torch.float32, "normed"), path, _dev(ws, torch.uint8, "ws"),
                                                ws.numel(), _stream(stream))
    _check(rc, "moe_ffn_prefill_residual_rmsnorm")
    return out, normed


def moe_ffn_prefill(w: MoeWeights, hidden, routerW, shexp_gate, top_k, norm_topk_prob, ws, out=None,
                    path=MOE_PATH_AUTO, stream=None):
    N = hidden.shape[0]
    if out is None:
        out = torch.empty((N, w.D), dtype=torch.float32, device=hidden.device)
    rc = lib().moe_ffn_prefill_ex(w.handle, _dev(hidden, torch.float32, "hidden"),
                                  _dev(routerW, torch.float32, "routerW"), _dev(shexp_gate, torch.float32),
                                  N, top_k, int(norm_topk_prob), _dev(out, torch.float32, "out"), path,
                                  _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check(rc, "moe_ffn_prefill")
    return out


def _host(t: torch.Tensor, name: str):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous() or t.dtype != torch.float32:
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    return _P(t.data_ptr())


def moe_device_host_numa_node() -> int:
    """Host NUMA node closest to the current device, or -1 (no NUMA placement reported)."""
    node = ctypes.c_int(-1)
    _check(lib().moe_device_host_numa_node(ctypes.byref(node)), "moe_device_host_numa_node")
    return node.value


def moe_host_memory_addressable(t: torch.Tensor) -> bool:
    """Whether the tensor's memory can be passed to moe_ffn_prefill_host (host memory the device reaches)."""
    return bool(lib().moe_host_memory_addressable(_P(t.data_ptr())))


def moe_ffn_prefill_host(w: MoeWeights, hidden_host, routerW, shexp_gate, top_k, norm_topk_prob, ws, out_host,
                         path=MOE_PATH_AUTO, stream=None):
    """moe_ffn_prefill with hidden and the output in host memory (pinned, or pageable where the device
    walks the host page tables): the kernels read and write them in place.  Asynchronous: out_host is
    complete once `stream` is."""
    N = hidden_host.shape[0]
    if tuple(out_host.shape) != (N, w.D):
        raise ValueError("out_host must be [N, D]")
    rc = lib().moe_ffn_prefill_host(w.handle, _host(hidden_host, "hidden_host"),
                                    _dev(routerW, torch.float32, "routerW"), _dev(shexp_gate, torch.float32),
                                    N, top_k, int(norm_topk_prob), _host(out_host, "out_host"), path,
                                    _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    _check(rc, "moe_ffn_prefill_host")
    return out_host


PREFILL_STAGES = ["router", "bucket", "gather", "gate_up", "down", "combine"]


def moe_ffn_prefill_timed(w: MoeWeights, hidden, routerW, shexp_gate, top_k, norm_topk_prob, ws, events, out=None,
                          path=MOE_PATH_AUTO, stream=None):
    """moe_ffn_prefill recording 7 torch.cuda.Event objects between its stages (see PREFILL_STAGES)."""
    N = hidden.shape[0]
    if out is None:
        out = torch.empty((N, w.D), dtype=torch.float32, device=hidden.device)
    for e in events:
        if e.cuda_event == 0:
            e.record()  # creates the underlying CUDA event
    arr = (_P * 7)(*[_P(e.cuda_event) for e in events])
    rc = lib().moe_ffn_prefill_timed(w.handle, _dev(hidden, torch.float32, "hidden"),
                                     _dev(routerW, torch.float32, "routerW"), _dev(shexp_gate, torch.float32),
                                     N, top_k, int(norm_topk_prob), _dev(out, torch.float32, "out"), path,
                                     _dev(ws, torch.uint8, "ws"), ws.numel(), _stream(stream), arr)
    _check(rc, "moe_ffn_prefill_timed")
    return out


def moe_workspace_views(ws, N, D, E, F, top_k, Fs=0):
    """Device addresses of moe_ffn_prefill's intermediates inside ws, as torch views."""
    ptrs = [_P() for _ in range(10)]
    _check(lib().moe_workspace_views(_dev(ws, torch.uint8), N, D, E, F, top_k, Fs,
                                     *[ctypes.byref(p) for p in ptrs]), "moe_workspace_views")
    base = ws.data_ptr()
    names = ["topk_idx", "topk_w", "shexp_scale", "x_q", "x_d", "expStart", "expTokI", "expTokK", "partials",
             "shared_out"]
    shapes = [((N, top_k), torch.int32), ((N, top_k), torch.float32), ((N,), torch.float32), ((N, D), torch.int8),
              ((N, D // QK), torch.float32), ((E + 1,), torch.int32), ((N * top_k,), torch.int32),
              ((N * top_k,), torch.int32), ((N * top_k, D), torch.float32), ((N, D), torch.float32)]
    out = {}
    for name, p, (shape, dt) in zip(names, ptrs, shapes):
        if not p.value:
            out[name] = None
            continue
        off = p.value - base
        nbytes = int(torch.tensor([], dtype=dt).element_size()) * int(torch.Size(shape).numel())
        out[name] = ws[off:off + nbytes].view(dt).view(shape)
    return out


# ------------------------------------------------------------------ layer ---
class MoeLayer:
    """One routed-MoE FFN layer resident on a GPU: weights handle, router, workspace."""

    def __init__(self, weights: MoeWeights, routerW: torch.Tensor, shexp_gate: torch.Tensor | None,
                 max_tokens: int, top_k: int):
        self.w = weights
        self.routerW = routerW
        self.shexp_gate = shexp_gate
        self.top_k = top_k
        self.max_tokens = max_tokens
        self.ws = new_workspace(max_tokens, weights.D, weights.E, weights.F, top_k, weights.Fs,
                                device=routerW.device)

    @classmethod
    def from_numpy(cls, inp: dict, device="cuda", top_k: int | None = None, max_tokens: int | None = None):
        """Upload a workloads.make_inputs dict."""
        dev = torch.device(device)
        E, F = inp["gate"].shape[0], inp["gate"].shape[1]
        D = inp["down"].shape[1]
        Fs = 0 if inp.get("sh_gate") is None else inp["sh_gate"].shape[0]

        def up(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            return torch.from_numpy(a if a.flags.writeable else a.copy()).to(dev)

        w = MoeWeights(up(inp["gate"]), up(inp["up"]), up(inp["down"]), E, D, F, up(inp.get("sh_gate")),
                       up(inp.get("sh_up")), up(inp.get("sh_down")), Fs, wfmt=inp.get("wfmt", "q8_0"))
        k = top_k if top_k is not None else min(8, E)
        N = max_tokens if max_tokens is not None else inp["hidden"].shape[0]
        return cls(w, up(inp["routerW"]), up(inp.get("shexp_gate")), N, k)

    def prefill(self, hidden: torch.Tensor, top_k: int | None = None, norm_topk_prob: bool = False, out=None,
                path=MOE_PATH_AUTO, stream=None):
        k = self.top_k if top_k is None else top_k
        if hidden.shape[0] > self.max_tokens or k != self.top_k:
            self.max_tokens = max(self.max_tokens, hidden.shape[0])
            self.top_k = k
            self.ws = new_workspace(self.max_tokens, self.w.D, self.w.E, self.w.F, k, self.w.Fs, device=hidden.device)
        return moe_ffn_prefill(self.w, hidden, self.routerW, self.shexp_gate, k, norm_topk_prob, self.ws, out, path,
                               stream)

    def status(self, clear: bool = True) -> int:
        return moe_workspace_status(self.ws, clear)

    def views(self, N: int):
        return moe_workspace_views(self.ws, N, self.w.D, self.w.E, self.w.F, self.top_k, self.w.Fs)
