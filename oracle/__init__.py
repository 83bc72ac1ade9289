"""CPU oracle for the batched routed-MoE FFN -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
(the ``cpu_baseline`` leg and ``--impl reference``) may import this package.
The product path (``mixture_experts_ffn_top_gb300``) never imports it and
shares no code with it; ``moe_oracle.c`` is plain C built with gcc.

This module is argument marshalling around ``moe_oracle.c`` (numpy <->
ctypes) plus ``moe_ffn``, which chains the oracle's steps in the order the
pages give: router -> softmax/top-k -> Q8_1 of x -> CSR bucketing ->
grouped gate/up/down -> (shared expert) -> combine.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

QK = 32
Q8_0_BYTES = 34  # fp16 scale + 32 int8 quants
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_half_to_float.restype = ctypes.c_float
            lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
            lib.oracle_float_to_half.restype = ctypes.c_uint16
            lib.oracle_float_to_half.argtypes = [ctypes.c_float]
            lib.oracle_bucket.restype = _I
            lib.oracle_num_threads.restype = _I
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(_P)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return int(_L().oracle_num_threads())


# ---------------------------------------------------------------- fp16 ----
def half_to_float(h: np.ndarray) -> np.ndarray:
    lib = _L()
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib.oracle_half_to_float(int(v)) for v in h], dtype=np.float32)


def float_to_half(f: np.ndarray) -> np.ndarray:
    lib = _L()
    f = np.asarray(f, dtype=np.float32).ravel()
    return np.array([lib.oracle_float_to_half(float(v)) for v in f], dtype=np.uint16)


def halves(h: np.ndarray) -> np.ndarray:
    """Fast fp16 bits -> fp32 for large arrays (numpy's conversion is exact)."""
    return np.asarray(h, dtype=np.uint16).view(np.float16).astype(np.float32)


# ---------------------------------------------------------------- steps ---
def quantize_q8_1(x: np.ndarray):
    """Q8_1 of a float array whose last dim is a multiple of 32 -> (q int8, d16 u16, s16 u16)."""
    x = _f32(x)
    assert x.shape[-1] % QK == 0
    nblk = x.size // QK
    q = np.empty(x.shape, np.int8)
    d16 = np.empty(x.shape[:-1] + (x.shape[-1] // QK,), np.uint16)
    s16 = np.empty_like(d16)
    _L().oracle_quantize_q8_1(_p(x), _I64(nblk), _p(q), _p(d16), _p(s16))
    return q, d16, s16


def router_logits(x: np.ndarray, W: np.ndarray) -> np.ndarray:
    x, W = _f32(x), _f32(W)
    N, D = x.shape
    E = W.shape[0]
    out = np.empty((N, E), np.float32)
    _L().oracle_router_logits(_p(x), _p(W), _I64(N), _I(D), _I(E), _p(out))
    return out


def softmax_topk(logits: np.ndarray, k: int, norm: bool):
    logits = _f32(logits)
    N, E = logits.shape
    idx = np.empty((N, k), np.int32)
    w = np.empty((N, k), np.float32)
    p = np.empty((N, E), np.float32)
    _L().oracle_softmax_topk(_p(logits), _I64(N), _I(E), _I(k), _I(int(norm)), _p(idx), _p(w), _p(p))
    return idx, w, p


def sigmoid(g: np.ndarray) -> np.ndarray:
    g = _f32(g).ravel()
    s = np.empty_like(g)
    _L().oracle_sigmoid(_p(g), _I64(g.size), _p(s))
    return s


def bucket(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, k = idx.shape
    expStart = np.empty(E + 1, np.int32)
    expTokI = np.empty(N * k, np.int32)
    expTokK = np.empty(N * k, np.int32)
    rc = _L().oracle_bucket(_p(idx), _I64(N), _I(k), _I(E), _p(expStart), _p(expTokI), _p(expTokK))
    if rc != 0:
        raise ValueError({-1: "expert index out of range", -2: "token selects an expert twice"}[rc])
    return expStart, expTokI, expTokK


def block_dots(w_row: np.ndarray, aq: np.ndarray) -> np.ndarray:
    w_row = np.ascontiguousarray(w_row, dtype=np.uint8)
    aq = np.ascontiguousarray(aq, dtype=np.int8)
    nblk = aq.size // QK
    out = np.empty(nblk, np.int32)
    _L().oracle_block_dots(_p(w_row), _p(aq), _I(nblk), _p(out))
    return out


def block_dots_csr(W: np.ndarray, act: np.ndarray, expStart: np.ndarray, sel: np.ndarray | None,
                   block: int) -> np.ndarray:
    """int32 dots of one 32-wide block for every CSR entry and every weight row of its expert
    (Q8_0 weights W [E][rows][K/32 blocks of 34 bytes]): out[j, r].  The activation row of entry
    j is act[sel[j]] (token rows of x_q, sel = expTokI) or act[j] (h_q in entry order)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    act = np.ascontiguousarray(act, dtype=np.int8)
    expStart = np.ascontiguousarray(expStart, dtype=np.int32)
    E, rows = W.shape[0], W.shape[1]
    K = act.shape[1]
    assert W.shape[2] == K // QK * Q8_0_BYTES and 0 <= block < K // QK
    n = int(expStart[E])
    out = np.empty((n, rows), np.int32)
    s = None if sel is None else np.ascontiguousarray(sel, dtype=np.int32)
    _L().oracle_block_dots_csr(_p(W), _I(E), _I(rows), _I(K), _p(act), _p(expStart), _p(s), _I(block), _p(out))
    return out


FORMATS = {"q8_0": 0, "q4_k": 1, "q3_k": 2}  # weight formats the oracle reads (GGUF block layouts)


def _fmt(fmt: str) -> int:
    if fmt not in FORMATS:
        raise ValueError(f"unknown weight format {fmt!r}")
    return FORMATS[fmt]


def block_dots_q4_k(w_row: np.ndarray, aq: np.ndarray) -> np.ndarray:
    """int32 dots of a Q4_K row's 32-wide sub-blocks (quants 0..15) with an activation row."""
    w_row = np.ascontiguousarray(w_row, dtype=np.uint8)
    aq = np.ascontiguousarray(aq, dtype=np.int8)
    out = np.empty(aq.size // QK, np.int32)
    _L().oracle_block_dots_q4_k(_p(w_row), _p(aq), _I(aq.size), _p(out))
    return out


def q4_k_dequant(w_row: np.ndarray, K: int) -> np.ndarray:
    """A Q4_K row decoded to K fp32 values (d*sc*q - dmin*m, rounded once)."""
    w_row = np.ascontiguousarray(w_row, dtype=np.uint8)
    out = np.empty(K, np.float32)
    _L().oracle_q4_k_dequant(_p(w_row), _I(K), _p(out))
    return out


def block_dots_q3_k(w_row: np.ndarray, aq: np.ndarray) -> np.ndarray:
    """Per 32-wide block of a Q3_K row: s_2b*isum_2b + s_2b+1*isum_2b+1 (int32)."""
    w_row = np.ascontiguousarray(w_row, dtype=np.uint8)
    aq = np.ascontiguousarray(aq, dtype=np.int8)
    out = np.empty(aq.size // QK, np.int32)
    _L().oracle_block_dots_q3_k(_p(w_row), _p(aq), _I(aq.size), _p(out))
    return out


def q3_k_dequant(w_row: np.ndarray, K: int) -> np.ndarray:
    """A Q3_K row decoded to K fp32 values (d*s_j*q, rounded once)."""
    w_row = np.ascontiguousarray(w_row, dtype=np.uint8)
    out = np.empty(K, np.float32)
    _L().oracle_q3_k_dequant(_p(w_row), _I(K), _p(out))
    return out


def expert_gate_up(Wg, Wu, D: int, F: int, xq, xd16, fmt: str = "q8_0"):
    """One activation row through one expert's gate/up half -> (h, hq, hd16, g, u)."""
    Wg = np.ascontiguousarray(Wg, np.uint8)
    Wu = np.ascontiguousarray(Wu, np.uint8)
    xq = np.ascontiguousarray(xq, np.int8)
    xd16 = np.ascontiguousarray(xd16, np.uint16)
    h = np.empty(F, np.float32)
    hq = np.empty(F, np.int8)
    hd16 = np.empty(F // QK, np.uint16)
    g = np.empty(F, np.float64)
    u = np.empty(F, np.float64)
    _L().oracle_expert_gate_up_fmt(_I(_fmt(fmt)), _p(Wg), _p(Wu), _I(D), _I(F), _p(xq), _p(xd16),
                                   _p(h), _p(hq), _p(hd16), _p(g), _p(u))
    return h, hq, hd16, g, u


def expert_down(Wd, D: int, F: int, hq, hd16, fmt: str = "q8_0") -> np.ndarray:
    Wd = np.ascontiguousarray(Wd, np.uint8)
    hq = np.ascontiguousarray(hq, np.int8)
    hd16 = np.ascontiguousarray(hd16, np.uint16)
    y = np.empty(D, np.float64)
    _L().oracle_expert_down_fmt(_I(_fmt(fmt)), _p(Wd), _I(D), _I(F), _p(hq), _p(hd16), _p(y))
    return y


def grouped_ffn(gate, up, down, xq, xd16, expStart, expTokI, expTokK, k: int, fmt: str = "q8_0"):
    """Routed experts over the CSR -> (partials f32[N*k, D], hq int8[N*k, F], hd16 u16[N*k, F/32])."""
    E, F, _ = gate.shape
    D = down.shape[1]
    N = xq.shape[0]
    partials = np.zeros((N * k, D), np.float32)
    total = int(expStart[E])
    hq = np.zeros((max(total, 1), F), np.int8)
    hd16 = np.zeros((max(total, 1), F // QK), np.uint16)
    _L().oracle_grouped_ffn_fmt(_I(_fmt(fmt)), _p(np.ascontiguousarray(gate)), _p(np.ascontiguousarray(up)),
                            _p(np.ascontiguousarray(down)), _I(E), _I(D), _I(F),
                            _p(np.ascontiguousarray(xq)), _p(np.ascontiguousarray(xd16)),
                            _p(np.ascontiguousarray(expStart, np.int32)),
                            _p(np.ascontiguousarray(expTokI, np.int32)),
                            _p(np.ascontiguousarray(expTokK, np.int32)), _I(k),
                            _p(partials), _p(hq), _p(hd16))
    return partials, hq[:total], hd16[:total]


def shared_expert(sh_gate, sh_up, sh_down, xq, xd16, s, fmt: str = "q8_0"):
    """Sigmoid-gated shared expert -> (S f32[N, D], hq int8[N, Fs], hd16)."""
    Fs = sh_gate.shape[0]
    D = sh_down.shape[0]
    N = xq.shape[0]
    S = np.empty((N, D), np.float32)
    hq = np.empty((N, Fs), np.int8)
    hd16 = np.empty((N, Fs // QK), np.uint16)
    _L().oracle_shared_expert_fmt(_I(_fmt(fmt)), _p(np.ascontiguousarray(sh_gate)), _p(np.ascontiguousarray(sh_up)),
                              _p(np.ascontiguousarray(sh_down)), _I(D), _I(Fs),
                              _p(np.ascontiguousarray(xq)), _p(np.ascontiguousarray(xd16)),
                              _p(_f32(s)), _I64(N), _p(S), _p(hq), _p(hd16))
    return S, hq, hd16


def combine(partials, w, S=None, R=None):
    """Slot-order combine, then the shared row S; with a residual R also + R (the host combine's
    (routed + shared) + resid)."""
    partials = _f32(partials)
    w = _f32(w)
    N, k = w.shape
    D = partials.shape[1]
    assert partials.shape[0] == N * k
    out = np.empty((N, D), np.float32)
    Sp = _p(None if S is None else _f32(S))
    if R is None:
        _L().oracle_combine(_p(partials), _p(w), Sp, _I64(N), _I(k), _I(D), _p(out))
    else:
        R = _f32(R)
        assert R.shape == (N, D)
        _L().oracle_combine_residual(_p(partials), _p(w), Sp, _p(R), _I64(N), _I(k), _I(D), _p(out))
    return out


def combine_residual_rmsnorm(partials, w, S, R, gamma, eps: float):
    """The combine with residual R, then RMSNorm of that row with weight gamma [D] and eps (the
    next layer's input): returns (out, normed)."""
    partials = _f32(partials)
    w = _f32(w)
    N, k = w.shape
    D = partials.shape[1]
    assert partials.shape[0] == N * k
    R = _f32(R)
    gamma = _f32(gamma)
    assert R.shape == (N, D) and gamma.shape == (D,)
    out = np.empty((N, D), np.float32)
    normed = np.empty((N, D), np.float32)
    Sp = _p(None if S is None else _f32(S))
    _L().oracle_combine_residual_rmsnorm(_p(partials), _p(w), Sp, _p(R), _p(gamma), ctypes.c_double(eps), _I64(N),
                                         _I(k), _I(D), _p(out), _p(normed))
    return out, normed


def rmsnorm(x, gamma, eps: float):
    """RMSNorm of rows x with weight gamma: the residual combine's norm with no routed slot
    (one slot of weight 0 contributes +0, then the row x is added)."""
    x = _f32(x)
    N, D = x.shape
    _, normed = combine_residual_rmsnorm(np.zeros((N, D), np.float32), np.zeros((N, 1), np.float32), None, x, gamma,
                                         eps)
    return normed


# ---------------------------------------------------------- whole layer ---
def moe_ffn(hidden, routerW, gate, up, down, top_k: int, norm_topk_prob: bool,
            shexp_gate=None, sh_gate=None, sh_up=None, sh_down=None, keep: bool = True, fmt: str = "q8_0") -> dict:
    """The whole layer, step by step.  Returns every intermediate (keep=True) and ``out``."""
    hidden = _f32(hidden)
    N, D = hidden.shape
    E = routerW.shape[0]
    r = {}
    r["logits"] = router_logits(hidden, routerW)
    r["topk_idx"], r["topk_w"], r["probs"] = softmax_topk(r["logits"], top_k, norm_topk_prob)
    shared = shexp_gate is not None
    if shared:
        r["gate_logit"] = router_logits(hidden, np.asarray(shexp_gate, np.float32).reshape(1, D))[:, 0]
        r["shexp_scale"] = sigmoid(r["gate_logit"])
    r["x_q"], r["x_d16"], r["x_s16"] = quantize_q8_1(hidden)
    r["expStart"], r["expTokI"], r["expTokK"] = bucket(r["topk_idx"], E)
    r["partials"], r["h_q"], r["h_d16"] = grouped_ffn(gate, up, down, r["x_q"], r["x_d16"], r["expStart"],
                                                      r["expTokI"], r["expTokK"], top_k, fmt)
    S = None
    if shared:
        S, r["sh_h_q"], r["sh_h_d16"] = shared_expert(sh_gate, sh_up, sh_down, r["x_q"], r["x_d16"],
                                                      r["shexp_scale"], fmt)
        r["shared_out"] = S
    r["out"] = combine(r["partials"], r["topk_w"], S)
    if not keep:
        r = {"out": r["out"], "topk_idx": r["topk_idx"], "logits": r["logits"]}
    return r


def moe_ffn_inputs(inp: dict, top_k: int, norm_topk_prob: bool, keep: bool = True) -> dict:
    """``moe_ffn`` over a dict made by ``mixture_experts_ffn_top_gb300.workloads.make_inputs``."""
    return moe_ffn(inp["hidden"], inp["routerW"], inp["gate"], inp["up"], inp["down"], top_k,
                   norm_topk_prob, inp.get("shexp_gate"), inp.get("sh_gate"), inp.get("sh_up"),
                   inp.get("sh_down"), keep=keep, fmt=inp.get("wfmt", "q8_0"))
