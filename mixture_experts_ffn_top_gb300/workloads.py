"""Seeded synthetic workloads for the batched routed-MoE FFN layer.

This is the one module that both the CUDA path and the CPU oracle consume.
It draws random numbers and packs them into the layer's input formats; it
holds none of the layer's own arithmetic (no router, no activation
quantiser, no expert FFN, no combine).

Input recipe (numpy ``default_rng``, platform independent; float32
``standard_normal`` draws scaled to the stated standard deviation).  Each
tensor family has its own seeded stream, so expert weights do not depend on N
and can be drawn in parallel:

1. stream ``[seed, 0]``: hidden ``[N, D]`` ~ N(0, 1)
2. stream ``[seed, 1]``: routerW ``[E, D]`` ~ N(0, 1/sqrt(D)) (router logits
   ~N(0, 1)), then the shared-expert gate vector ``[D]`` ~ N(0, 1/sqrt(D))
   (shared expert only), then the skew permutation (skewed routing only)
3. stream ``[seed, 2, e]`` for expert e: gate ``[F, D]``, up ``[F, D]``,
   down ``[D, F]``, each ~ N(0, 0.02), stored as Q8_0 blocks
4. stream ``[seed, 3]``: shared expert gate ``[Fs, D]``, up ``[Fs, D]``,
   down ``[D, Fs]`` ~ N(0, 0.02), Q8_0
5. skewed routing: expert e gets the logit bias
   1.5 * ln(Zipf_{s=1.2} pmf(rank_e)) = -1.8 ln(rank_e) + const with
   rank_e = perm[e] + 1.  The bias is folded into the data (hidden[:, D-1] = 1,
   routerW[:, D-1] = bias) so the layer's arguments stay as the pages state
   them; the constant cancels in the softmax.

Expert weights arrive in the GGUF Q8_0 block format, as a quantised model file
would deliver them: per 32-block an fp16 scale d = fp16(amax/127) followed by
32 int8 quants round(w/d) (half away from zero), 34 bytes per block, blocks
row-major along the reduction dimension.  Packing the weights is how the
synthetic *inputs* are manufactured; both the oracle and the CUDA path take
the resulting bytes as given.

Workloads with ``wfmt="q4_k"`` deliver the same draws as GGUF Q4_K
super-blocks instead (256 values in 144 bytes: fp16 d and dmin, twelve bytes
of packed 6-bit sub-block scales and mins, 4-bit quants; value
d*sc_j*q - dmin*m_j), the K-quant the pages name next to Q8_0 (#406
references: "Q8_0/Q4_K MMQ").  The packer below picks, per 32-wide sub-block,
the step (max - min)/15 and the offset -min (min clipped at 0), codes them
against the super-block's fp16 d = max step/63 and dmin = max offset/63, then
rounds every value to its 4-bit code; any valid encoding would do, since both
sides decode the bytes.

Workloads with ``wfmt="q3_k"`` deliver GGUF Q3_K super-blocks (256 values in
110 bytes: a 32-byte high-bit mask, 64 bytes of 2-bit low parts, twelve bytes
of sixteen packed 6-bit signed sub-block scales s_j, fp16 d; value d*s_j*q with
q in [-4, 3]), the format of the routed experts on the Carnice prefill page
(#388 "Key references": the Q3_K GPU kernel).  The packer takes, per 16-wide
sub-block, the value of largest magnitude v and the step -v/4 (so v codes to
-4, the longer side of the range), codes the steps against the super-block's
fp16 d = max |step|/32, clips s_j to [-32, 31], then rounds every value to its
3-bit code.  Steps of either sign occur, and so do s_j = -32 with q = -4.

The pages ("batched int8-MMQ trunk prefill gated off for MoE", #406; "Carnice
prefill toward llama.cpp 676 t/s", #388) benchmark whole models (OLMoE-1B-7B,
a 35B-A3B hybrid) whose trained weights are not used here: these synthetic
layers stand in for them with the same shapes.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace
from functools import lru_cache

import numpy as np

QK = 32
Q8_0_BYTES = 34
QK_K = 256
Q4_K_BYTES = 144
Q3_K_BYTES = 110


@dataclass(frozen=True)
class Workload:
    name: str
    N: int          # tokens
    D: int          # hidden size (embDim)
    E: int          # routed experts
    top_k: int      # active experts per token (na)
    F: int          # routed expert intermediate size
    Fs: int         # shared expert intermediate size (0 = none)
    norm_topk_prob: bool
    seed: int
    skew: bool = False
    wfmt: str = "q8_0"  # expert weight format: "q8_0", "q4_k" or "q3_k"

    @property
    def has_shared(self) -> bool:
        return self.Fs > 0

    def with_tokens(self, N: int) -> "Workload":
        return replace(self, N=N, name=f"{self.name.split('_n')[0]}_n{N}")

    def describe(self) -> str:
        s = (f"N={self.N} D={self.D} E={self.E} top_k={self.top_k} F={self.F}"
             f" norm_topk_prob={int(self.norm_topk_prob)}")
        if self.Fs:
            s += f" shared_Fs={self.Fs}"
        if self.skew:
            s += " zipf_skew=1.2"
        if self.wfmt != "q8_0":
            s += f" weights={self.wfmt}"
        return s + f" seed={self.seed}"


WORKLOADS = {
    "tiny": Workload("tiny", N=64, D=256, E=8, top_k=2, F=128, Fs=0, norm_topk_prob=False, seed=0),
    "olmoe": Workload("olmoe", N=2048, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False, seed=1),
    "decode_n1": Workload("decode_n1", N=1, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False, seed=2),
    "decode_n4": Workload("decode_n4", N=4, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False, seed=2),
    "decode_n8": Workload("decode_n8", N=8, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False, seed=2),
    "qwen3moe_shared": Workload("qwen3moe_shared", N=512, D=2048, E=256, top_k=8, F=512, Fs=512,
                                norm_topk_prob=True, seed=3),
    "skewed": Workload("skewed", N=4096, D=2048, E=128, top_k=8, F=768, Fs=0, norm_topk_prob=True,
                       seed=4, skew=True),
    # the same layer family with Q4_K expert weights (D, F, Fs multiples of 256)
    "tiny_q4k": Workload("tiny_q4k", N=64, D=256, E=8, top_k=2, F=256, Fs=0, norm_topk_prob=False, seed=0,
                         wfmt="q4_k"),
    "q4k_shared": Workload("q4k_shared", N=256, D=512, E=16, top_k=4, F=256, Fs=256, norm_topk_prob=True,
                           seed=5, wfmt="q4_k"),
    "olmoe_q4k": Workload("olmoe_q4k", N=2048, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False,
                          seed=1, wfmt="q4_k"),
    "decode_n8_q4k": Workload("decode_n8_q4k", N=8, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False,
                              seed=2, wfmt="q4_k"),
    # and with Q3_K expert weights
    "tiny_q3k": Workload("tiny_q3k", N=64, D=256, E=8, top_k=2, F=256, Fs=0, norm_topk_prob=False, seed=0,
                         wfmt="q3_k"),
    "q3k_shared": Workload("q3k_shared", N=256, D=512, E=16, top_k=4, F=256, Fs=256, norm_topk_prob=True,
                           seed=6, wfmt="q3_k"),
    "olmoe_q3k": Workload("olmoe_q3k", N=2048, D=2048, E=64, top_k=8, F=1024, Fs=0, norm_topk_prob=False,
                          seed=1, wfmt="q3_k"),
}


def row_bytes(wfmt: str, K: int) -> int:
    """Bytes of one weight row of K values in the given block format."""
    if wfmt in ("q4_k", "q3_k"):
        assert K % QK_K == 0
        return K // QK_K * (Q4_K_BYTES if wfmt == "q4_k" else Q3_K_BYTES)
    assert wfmt == "q8_0" and K % QK == 0
    return K // QK * Q8_0_BYTES


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def pack_q8_0(w: np.ndarray) -> np.ndarray:
    """Pack fp32 weights ``[rows, K]`` into GGUF Q8_0 blocks ``uint8[rows, K/32*34]``."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % QK == 0
    b = w.reshape(rows, K // QK, QK)
    amax = np.abs(b).max(axis=2)
    d = (amax / np.float32(127.0)).astype(np.float32)
    inv = np.zeros_like(d)
    nz = d != 0
    inv[nz] = (np.float32(1.0) / d[nz]).astype(np.float32)
    v = (b * inv[..., None]).astype(np.float32)
    q = np.sign(v) * np.floor(np.abs(v).astype(np.float64) + 0.5)
    out = np.empty((rows, K // QK, Q8_0_BYTES), np.uint8)
    out[..., 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, K // QK, 2)
    out[..., 2:] = q.astype(np.int8).view(np.uint8)
    return out.reshape(rows, (K // QK) * Q8_0_BYTES)


def pack_q4_k(w: np.ndarray) -> np.ndarray:
    """Pack fp32 weights ``[rows, K]`` into GGUF Q4_K super-blocks ``uint8[rows, K/256*144]``."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % QK_K == 0
    nsb = K // QK_K
    x = w.reshape(rows, nsb, 8, QK).astype(np.float64)
    lo = np.minimum(x.min(axis=3), 0.0)
    step = (x.max(axis=3) - lo) / 15.0
    off = -lo
    d16 = (step.max(axis=2) / 63.0).astype(np.float16)
    dmin16 = (off.max(axis=2) / 63.0).astype(np.float16)
    d = d16.astype(np.float64)[..., None]
    dmin = dmin16.astype(np.float64)[..., None]
    sc = np.where(d > 0, np.clip(np.rint(step / np.where(d > 0, d, 1.0)), 0, 63), 0).astype(np.uint8)
    m = np.where(dmin > 0, np.clip(np.rint(off / np.where(dmin > 0, dmin, 1.0)), 0, 63), 0).astype(np.uint8)
    qstep = (d * sc)[..., None]
    qoff = (dmin * m)[..., None]
    q = np.where(qstep > 0, np.clip(np.rint((x + qoff) / np.where(qstep > 0, qstep, 1.0)), 0, 15), 0)
    q = q.astype(np.uint8)  # [rows, nsb, 8, 32]
    out = np.zeros((rows, nsb, Q4_K_BYTES), np.uint8)
    out[..., 0:2] = d16.view(np.uint8).reshape(rows, nsb, 2)
    out[..., 2:4] = dmin16.view(np.uint8).reshape(rows, nsb, 2)
    out[..., 4:8] = sc[..., 0:4] | ((sc[..., 4:8] >> 4) << 6)
    out[..., 8:12] = m[..., 0:4] | ((m[..., 4:8] >> 4) << 6)
    out[..., 12:16] = (sc[..., 4:8] & 15) | ((m[..., 4:8] & 15) << 4)
    for g in range(4):
        out[..., 16 + 32 * g:48 + 32 * g] = q[..., 2 * g, :] | (q[..., 2 * g + 1, :] << 4)
    return out.reshape(rows, nsb * Q4_K_BYTES)


def pack_q3_k(w: np.ndarray) -> np.ndarray:
    """Pack fp32 weights ``[rows, K]`` into GGUF Q3_K super-blocks ``uint8[rows, K/256*110]``."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, K = w.shape
    assert K % QK_K == 0
    nsb = K // QK_K
    x = w.reshape(rows, nsb, 16, 16).astype(np.float64)
    big = np.take_along_axis(x, np.abs(x).argmax(axis=3)[..., None], axis=3)[..., 0]
    step = -big / 4.0  # [rows, nsb, 16]
    d16 = (np.abs(step).max(axis=2) / 32.0).astype(np.float16)
    d = d16.astype(np.float64)[..., None]
    s = np.where(d > 0, np.clip(np.rint(step / np.where(d > 0, d, 1.0)), -32, 31), 0)
    qstep = (d * s)[..., None]
    q = np.where(qstep != 0, np.clip(np.rint(x / np.where(qstep != 0, qstep, 1.0)), -4, 3), 0)
    q = (q.astype(np.int64) + 4).reshape(rows, nsb, QK_K)  # 0..7: low two bits + high bit
    raw = (s.astype(np.int64) + 32).astype(np.uint8)  # [rows, nsb, 16], 0..63
    out = np.zeros((rows, nsb, Q3_K_BYTES), np.uint8)
    hbit = (q >> 2) & 1
    low = q & 3
    for b in range(8):  # hmask: bit b of byte l holds value 32*b + l
        out[..., 0:32] |= (hbit[..., 32 * b:32 * b + 32] << b).astype(np.uint8)
    for i0 in range(0, QK_K, 32):  # qs: value i in byte 32 + 32*(i/128) + i%32 at bits 2*((i%128)/32)
        byte0 = 32 + 32 * (i0 // 128)
        shift = 2 * ((i0 % 128) // 32)
        out[..., byte0:byte0 + 32] |= (low[..., i0:i0 + 32] << shift).astype(np.uint8)
    out[..., 96:104] = (raw[..., 0:8] & 15) | ((raw[..., 8:16] & 15) << 4)
    for g in range(4):  # byte 100 + 8 + m: high bits of scales m, m+4, m+8, m+12
        out[..., 104:108] |= ((raw[..., 4 * g:4 * g + 4] >> 4) << (2 * g)).astype(np.uint8)
    out[..., 108:110] = d16.view(np.uint8).reshape(rows, nsb, 2)
    return out.reshape(rows, nsb * Q3_K_BYTES)


def pack_weights(w: np.ndarray, wfmt: str) -> np.ndarray:
    if wfmt == "q4_k":
        return pack_q4_k(w)
    if wfmt == "q3_k":
        return pack_q3_k(w)
    return pack_q8_0(w)


def _expert(seed: int, e: int, D: int, F: int, wfmt: str = "q8_0"):
    rng = np.random.default_rng([seed, 2, e])
    g = pack_weights(_normal(rng, (F, D), 0.02), wfmt)
    u = pack_weights(_normal(rng, (F, D), 0.02), wfmt)
    d = pack_weights(_normal(rng, (D, F), 0.02), wfmt)
    return g, u, d


@lru_cache(maxsize=8)
def _experts(seed: int, E: int, D: int, F: int, wfmt: str = "q8_0"):
    gate = np.empty((E, F, row_bytes(wfmt, D)), np.uint8)
    up = np.empty_like(gate)
    down = np.empty((E, D, row_bytes(wfmt, F)), np.uint8)

    def one(e):
        gate[e], up[e], down[e] = _expert(seed, e, D, F, wfmt)

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(one, range(E)))
    for a in (gate, up, down):
        a.setflags(write=False)
    return gate, up, down


def make_inputs(wl: Workload) -> dict:
    """Draw one workload's inputs.  Returns numpy arrays:

    hidden f32[N,D], routerW f32[E,D], shexp_gate f32[D] or None,
    gate/up u8[E,F,row_bytes(D)], down u8[E,D,row_bytes(F)],
    sh_gate/sh_up u8[Fs,row_bytes(D)], sh_down u8[D,row_bytes(Fs)] (or None),
    wfmt: the block format of those byte rows ("q8_0": D/32*34 bytes, "q4_k": D/256*144,
    "q3_k": D/256*110).
    The expert arrays are shared read-only between calls with equal shapes.
    """
    N, D, E, F, Fs = wl.N, wl.D, wl.E, wl.F, wl.Fs
    assert D % QK == 0 and F % QK == 0 and Fs % QK == 0
    hidden = _normal(np.random.default_rng([wl.seed, 0]), (N, D), 1.0)
    rng = np.random.default_rng([wl.seed, 1])
    routerW = _normal(rng, (E, D), 1.0 / np.sqrt(D))
    shexp_gate = _normal(rng, (D,), 1.0 / np.sqrt(D)) if Fs else None
    gate, up, down = _experts(wl.seed, E, D, F, wl.wfmt)
    sh_gate = sh_up = sh_down = None
    if Fs:
        srng = np.random.default_rng([wl.seed, 3])
        sh_gate = pack_weights(_normal(srng, (Fs, D), 0.02), wl.wfmt)
        sh_up = pack_weights(_normal(srng, (Fs, D), 0.02), wl.wfmt)
        sh_down = pack_weights(_normal(srng, (D, Fs), 0.02), wl.wfmt)
    if wl.skew:
        perm = rng.permutation(E)
        bias = (1.5 * -1.2 * np.log(perm + 1.0)).astype(np.float32)
        hidden[:, D - 1] = 1.0
        routerW[:, D - 1] = bias
    return dict(hidden=hidden, routerW=routerW, shexp_gate=shexp_gate,
                gate=gate, up=up, down=down, sh_gate=sh_gate, sh_up=sh_up, sh_down=sh_down, wfmt=wl.wfmt)


def make_hidden(wl: Workload, seed_offset: int = 0) -> np.ndarray:
    """A fresh hidden batch of the workload's shape (used to vary inputs between steps)."""
    rng = np.random.default_rng([wl.seed, 4, seed_offset])
    h = _normal(rng, (wl.N, wl.D), 1.0)
    if wl.skew:
        h[:, wl.D - 1] = 1.0
    return h


def expert_weight_bytes(wl: Workload) -> int:
    """Q8_0 bytes of one routed expert (gate + up + down)."""
    return 3 * wl.F * wl.D // QK * Q8_0_BYTES
