"""Expert parallelism for the batched routed-MoE FFN across GPUs of one node.

The layer shards by expert with one exchange each way (the grouped expert GEMM
of "Carnice prefill toward llama.cpp 676 t/s", #388, "Remaining levers" 3,
spread over several GPUs).  Rank g of G owns the routed experts
[lo_g, hi_g) (contiguous, near-equal ranges; ``expert_ranges``) and a copy of
the router and of the shared expert.  One layer pass on every rank, over that
rank's own token batch:

  1. route locally: router logits, softmax/top-k, shared-expert scale, Q8_1 of
     the hidden rows;
  2. bucket locally into the CSR (expStart/expTokI/expTokK).  Its entries are
     grouped by expert, so the entries of owner g are one contiguous run;
  3. exchange the counts, then each entry's quantised activation row (codes
     and block scales) and its expert index local to the owner, with one
     ``all_to_all_single``; the rows land in the owner's memory;
  4. the owner runs its experts over the received rows, each row one token
     with top_k = 1 routed to its local expert, giving one unweighted fp32
     partial row per received entry;
  5. ``all_to_all_single`` returns the partial rows to the token owners, which
     put entry (t, slot) at partials[t * top_k + slot];
  6. the token owner adds its shared expert and runs the combine.

A partial row depends on its token's activation row and its expert only, so
every rank's output equals the single-GPU layer's output on the same tokens
bit for bit, provided the owners' expert kernels compute each row the way the
single-GPU call would (the same expert path).  The combine's fixed slot order
is untouched by the exchange.

The compute steps come from a backend object (``DeviceBackend`` below runs the
library's kernels through the C ABI on the rank's GPU); the exchange is plain
``torch.distributed`` collectives on the backend's tensors, so the same code
runs over NCCL on device tensors or over gloo on host tensors.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import ops


def expert_ranges(E: int, world: int) -> list[tuple[int, int]]:
    """Contiguous expert ranges [lo, hi) of the ranks: sizes differ by at most one, larger first."""
    if world < 1 or E < world:
        raise ValueError(f"{E} experts cannot be split over {world} ranks")
    base, extra = divmod(E, world)
    out, lo = [], 0
    for g in range(world):
        hi = lo + base + (1 if g < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def _pack_rows(x_q: torch.Tensor, x_d: torch.Tensor, local_expert: torch.Tensor) -> torch.Tensor:
    """One uint8 row per entry: the activation codes, the raw bytes of its block scales, and its
    local expert index (int32)."""
    R = x_q.shape[0]
    parts = [x_q.reshape(R, -1).view(torch.uint8),
             x_d.reshape(R, -1).contiguous().view(torch.uint8),
             local_expert.to(torch.int32).reshape(R, 1).contiguous().view(torch.uint8)]
    return torch.cat(parts, dim=1).contiguous()


def _unpack_rows(buf: torch.Tensor, D: int, scale_dtype: torch.dtype, scale_cols: int):
    sbytes = scale_cols * torch.empty((), dtype=scale_dtype).element_size()
    x_q = buf[:, :D].contiguous().view(torch.int8)
    x_d = buf[:, D:D + sbytes].contiguous().view(scale_dtype)
    loc = buf[:, D + sbytes:D + sbytes + 4].contiguous().view(torch.int32).reshape(-1)
    return x_q, x_d, loc


def _all_to_all_rows(send: torch.Tensor, send_counts: list[int], recv_counts: list[int], group=None) -> torch.Tensor:
    recv = send.new_empty((sum(recv_counts),) + tuple(send.shape[1:]))
    dist.all_to_all_single(recv, send, output_split_sizes=recv_counts, input_split_sizes=send_counts, group=group)
    return recv


def expert_parallel_forward(backend, hidden: torch.Tensor, E: int, top_k: int, norm_topk_prob: bool,
                            group=None) -> torch.Tensor:
    """One layer pass over this rank's tokens with the routed experts sharded over the group
    (the experts of this rank's range are the backend's)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    ranges = expert_ranges(E, world)
    lo, hi = ranges[rank]
    N, D = hidden.shape
    r = backend.route(hidden, top_k, norm_topk_prob)
    expStart, expTokI, expTokK = backend.bucket(r["topk_idx"], E)
    es = expStart.cpu().numpy()
    send_counts = [int(es[h] - es[l]) for l, h in ranges]
    total = int(es[E])
    # entry j's expert: the segment holding j; its index inside the owner's range
    ent_expert = torch.from_numpy(np.repeat(np.arange(E, dtype=np.int32), np.diff(es))).to(hidden.device)
    owner_lo = torch.from_numpy(np.repeat(np.array([l for l, _ in ranges], np.int32), send_counts)).to(hidden.device)
    tok = expTokI[:total].long()
    payload = _pack_rows(r["x_q"][tok], r["x_d"][tok], ent_expert - owner_lo)
    counts = torch.tensor(send_counts, dtype=torch.int64, device=hidden.device)
    recv_counts_t = torch.empty_like(counts)
    dist.all_to_all_single(recv_counts_t, counts, group=group)
    recv_counts = [int(c) for c in recv_counts_t.cpu().tolist()]
    recv = _all_to_all_rows(payload, send_counts, recv_counts, group)
    x_q_r, x_d_r, loc = _unpack_rows(recv, D, r["x_d"].dtype, r["x_d"].shape[1])
    if int(loc.numel()) and (int(loc.min()) < 0 or int(loc.max()) >= hi - lo):
        raise RuntimeError("received an entry for an expert outside this rank's range")
    rows = backend.experts(x_q_r, x_d_r, loc)  # [R, D] fp32, row i for received entry i
    back = _all_to_all_rows(rows, recv_counts, send_counts, group)
    partials = torch.zeros((N * top_k, D), dtype=torch.float32, device=hidden.device)
    dst = expTokI[:total].long() * top_k + expTokK[:total].long()
    partials[dst] = back
    S = backend.shared(r)
    return backend.combine(partials, r["topk_w"], S)


class DeviceBackend:
    """The library's kernels on this rank's GPU (C ABI through ``ops``): the router over all E
    experts, the rank's routed experts [lo, hi) and the shared expert.  The experts run on the
    expert path the single-GPU layer would take for the same batch (tensor cores once the batch
    holds N >= 64 tokens and N * top_k / E >= 8 rows per expert, else the matvec path), so every
    partial row is computed exactly as there."""

    def __init__(self, inp: dict, lo: int, hi: int, device, top_k: int, max_tokens: int):
        self.device = torch.device(device)
        self.E_all = inp["gate"].shape[0]
        self.D = inp["down"].shape[1]
        local = dict(inp)
        local["gate"], local["up"], local["down"] = inp["gate"][lo:hi], inp["up"][lo:hi], inp["down"][lo:hi]
        self.layer = ops.MoeLayer.from_numpy(local, device=self.device, top_k=1, max_tokens=max(1, max_tokens))
        self.w = self.layer.w
        self.routerW = self.layer.routerW
        self.shexp_gate = self.layer.shexp_gate
        self.top_k = top_k
        self.max_tokens = max_tokens
        F, Fs = inp["gate"].shape[1], (0 if inp.get("sh_gate") is None else inp["sh_gate"].shape[0])
        self.route_ws = ops.new_workspace(max_tokens, self.D, self.E_all, F, top_k, Fs, device=self.device)
        self._exp_ws = None
        self._exp_rows = 0

    def route(self, hidden, top_k, norm_topk_prob):
        r = ops.moe_router_topk(hidden, self.routerW, self.shexp_gate, top_k, norm_topk_prob, self.route_ws)
        N = hidden.shape[0]
        tensor = ops.moe_weights_tensor_path(self.w) and N >= 64 and N * top_k // self.E_all >= 8
        self.path = ops.MOE_PATH_TENSOR if tensor else ops.MOE_PATH_MATVEC
        return r

    def bucket(self, topk_idx, E):
        return ops.moe_bucket(topk_idx, E, self.route_ws)

    def experts(self, x_q, x_d, loc):
        R = x_q.shape[0]
        if R == 0:
            return torch.empty((0, self.D), dtype=torch.float32, device=self.device)
        if R > self._exp_rows:
            self._exp_rows = R
            self._exp_ws = ops.new_workspace(R, self.D, self.w.E, self.w.F, 1, self.w.Fs, device=self.device)
        es, ti, tk = ops.moe_bucket(loc.reshape(R, 1), self.w.E, self._exp_ws)
        part, _ = ops.moe_grouped_ffn(self.w, x_q, x_d, es, ti, tk, 1, self._exp_ws, path=self.path)
        return part

    def shared(self, r):
        if self.shexp_gate is None:
            return None
        N = r["x_q"].shape[0]
        empty = torch.zeros(self.w.E + 1, dtype=torch.int32, device=self.device)
        none = torch.zeros(max(1, N), dtype=torch.int32, device=self.device)
        ws = ops.new_workspace(N, self.D, self.w.E, self.w.F, 1, self.w.Fs, device=self.device)
        _, S = ops.moe_grouped_ffn(self.w, r["x_q"], r["x_d"], empty, none, none, 1, ws,
                                   shexp_scale=r["shexp_scale"], path=self.path)
        return S

    def combine(self, partials, topk_w, S):
        return ops.moe_combine(partials, topk_w, S)
