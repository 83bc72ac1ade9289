"""Expert parallelism's partition, exchange and reassembly on CPU ranks (gloo): every rank owns
a contiguous range of the routed experts, routes and buckets its own tokens, ships each
(token, slot) entry's quantised activation row to the expert's owner with all_to_all_single,
gets the fp32 partial rows back and combines locally.  The compute steps are the oracle's
(a backend defined here, on the host); the layer output of every rank must equal the
single-rank oracle layer on the same tokens bit for bit.  No GPU is touched."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleBackend:
    """The oracle's steps for one rank: the router over all experts, the routed experts [lo, hi)
    and the shared expert.  Block scales travel as their fp16 bit patterns (int16)."""

    def __init__(self, inp, lo, hi):
        import oracle as O

        self.O = O
        self.inp = inp
        self.gate, self.up, self.down = inp["gate"][lo:hi], inp["up"][lo:hi], inp["down"][lo:hi]
        self.E_local = hi - lo
        self.fmt = inp.get("wfmt", "q8_0")

    def route(self, hidden, top_k, norm):
        O = self.O
        h = hidden.numpy()
        logits = O.router_logits(h, self.inp["routerW"])
        idx, w, _ = O.softmax_topk(logits, top_k, norm)
        xq, xd16, _ = O.quantize_q8_1(h)
        r = dict(topk_idx=torch.from_numpy(idx), topk_w=torch.from_numpy(w), x_q=torch.from_numpy(xq),
                 x_d=torch.from_numpy(xd16.view(np.int16)), shexp_scale=None)
        if self.inp.get("shexp_gate") is not None:
            g = O.router_logits(h, np.asarray(self.inp["shexp_gate"], np.float32).reshape(1, -1))[:, 0]
            r["shexp_scale"] = torch.from_numpy(O.sigmoid(g))
        return r

    def bucket(self, topk_idx, E):
        es, ti, tk = self.O.bucket(topk_idx.numpy(), E)
        return torch.from_numpy(es), torch.from_numpy(ti), torch.from_numpy(tk)

    def experts(self, x_q, x_d, loc):
        O = self.O
        R = x_q.shape[0]
        D = self.down.shape[1]
        if R == 0:
            return torch.zeros((0, D), dtype=torch.float32)
        es, ti, tk = O.bucket(loc.numpy().reshape(R, 1).astype(np.int32), self.E_local)
        part, _, _ = O.grouped_ffn(self.gate, self.up, self.down, x_q.numpy(), x_d.numpy().view(np.uint16), es, ti,
                                   tk, 1, self.fmt)
        return torch.from_numpy(part)

    def shared(self, r):
        if r["shexp_scale"] is None:
            return None
        S, _, _ = self.O.shared_expert(self.inp["sh_gate"], self.inp["sh_up"], self.inp["sh_down"], r["x_q"].numpy(),
                                       r["x_d"].numpy().view(np.uint16), r["shexp_scale"].numpy(), self.fmt)
        return torch.from_numpy(S)

    def combine(self, partials, topk_w, S):
        return torch.from_numpy(self.O.combine(partials.numpy(), topk_w.numpy(), None if S is None else S.numpy()))


def _workload(name):
    from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, Workload

    if name in WORKLOADS:
        return WORKLOADS[name]
    # small layers with a shared expert, and one whose routing leaves an owner without entries
    return {"small_shared": Workload("small_shared", 48, 128, 6, 2, 64, 64, True, 21),
            "few_tokens": Workload("few_tokens", 3, 128, 12, 2, 64, 0, False, 22)}[name]


def _rank_main(rank, world, port, out_dir, name):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as O
        from mixture_experts_ffn_top_gb300.expert_parallel import expert_parallel_forward, expert_ranges
        from mixture_experts_ffn_top_gb300.workloads import make_hidden, make_inputs

        wl = _workload(name)
        inp = make_inputs(wl)
        inp["hidden"] = make_hidden(wl, seed_offset=rank)  # every rank its own tokens
        lo, hi = expert_ranges(wl.E, world)[rank]
        be = OracleBackend(inp, lo, hi)
        out = expert_parallel_forward(be, torch.from_numpy(inp["hidden"]), wl.E, wl.top_k, wl.norm_topk_prob)
        ref = O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)["out"]
        np.save(os.path.join(out_dir, f"out{rank}.npy"), out.numpy())
        np.save(os.path.join(out_dir, f"ref{rank}.npy"), ref)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name,world", [("tiny", 2), ("small_shared", 2), ("small_shared", 3), ("few_tokens", 4)])
def test_expert_parallel_matches_single_rank(tmp_path, name, world):
    port = _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path), name), nprocs=world, start_method="spawn",
                       join=True)
    for r in range(world):
        out, ref = np.load(tmp_path / f"out{r}.npy"), np.load(tmp_path / f"ref{r}.npy")
        assert out.shape == ref.shape
        assert np.array_equal(out.view(np.uint32), ref.view(np.uint32)), f"rank {r}: not bit-identical"


def test_expert_ranges():
    from mixture_experts_ffn_top_gb300.expert_parallel import expert_ranges

    assert expert_ranges(8, 2) == [(0, 4), (4, 8)]
    assert expert_ranges(8, 3) == [(0, 3), (3, 6), (6, 8)]
    assert expert_ranges(64, 8)[-1] == (56, 64)
    for E, G in [(7, 3), (256, 8), (5, 5)]:
        rs = expert_ranges(E, G)
        assert rs[0][0] == 0 and rs[-1][1] == E
        assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
        assert max(h - l for l, h in rs) - min(h - l for l, h in rs) <= 1
    with pytest.raises(ValueError):
        expert_ranges(3, 4)
