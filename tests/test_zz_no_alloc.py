"""moe_router_topk_noalloc: the router for callers that cannot allocate device memory.

Hosts whose device memory belongs to another allocator (or that forbid cudaMalloc
after start-up) cannot hand the library a workspace; this entry point keeps the
router's scratch in a fixed array inside the library instead.  Its results must
equal those of moe_router_topk (same kernels, same split-K order) on two calls
in a row, and a problem too large for the fixed array must be refused before
anything runs.  This file is collected last on purpose.
"""
import numpy as np
import pytest

from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_top_gb300 import build, ops as _ops

    build.build()
    torch.cuda.set_device(0)
    return _ops


@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared"])
def test_noalloc_router_matches_workspace_router(ops, name):
    """The no-alloc router (always the fp32 SIMT kernels) against moe_router_topk, which takes the
    tensor-core router where it applies (OLMoE): identical quantised activations, logits within the
    router's tolerance, identical routing on tokens whose k-th / (k+1)-th logit gap is clear."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    hidden = torch.from_numpy(inp["hidden"]).cuda()
    routerW = torch.from_numpy(inp["routerW"]).cuda()
    shg = None if inp["shexp_gate"] is None else torch.from_numpy(inp["shexp_gate"]).cuda()
    ws = ops.new_workspace(wl.N, wl.D, wl.E, wl.F, wl.top_k, wl.Fs)
    ref = ops.moe_router_topk(hidden, routerW, shg, wl.top_k, wl.norm_topk_prob, ws, want_logits=True)
    torch.cuda.synchronize()
    for _ in range(2):  # the shared scratch keeps the previous call's contents
        got = ops.moe_router_topk_noalloc(hidden, routerW, shg, wl.top_k, wl.norm_topk_prob, want_logits=True)
        torch.cuda.synchronize()
        lg, lr = got["logits"].cpu().numpy(), ref["logits"].cpu().numpy()
        scale = np.maximum(np.abs(lr).max(axis=1), np.sqrt((lr ** 2).mean(axis=1)))
        assert (np.abs(lg - lr).max(axis=1) <= 2e-4 * scale).all()
        srt = np.sort(lr, axis=1)[:, ::-1]
        clear = (srt[:, wl.top_k - 1] - srt[:, wl.top_k]) > 4e-4 * scale
        assert clear.mean() > 0.9
        np.testing.assert_array_equal(got["topk_idx"].cpu().numpy()[clear], ref["topk_idx"].cpu().numpy()[clear])
        np.testing.assert_allclose(got["topk_w"].cpu().numpy()[clear], ref["topk_w"].cpu().numpy()[clear],
                                   rtol=2e-4, atol=1e-6)
        np.testing.assert_array_equal(got["x_q"].cpu().numpy(), ref["x_q"].cpu().numpy())
        np.testing.assert_array_equal(got["x_d"].cpu().numpy(), ref["x_d"].cpu().numpy())
        if shg is not None:
            np.testing.assert_allclose(got["shexp_scale"].cpu().numpy(), ref["shexp_scale"].cpu().numpy(),
                                       rtol=1e-4, atol=1e-6)


def test_noalloc_router_refuses_oversized_problem(ops):
    # N * (E + 1) alone exceeds the 2^22-float scratch: refused on the host, nothing launched
    N, D, E = 40000, 64, 128
    hidden = torch.zeros((N, D), dtype=torch.float32, device="cuda")
    routerW = torch.zeros((E, D), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.MoeError) as exc:
        ops.moe_router_topk_noalloc(hidden, routerW, None, 8, False)
    assert exc.value.code == -3


def _split_used(N, D, E, sms):
    """The router's split-K factor as the header states it."""
    if N <= 8 and D % 4 == 0:
        return 1
    tiles = -(-N // 64) * -(-E // 64)
    depth = 32 if tiles <= 4 else 128
    cap = min(-(-4 * sms // tiles), max(1, D // depth))
    s = max(1, cap)
    while s > 1 and (D // 32) % s != 0:
        s -= 1
    return s


def test_noalloc_router_refuses_when_the_split_decides(ops):
    # N * (E + 1) fits the 2^22-float scratch, the split-K table does not: refused on the host
    # before anything runs, and no output is written
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N, D, E = 2048, 2048, 1024
    split = _split_used(N, D, E, sms)
    if not (N * (E + 1) <= 1 << 22 < split * N * (E + 1)):
        pytest.skip(f"split {split} on {sms} SMs does not decide this shape")
    hidden = torch.randn((N, D), dtype=torch.float32, device="cuda")
    routerW = torch.randn((E, D), dtype=torch.float32, device="cuda")
    outs = dict(topk_idx=torch.full((N, 8), -7, dtype=torch.int32, device="cuda"),
                topk_w=torch.full((N, 8), -7.0, dtype=torch.float32, device="cuda"),
                shexp_scale=None,
                x_q=torch.full((N, D), -7, dtype=torch.int8, device="cuda"),
                x_d=torch.full((N, D // 32), -7.0, dtype=torch.float32, device="cuda"),
                logits=torch.full((N, E), -7.0, dtype=torch.float32, device="cuda"))
    with pytest.raises(ops.MoeError) as exc:
        ops.moe_router_topk_noalloc(hidden, routerW, None, 8, False, want_logits=True, outputs=outs)
    assert exc.value.code == -3
    torch.cuda.synchronize()
    for name, t in outs.items():
        if t is not None:
            assert (t == -7).all(), f"{name} was written"


def test_noalloc_router_small_batch_uses_one_split(ops):
    # a decode-sized batch is routed in one pass (no split-K table beyond N * (E + 1))
    wl = WORKLOADS["decode_n8"]
    inp = make_inputs(wl)
    hidden = torch.from_numpy(inp["hidden"]).cuda()
    routerW = torch.from_numpy(inp["routerW"]).cuda()
    ws = ops.new_workspace(wl.N, wl.D, wl.E, wl.F, wl.top_k, wl.Fs)
    ref = ops.moe_router_topk(hidden, routerW, None, wl.top_k, wl.norm_topk_prob, ws, want_logits=True)
    got = ops.moe_router_topk_noalloc(hidden, routerW, None, wl.top_k, wl.norm_topk_prob, want_logits=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["topk_idx"].cpu().numpy(), ref["topk_idx"].cpu().numpy())
    np.testing.assert_array_equal(got["logits"].cpu().numpy(), ref["logits"].cpu().numpy())
