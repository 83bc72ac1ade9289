"""Failure detection on the GPU without a fault: a device wait that can never be
satisfied runs out after its bound, the kernel reports MOE_DEV_TIMEOUT in the status
word, and the context stays usable (the next layer call is correct)."""
import time

import numpy as np
import pytest

import oracle as O
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


def test_starved_gemm_times_out_and_context_survives(ops):
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl)
    ref = O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)
    layer = ops.MoeLayer.from_numpy(inp, device="cuda:0", top_k=wl.top_k, max_tokens=wl.N)
    if not ops.moe_weights_tensor_path(layer.w):
        pytest.skip("tensor path unavailable")
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t0 = time.time()
    ops.moe_debug_expert_wait_timeout(layer.w, d(ref["x_q"]), d(O.halves(ref["x_d16"])), d(ref["expStart"]),
                                      d(ref["expTokI"]), wl.top_k, 100, layer.ws)
    word = layer.status()  # synchronises
    elapsed = time.time() - t0
    assert word & 0x4, f"status word {word}: no timeout reported"
    assert ops.lib().moe_status_from_word(word) == -5
    assert elapsed < 30
    # the context is still usable and the status was cleared
    out = layer.prefill(d(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=2)
    assert layer.status() == 0
    got = out.cpu().numpy().astype(np.float64)
    r = ref["out"].astype(np.float64)
    assert np.linalg.norm(got - r) / np.linalg.norm(r) < 2e-3


def test_bucket_barrier_times_out_and_workspace_recovers(ops):
    """The bucketing kernel's grid barrier told to wait for one CTA more than were launched: every
    CTA gives up after the limit, the status word says timeout, the CSR is left unwritten; after
    moe_workspace_init the same workspace buckets correctly."""
    N, E, k = 4096, 64, 8
    rng = np.random.default_rng(5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    ws = ops.new_workspace(N, 32, E, 32, k)  # holds the bucketing scratch
    d_idx = torch.from_numpy(idx).cuda()
    t0 = time.time()
    es, ti, tk = ops.moe_debug_bucket_barrier_timeout(d_idx, E, 20, ws)
    word = ops.moe_workspace_status(ws)  # synchronises
    elapsed = time.time() - t0
    assert word & 0x4, f"status word {word}: no timeout reported"
    assert ops.lib().moe_status_from_word(word) == -5
    assert elapsed < 30
    assert (es.cpu().numpy() == -7).all() and (ti.cpu().numpy() == -7).all()  # nothing written
    ops.moe_workspace_init(ws)
    es, ti, tk = ops.moe_bucket(d_idx, E, ws)
    assert ops.moe_workspace_status(ws) == 0
    res, rti, rtk = O.bucket(idx, E)
    np.testing.assert_array_equal(es.cpu().numpy(), res)
    np.testing.assert_array_equal(ti.cpu().numpy(), rti)
    np.testing.assert_array_equal(tk.cpu().numpy(), rtk)
