"""GPU parity: every step of the CUDA path, called through the C ABI, against
the CPU oracle on the same seeded inputs.

Bars (from the layer's contract):
  - routing indices, CSR arrays, Q8_1 codes of x and the int32 block dot
    products: bit-exact (routing given the same logits, or on tokens whose
    k-th/(k+1)-th logit gap exceeds twice the logit tolerance);
  - router logits: |dl| <= 1e-4 * max(|l_ref|_max, rms(l_ref)) per token row;
  - FFN outputs: relative L2 <= 2e-3 and max-abs <= 1e-2 of the oracle;
  - the combine, given identical partials and weights: bit-exact.
"""
import numpy as np
import pytest

import oracle as O
from mixture_experts_ffn_top_gb300.workloads import Q8_0_BYTES, WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LOGIT_RTOL = 1e-4
OUT_REL_L2 = 2e-3
OUT_MAX_ABS = 1e-2
W_RTOL = 2e-5

CONFIGS = ["tiny", "olmoe", "decode_n1", "decode_n4", "decode_n8", "qwen3moe_shared", "skewed"]
SMALL = ["tiny", "decode_n4", "qwen3moe_shared"]
Q4K = ["tiny_q4k", "q4k_shared", "olmoe_q4k"]  # the same layer with Q4_K expert weights
Q3K = ["tiny_q3k", "q3k_shared", "olmoe_q3k"]  # and with Q3_K expert weights


@pytest.fixture(scope="module")
def ops():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mixture_experts_ffn_top_gb300 import build, ops as _ops

    build.build()
    torch.cuda.set_device(0)
    return _ops


_cache = {}


def case(name, full=True):
    """(workload, inputs, oracle results) for a named workload, cached for the module."""
    key = (name, full)
    if key not in _cache:
        wl = WORKLOADS[name]
        inp = make_inputs(wl)
        ref = O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)
        _cache[key] = (wl, inp, ref)
    return _cache[key]


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def logit_tol(ref_logits):
    row_max = np.abs(ref_logits).max(axis=1)
    row_rms = np.sqrt((ref_logits.astype(np.float64) ** 2).mean(axis=1))
    return LOGIT_RTOL * np.maximum(row_max, row_rms)


def clear_tokens(ref_logits, k):
    """Tokens whose routing is decided by more than twice the logit tolerance."""
    E = ref_logits.shape[1]
    if k >= E:
        return np.ones(ref_logits.shape[0], bool)
    srt = np.sort(ref_logits, axis=1)[:, ::-1]
    gap = srt[:, k - 1] - srt[:, k]
    return gap > 2 * logit_tol(ref_logits)


def assert_out_close(got, ref, mask=None, what="output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if mask is not None:
        got, ref = got[mask], ref[mask]
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() if got.size else 0.0
    assert rel <= OUT_REL_L2 and mx <= OUT_MAX_ABS, f"{what}: rel L2 {rel:.3e}, max abs {mx:.3e}"
    return rel, mx


def new_ws(ops, wl, N=None):
    return ops.new_workspace(N or wl.N, wl.D, wl.E, wl.F, wl.top_k, wl.Fs)


def layer_for(ops, inp, wl):
    return ops.MoeLayer.from_numpy(inp, device="cuda:0", top_k=wl.top_k, max_tokens=wl.N)


# -------------------------------------------------------------- router ----
@pytest.mark.parametrize("name", CONFIGS)
def test_router_parity(ops, name):
    wl, inp, ref = case(name)
    ws = new_ws(ops, wl)
    r = ops.moe_router_topk(dev(inp["hidden"]), dev(inp["routerW"]),
                            None if inp["shexp_gate"] is None else dev(inp["shexp_gate"]),
                            wl.top_k, wl.norm_topk_prob, ws, want_logits=True)
    assert ops.moe_workspace_status(ws) == 0
    logits = r["logits"].cpu().numpy()
    tol = logit_tol(ref["logits"])
    assert np.all(np.abs(logits - ref["logits"]) <= tol[:, None])
    clear = clear_tokens(ref["logits"], wl.top_k)
    idx = r["topk_idx"].cpu().numpy()
    np.testing.assert_array_equal(idx[clear], ref["topk_idx"][clear])
    np.testing.assert_allclose(r["topk_w"].cpu().numpy()[clear], ref["topk_w"][clear], rtol=W_RTOL, atol=1e-7)
    # Q8_1 of x: the same fp32 inputs give the same codes and scales
    np.testing.assert_array_equal(r["x_q"].cpu().numpy(), ref["x_q"])
    np.testing.assert_array_equal(r["x_d"].cpu().numpy(), O.halves(ref["x_d16"]))
    if wl.has_shared:
        np.testing.assert_allclose(r["shexp_scale"].cpu().numpy(), ref["shexp_scale"], rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("N,D,E,k,Fs,norm", [
    (1100, 512, 48, 6, 32, True),    # ragged last token tile, shared gate row
    (1024, 2048, 64, 8, 0, False),   # one full expert tile
    (1040, 256, 33, 3, 0, True),     # one expert past a 32-wide lane group
    (300, 256, 8, 2, 32, True),      # 8 experts: the tensor-core router's N padded to 16, shared gate row
    (520, 512, 24, 4, 0, False),     # 24 experts: N padded to 32 (8 zero router rows on chip)
    (130, 1024, 40, 8, 0, True),     # 40 experts, two token tiles (one of 2 rows)
])
def test_router_ragged_shapes(ops, N, D, E, k, Fs, norm):
    """Router, routing and Q8_1 of x on shapes with ragged token and expert tiles."""
    wl, inp = _random_layer(N, D, E, k, 32, Fs, norm, seed=N + E)
    ws = new_ws(ops, wl)
    gate = None if inp["shexp_gate"] is None else dev(inp["shexp_gate"])
    r = ops.moe_router_topk(dev(inp["hidden"]), dev(inp["routerW"]), gate, k, norm, ws, want_logits=True)
    assert ops.moe_workspace_status(ws) == 0
    ref_logits = O.router_logits(inp["hidden"], inp["routerW"])
    tol = logit_tol(ref_logits)
    assert np.all(np.abs(r["logits"].cpu().numpy() - ref_logits) <= tol[:, None])
    ridx, rw, _ = O.softmax_topk(ref_logits, k, norm)
    clear = clear_tokens(ref_logits, k)
    assert clear.mean() > 0.9
    np.testing.assert_array_equal(r["topk_idx"].cpu().numpy()[clear], ridx[clear])
    np.testing.assert_allclose(r["topk_w"].cpu().numpy()[clear], rw[clear], rtol=W_RTOL, atol=1e-7)
    xq, xd16, _ = O.quantize_q8_1(inp["hidden"])
    np.testing.assert_array_equal(r["x_q"].cpu().numpy(), xq)
    np.testing.assert_array_equal(r["x_d"].cpu().numpy(), O.halves(xd16))
    if Fs:
        g = O.router_logits(inp["hidden"], inp["shexp_gate"].reshape(1, D))[:, 0]
        np.testing.assert_allclose(r["shexp_scale"].cpu().numpy(), O.sigmoid(g), rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared", "skewed"])
def test_topk_from_oracle_logits_bit_exact(ops, name):
    """Given the oracle's logits, every token's routing is identical (ties to the lower index)."""
    wl, inp, ref = case(name)
    idx, w = ops.moe_topk_from_logits(dev(ref["logits"]), wl.top_k, wl.norm_topk_prob)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref["topk_idx"])
    np.testing.assert_allclose(w.cpu().numpy(), ref["topk_w"], rtol=W_RTOL, atol=1e-7)


def test_topk_ties_and_norm(ops):
    rng = np.random.default_rng(20)
    for E, k in [(8, 2), (64, 8), (256, 8), (16, 16), (1024, 32)]:
        logits = rng.integers(-2, 3, (300, E)).astype(np.float32)
        for norm in (False, True):
            ridx, rw, _ = O.softmax_topk(logits, k, norm)
            idx, w = ops.moe_topk_from_logits(dev(logits), k, norm)
            np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
            np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=W_RTOL, atol=1e-7)


def test_quantize_bit_exact(ops):
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((4096, 64)) * np.exp(rng.uniform(-10, 10, (4096, 1)))).astype(np.float32)
    x[0] = 0.0
    x[1, :32] = np.arange(32)
    x[2, 0] = 127.0
    x[2, 1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, 126.5, -3.5, 0.49999997]
    x[3, 0] = 127.0 * (1.0 + 2.0 ** -12)
    x[3, 1] = 63.5
    q, d = ops.moe_quantize_q8_1(dev(x))
    rq, rd16, _ = O.quantize_q8_1(x)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(d.cpu().numpy(), O.halves(rd16))


# ------------------------------------------------------------- bucketing ---
@pytest.mark.parametrize("name", CONFIGS)
def test_bucket_bit_exact(ops, name):
    wl, inp, ref = case(name)
    ws = new_ws(ops, wl)
    es, ti, tk = ops.moe_bucket(dev(ref["topk_idx"]), wl.E, ws)
    assert ops.moe_workspace_status(ws) == 0
    np.testing.assert_array_equal(es.cpu().numpy(), ref["expStart"])
    np.testing.assert_array_equal(ti.cpu().numpy(), ref["expTokI"])
    np.testing.assert_array_equal(tk.cpu().numpy(), ref["expTokK"])


@pytest.mark.parametrize("N,E,k", [(1, 8, 2), (3, 8, 8), (1025, 64, 8), (4096, 128, 8), (2500, 1024, 32),
                                   (7, 1, 1), (40000, 64, 8), (20000, 1024, 2)])
def test_bucket_random_shapes(ops, N, E, k):
    rng = np.random.default_rng(N + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    ws = ops.new_workspace(N, 64, E, 64, k)
    es, ti, tk = ops.moe_bucket(dev(idx), E, ws)
    assert ops.moe_workspace_status(ws) == 0
    res, rti, rtk = O.bucket(idx, E)
    np.testing.assert_array_equal(es.cpu().numpy(), res)
    np.testing.assert_array_equal(ti.cpu().numpy(), rti)
    np.testing.assert_array_equal(tk.cpu().numpy(), rtk)


@pytest.mark.parametrize("bad", ["out_of_range", "negative", "repeated"])
def test_bucket_flags_bad_routing(ops, bad):
    idx = np.array([[0, 1], [2, 3], [4, 5]], np.int32)
    if bad == "out_of_range":
        idx[1, 1] = 8
    elif bad == "negative":
        idx[2, 0] = -1
    else:
        idx[0, 1] = 0
    ws = ops.new_workspace(3, 64, 8, 64, 2)
    es, ti, tk = ops.moe_bucket(dev(idx), 8, ws)
    word = ops.moe_workspace_status(ws)
    assert word & 0x1
    assert np.all(es.cpu().numpy() == 0)  # every segment left empty
    assert ops.moe_workspace_status(ws) == 0  # cleared


def test_decode_ring_flags_malformed_csr(ops):
    """The decode matvecs check every CSR-derived index before using it: a token index past N, a
    segment outside [0, N * top_k] or a slot past top_k raises MOE_DEV_BAD_CSR (the entry or the
    segment is skipped, nothing is read out of bounds), and the same workspace gives the right
    results again once the status is read."""
    wl, inp, ref = case("decode_n4")
    layer = layer_for(ops, inp, wl)
    xq, xd = dev(ref["x_q"]), dev(O.halves(ref["x_d16"]))
    es, ti, tk = ref["expStart"], ref["expTokI"], ref["expTokK"]
    want_hq, _ = ops.moe_expert_gate_up(layer.w, xq, xd, dev(es), dev(ti), wl.top_k, layer.ws, path=1)
    assert ops.moe_workspace_status(layer.ws) == 0
    ti_bad = ti.copy()
    ti_bad[0] = wl.N + 1000
    ops.moe_expert_gate_up(layer.w, xq, xd, dev(es), dev(ti_bad), wl.top_k, layer.ws, path=1)
    assert ops.moe_workspace_status(layer.ws) & 0x2
    es_bad = es.copy()
    es_bad[1] = -1
    ops.moe_expert_gate_up(layer.w, xq, xd, dev(es_bad), dev(ti), wl.top_k, layer.ws, path=1)
    assert ops.moe_workspace_status(layer.ws) & 0x2
    total = int(es[-1])
    hq = np.zeros((wl.N * wl.top_k, wl.F), np.int8)
    hd = np.zeros((wl.N * wl.top_k, wl.F // 32), np.float32)
    hq[:total] = ref["h_q"]
    hd[:total] = O.halves(ref["h_d16"])
    tk_bad = tk.copy()
    tk_bad[0] = wl.top_k + 3
    ops.moe_expert_down(layer.w, dev(hq), dev(hd), dev(es), dev(ti), dev(tk_bad), wl.N, wl.top_k, layer.ws, path=1)
    assert ops.moe_workspace_status(layer.ws) & 0x2
    # the workspace is still good
    got_hq, _ = ops.moe_expert_gate_up(layer.w, xq, xd, dev(es), dev(ti), wl.top_k, layer.ws, path=1)
    assert ops.moe_workspace_status(layer.ws) == 0
    np.testing.assert_array_equal(got_hq.cpu().numpy(), want_hq.cpu().numpy())


def test_bucket_flags_bad_routing_in_a_late_range(ops):
    # many CTAs: the bad entry sits in the last token range, far from CTA 0
    N, E, k = 5000, 64, 8
    rng = np.random.default_rng(7)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(N)]).astype(np.int32)
    idx[N - 1, 3] = idx[N - 1, 0]
    ws = ops.new_workspace(N, 64, E, 64, k)
    es, ti, tk = ops.moe_bucket(dev(idx), E, ws)
    assert ops.moe_workspace_status(ws) & 0x1
    assert np.all(es.cpu().numpy() == 0)
    # the barrier words are back at rest: a clean call on the same workspace works
    idx[N - 1, 3] = (idx[N - 1, 0] + E // 2) % E if (idx[N - 1, 0] + E // 2) % E not in idx[N - 1] else \
        next(e for e in range(E) if e not in idx[N - 1])
    es, ti, tk = ops.moe_bucket(dev(idx), E, ws)
    assert ops.moe_workspace_status(ws) == 0
    res, rti, rtk = O.bucket(idx, E)
    np.testing.assert_array_equal(es.cpu().numpy(), res)
    np.testing.assert_array_equal(ti.cpu().numpy(), rti)


# ------------------------------------------------------ grouped experts ---
def _csr(ref):
    return dev(ref["expStart"]), dev(ref["expTokI"]), dev(ref["expTokK"])


Q8_FULL = ["tiny", "qwen3moe_shared", "olmoe", "skewed"]  # Q8_0 workloads checked on every dot


def _check_blocks(nblk):
    """The first, second, a middle and the last block."""
    return sorted({0, 1, nblk // 2 + 1, nblk - 1})


@pytest.mark.parametrize("name", Q8_FULL)
@pytest.mark.parametrize("path", [1, 2])
def test_gate_up_block_dots_every_entry(ops, name, path):
    """Every CSR entry x every feature x both matrices, four blocks: bit-exact against the
    oracle's integer block dots."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    xq, xd = dev(ref["x_q"]), dev(O.halves(ref["x_d16"]))
    total = int(ref["expStart"][-1])
    for block in _check_blocks(wl.D // 32):
        dots = ops.moe_debug_gate_up_block_dots(layer.w, xq, xd, es, ti, wl.top_k, block, layer.ws, path=path)
        assert ops.moe_workspace_status(layer.ws) == 0
        dots = dots.cpu().numpy()[:total]
        for mat, W in ((0, inp["gate"]), (1, inp["up"])):
            rd = O.block_dots_csr(W, ref["x_q"], ref["expStart"], ref["expTokI"], block)
            bad = np.argwhere(dots[:, mat, :] != rd)
            assert bad.size == 0, (block, mat, bad[:5].tolist())


@pytest.mark.parametrize("name", Q8_FULL)
@pytest.mark.parametrize("path", [1, 2])
def test_down_block_dots_every_entry(ops, name, path):
    """The down GEMM's int32 block dots on the oracle's h_q: every entry x every output column,
    four blocks, bit-exact."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    total = int(ref["expStart"][-1])
    hq = np.zeros((wl.N * wl.top_k, wl.F), np.int8)
    hd = np.zeros((wl.N * wl.top_k, wl.F // 32), np.float32)
    hq[:total] = ref["h_q"]
    hd[:total] = O.halves(ref["h_d16"])
    for block in _check_blocks(wl.F // 32):
        dots = ops.moe_debug_down_block_dots(layer.w, dev(hq), dev(hd), es, ti, tk, wl.N, wl.top_k, block,
                                             layer.ws, path=path)
        assert ops.moe_workspace_status(layer.ws) == 0
        rd = O.block_dots_csr(inp["down"], ref["h_q"], ref["expStart"], None, block)
        got = dots.cpu().numpy()[:total]
        bad = np.argwhere(got != rd)
        assert bad.size == 0, (block, bad[:5].tolist())


def _decode_case(name):
    """Decode batches (at most 8 tokens: the matvec path streams the weights through its ring):
    the OLMoE-shaped Q8_0 workloads, and K-quant layers of the same batch sizes."""
    if name in WORKLOADS:
        return case(name)
    wfmt, n = name.split("_n")
    wl = Workload(name, N=int(n), D=512, E=16, top_k=4, F=256, Fs=256, norm_topk_prob=True, seed=80 + int(n),
                  wfmt=wfmt)
    inp = make_inputs(wl)
    return wl, inp, O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)


def _row_dots(wfmt, w_row, act_row):
    if wfmt == "q4_k":
        return O.block_dots_q4_k(w_row, act_row)
    if wfmt == "q3_k":  # the library stores the codes -s_j*q_i
        return -O.block_dots_q3_k(w_row, act_row)
    return O.block_dots(w_row, act_row)


@pytest.mark.parametrize("name", ["decode_n1", "decode_n8", "q4_k_n1", "q4_k_n8", "q3_k_n8"])
def test_decode_block_dots_every_entry(ops, name):
    """The decode matvecs (Q4_K from its nibble-packed copy): every CSR entry x every row of
    gate, up and down, three blocks, bit-exact against the oracle's integer block dots."""
    wl, inp, ref = _decode_case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    total = int(ref["expStart"][-1])
    xq, xd = dev(ref["x_q"]), dev(O.halves(ref["x_d16"]))
    ent_e = np.searchsorted(ref["expStart"], np.arange(total), side="right") - 1
    gu_blocks = sorted({0, wl.D // 64 + 1, wl.D // 32 - 1})
    gu = {b: ops.moe_debug_gate_up_block_dots(layer.w, xq, xd, es, ti, wl.top_k, b, layer.ws, path=1)
          .cpu().numpy()[:total] for b in gu_blocks}
    assert ops.moe_workspace_status(layer.ws) == 0
    hq = np.zeros((wl.N * wl.top_k, wl.F), np.int8)
    hd = np.zeros((wl.N * wl.top_k, wl.F // 32), np.float32)
    hq[:total] = ref["h_q"]
    hd[:total] = O.halves(ref["h_d16"])
    dn_blocks = sorted({0, wl.F // 64 + 1, wl.F // 32 - 1})
    dn = {b: ops.moe_debug_down_block_dots(layer.w, dev(hq), dev(hd), es, ti, tk, wl.N, wl.top_k, b, layer.ws,
                                           path=1).cpu().numpy()[:total] for b in dn_blocks}
    assert ops.moe_workspace_status(layer.ws) == 0
    for j in range(total):
        e, t = int(ent_e[j]), int(ref["expTokI"][j])
        for mat, W in ((0, inp["gate"]), (1, inp["up"])):
            want = np.stack([_row_dots(wl.wfmt, W[e, f], ref["x_q"][t]) for f in range(wl.F)])
            for b in gu_blocks:
                bad = np.argwhere(gu[b][j, mat] != want[:, b])
                assert bad.size == 0, (j, mat, b, bad[:5].tolist())
        want = np.stack([_row_dots(wl.wfmt, inp["down"][e, c], ref["h_q"][j]) for c in range(wl.D)])
        for b in dn_blocks:
            bad = np.argwhere(dn[b][j] != want[:, b])
            assert bad.size == 0, (j, b, bad[:5].tolist())


@pytest.mark.parametrize("name", ["tiny_q4k", "olmoe_q4k", "tiny_q3k", "olmoe_q3k"])
@pytest.mark.parametrize("path", [1, 2])
def test_gate_up_block_dots_bit_exact(ops, name, path):
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    ws = layer.ws
    es, ti, tk = _csr(ref)
    xq, xd = dev(ref["x_q"]), dev(O.halves(ref["x_d16"]))
    nblk = wl.D // 32
    rows = np.arange(ref["expStart"][-1])
    rng = np.random.default_rng(0)
    sample = rng.choice(rows, size=min(64, len(rows)), replace=False)
    for block in sorted({0, nblk // 2 + 1, nblk - 1}):
        dots = ops.moe_debug_gate_up_block_dots(layer.w, xq, xd, es, ti, wl.top_k, block, ws, path=path)
        assert ops.moe_workspace_status(ws) == 0
        dots = dots.cpu().numpy()
        for j in sample:
            e = int(np.searchsorted(ref["expStart"], j, side="right") - 1)
            t = int(ref["expTokI"][j])
            for mat, W in ((0, inp["gate"]), (1, inp["up"])):
                for f in sorted({0, 1, 31, 32, 63, 64, wl.F // 2 + 3, wl.F - 1}):
                    if wl.wfmt == "q4_k":
                        ref_dot = O.block_dots_q4_k(W[e, f], ref["x_q"][t])[block]
                    elif wl.wfmt == "q3_k":  # the library stores the codes -s_j*q_i
                        ref_dot = -O.block_dots_q3_k(W[e, f], ref["x_q"][t])[block]
                    else:
                        ref_dot = O.block_dots(W[e, f], ref["x_q"][t])[block]
                    assert dots[j, mat, f] == ref_dot, (j, mat, f, block)


@pytest.mark.parametrize("name", SMALL + ["olmoe", "skewed"] + Q4K + Q3K)
@pytest.mark.parametrize("path", [1, 2])
def test_gate_up_requantised_activations(ops, name, path):
    """h_q from the oracle's x_q and CSR: codes within +-1 (fp32 vs double accumulation can
    move a value across a rounding boundary), at most 1% of them different."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    hq, hd = ops.moe_expert_gate_up(layer.w, dev(ref["x_q"]), dev(O.halves(ref["x_d16"])), es, ti, wl.top_k,
                                    layer.ws, path=path)
    assert ops.moe_workspace_status(layer.ws) == 0
    total = int(ref["expStart"][-1])
    hq = hq.cpu().numpy()[:total].astype(np.int32)
    hd = hd.cpu().numpy()[:total]
    rq = ref["h_q"].astype(np.int32)
    diff = np.abs(hq - rq)
    assert diff.max() <= 1
    assert (diff > 0).mean() <= 0.01
    rd = O.halves(ref["h_d16"])
    np.testing.assert_allclose(hd, rd, rtol=1e-3, atol=1e-30)


def _abs_dot_bound(Wd, hq, hd, ref, wl):
    """sum_i |w[e][c][i]| * |h[j][i]| for every CSR entry j (rows in entry order) and output
    column c, from the dequantised Q8_0 down weights and the requantised activations."""
    E, D, F = wl.E, wl.D, wl.F
    out = np.zeros((hq.shape[0], D))
    habs = np.abs(hq.astype(np.float64)) * np.repeat(hd.astype(np.float64), 32, axis=1)
    es = ref["expStart"]
    for e in range(E):
        a, b = int(es[e]), int(es[e + 1])
        if a == b:
            continue
        blk = Wd[e].reshape(D, F // 32, Q8_0_BYTES)
        d = O.halves(blk[:, :, :2].copy().view(np.uint16)[..., 0]).astype(np.float64)
        q = blk[:, :, 2:].view(np.int8).astype(np.float64)
        wabs = np.abs(q * d[..., None]).reshape(D, F)
        out[a:b] = habs[a:b] @ wabs.T
    return out


@pytest.mark.parametrize("name", SMALL + ["olmoe", "skewed"] + Q4K + Q3K)
@pytest.mark.parametrize("path", [1, 2])
def test_down_given_oracle_h(ops, name, path):
    """The down half on the oracle's own h_q: partials to fp32 accumulation accuracy."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    total = int(ref["expStart"][-1])
    hq = np.zeros((wl.N * wl.top_k, wl.F), np.int8)
    hd = np.zeros((wl.N * wl.top_k, wl.F // 32), np.float32)
    hq[:total] = ref["h_q"]
    hd[:total] = O.halves(ref["h_d16"])
    part = ops.moe_expert_down(layer.w, dev(hq), dev(hd), es, ti, tk, wl.N, wl.top_k, layer.ws, path=path)
    assert ops.moe_workspace_status(layer.ws) == 0
    got = part.cpu().numpy().astype(np.float64)
    r = ref["partials"].astype(np.float64)
    rel = np.linalg.norm(got - r) / np.linalg.norm(r)
    assert rel <= 1e-5, rel
    # element-wise: the kernel adds F/32 exact block terms in fp32 (one rounding each), the oracle
    # rounds its double sum once, so |got - ref| <= (F/32 + 2) * 2^-24 * sum_b |term_b|, and
    # sum_b |term_b| <= sum_i |w_i| * |h_i| (dequantised); the K-quant min terms double the count
    if wl.wfmt == "q8_0":
        bound = (wl.F // 32 + 2) * 2.0 ** -24 * _abs_dot_bound(inp["down"], hq[:total], hd[:total], ref, wl)
        rows = (ref["expTokI"].astype(np.int64) * wl.top_k + ref["expTokK"])
        err = np.abs(got[rows] - r[rows])
        assert (err <= bound).all(), float((err / np.maximum(bound, 1e-300)).max())
    else:
        err = np.abs(got - r)
        assert (err <= 2 * (2 * wl.F // 32 + 2) * 2.0 ** -24 * np.abs(r).max(axis=1, keepdims=True) * 8).all()


@pytest.mark.parametrize("name", SMALL + ["olmoe", "skewed"] + Q4K + Q3K)
@pytest.mark.parametrize("path", [1, 2])
def test_grouped_ffn_partials(ops, name, path):
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    es, ti, tk = _csr(ref)
    sh = dev(ref["shexp_scale"]) if wl.has_shared else None
    part, shared = ops.moe_grouped_ffn(layer.w, dev(ref["x_q"]), dev(O.halves(ref["x_d16"])), es, ti, tk,
                                       wl.top_k, layer.ws, shexp_scale=sh, path=path)
    assert ops.moe_workspace_status(layer.ws) == 0
    assert_out_close(part.cpu().numpy(), ref["partials"], what="partials")
    if wl.has_shared:
        assert_out_close(shared.cpu().numpy(), ref["shared_out"], what="shared expert")


# -------------------------------------------------------------- combine ---
@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared"])
def test_combine_bit_exact(ops, name):
    wl, inp, ref = case(name)
    S = dev(ref["shared_out"]) if wl.has_shared else None
    out = ops.moe_combine(dev(ref["partials"]), dev(ref["topk_w"]), S)
    np.testing.assert_array_equal(out.cpu().numpy(), ref["out"])


def test_combine_order_sensitive_values(ops):
    """Values where the slot order, the fma and the shared-last order each change the bits."""
    p = np.zeros((4 * 3, 4), np.float32)
    w = np.ones((4, 3), np.float32)
    S = np.zeros((4, 4), np.float32)
    p[0:3, 0] = [2.0 ** 24, 1.0, 1.0]                       # slot order
    a = np.float32(1.0 + 2.0 ** -12)
    p[3:6, 0] = [-1.0, a, 0.0]
    w[1] = [1.0, a, 1.0]                                   # fma
    p[6:9, 0] = [1.0, 2.0 ** 24, 0.0]
    S[2, 0] = 1.0                                          # shared last
    rng = np.random.default_rng(3)
    p[9:12] = rng.standard_normal((3, 4)).astype(np.float32)
    w[3] = rng.standard_normal(3).astype(np.float32)
    out = ops.moe_combine(dev(p), dev(w), dev(S)).cpu().numpy()
    np.testing.assert_array_equal(out, O.combine(p, w, S))
    assert out[0, 0] == 2.0 ** 24 and out[1, 0] == 2.0 ** -11 + 2.0 ** -24 and out[2, 0] == 2.0 ** 24


@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared"])
def test_combine_residual_bit_exact(ops, name):
    """(routed + shared) + resid against the oracle, out of place and in place (out = residual)."""
    wl, inp, ref = case(name)
    R = np.random.default_rng(31).standard_normal((wl.N, wl.D)).astype(np.float32)
    S = dev(ref["shared_out"]) if wl.has_shared else None
    want = O.combine(ref["partials"], ref["topk_w"], ref["shared_out"] if wl.has_shared else None, R)
    out = ops.moe_combine_residual(dev(ref["partials"]), dev(ref["topk_w"]), S, dev(R))
    np.testing.assert_array_equal(out.cpu().numpy(), want)
    r_dev = dev(R)
    ops.moe_combine_residual(dev(ref["partials"]), dev(ref["topk_w"]), S, r_dev, out=r_dev)
    np.testing.assert_array_equal(r_dev.cpu().numpy(), want)


def test_combine_residual_order_sensitive_values(ops):
    """1 + 2^-24 ties to even before the residual 2^-23 is added: 1 + 2^-23, not 1 + 2^-22."""
    p = np.zeros((2, 4), np.float32)
    p[0, 0] = 1.0
    w = np.ones((2, 1), np.float32)
    S = np.zeros((2, 4), np.float32)
    S[0, 0] = 2.0 ** -24
    R = np.zeros((2, 4), np.float32)
    R[0, 0] = 2.0 ** -23
    R[1] = [1.0, -2.0, 3.5, -0.0]
    out = ops.moe_combine_residual(dev(p), dev(w), dev(S), dev(R)).cpu().numpy()
    np.testing.assert_array_equal(out, O.combine(p, w, S, R))
    assert out[0, 0] == 1.0 + 2.0 ** -23


@pytest.mark.parametrize("name", ["tiny", "qwen3moe_shared", "olmoe"])
def test_layer_with_residual(ops, name):
    """moe_ffn_prefill_residual = the layer output plus the residual row, bit for bit, also in place."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    R = torch.from_numpy(np.random.default_rng(32).standard_normal((wl.N, wl.D)).astype(np.float32)).cuda()
    plain = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob)
    want = (plain + R).cpu().numpy()
    got = ops.moe_ffn_prefill_residual(layer.w, dev(inp["hidden"]), layer.routerW, layer.shexp_gate, R, wl.top_k,
                                       wl.norm_topk_prob, layer.ws)
    assert layer.status() == 0
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    ops.moe_ffn_prefill_residual(layer.w, dev(inp["hidden"]), layer.routerW, layer.shexp_gate, R, wl.top_k,
                                 wl.norm_topk_prob, layer.ws, out=R)
    np.testing.assert_array_equal(R.cpu().numpy(), want)


# RMSNorm of the combined row: out is bit-exact, and only the row's factor r = 1/sqrt(ms + eps) carries
# rounding.  The kernel sums the squares in fp32: D/128 terms per thread (128 threads per row; D/512
# with 512), a 5-level warp butterfly, at most 16 warps in order, so the sum is within
# 2^-24 * (D/128 + 21) relative, r within half that plus 3 ulps (/D, + eps, square root, divide), and
# normed two products more: |normed - ref| <= 2e-6 * |ref| elementwise for D <= 4096 against the
# oracle's double evaluation.
NORM_RTOL = 2e-6


def _gamma(D, seed):
    return (1.0 + 0.25 * np.random.default_rng(seed).standard_normal(D)).astype(np.float32)


def _assert_normed(got, want):
    err = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bound = NORM_RTOL * np.abs(want.astype(np.float64))
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (bad[:5].tolist(), float((err / np.maximum(np.abs(want), 1e-30)).max()))


@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared"])
def test_combine_residual_rmsnorm_against_oracle(ops, name):
    """The combine with residual (bit-exact) and the next layer's RMSNorm of it (within NORM_RTOL of
    the oracle's double evaluation), out of place and in place (out = residual)."""
    wl, inp, ref = case(name)
    R = np.random.default_rng(33).standard_normal((wl.N, wl.D)).astype(np.float32)
    gamma = _gamma(wl.D, 34)
    S_np = ref["shared_out"] if wl.has_shared else None
    want_out, want_norm = O.combine_residual_rmsnorm(ref["partials"], ref["topk_w"], S_np, R, gamma, 1e-6)
    S = dev(S_np) if wl.has_shared else None
    out, normed = ops.moe_combine_residual_rmsnorm(dev(ref["partials"]), dev(ref["topk_w"]), S, dev(R), dev(gamma),
                                                   1e-6)
    np.testing.assert_array_equal(out.cpu().numpy(), want_out)
    _assert_normed(normed.cpu().numpy(), want_norm)
    r_dev = dev(R)
    _, normed2 = ops.moe_combine_residual_rmsnorm(dev(ref["partials"]), dev(ref["topk_w"]), S, r_dev, dev(gamma),
                                                  1e-6, out=r_dev)
    np.testing.assert_array_equal(r_dev.cpu().numpy(), want_out)
    np.testing.assert_array_equal(normed2.cpu().numpy(), normed.cpu().numpy())


def test_combine_rmsnorm_edge_rows(ops):
    """Constant rows (normed = sign * gamma up to the factor's rounding), a zero row (normed = 0,
    eps keeps it finite), a huge and a tiny row (no overflow or underflow in the sum of squares at
    these magnitudes), a ragged width (D = 260: 65 float4 columns over 128 threads), top_k = 3 (the
    generic slot loop)."""
    D, k = 260, 3
    rows = np.zeros((5, D), np.float32)
    rows[0] = 3.0
    rows[1] = -0.5
    rows[3] = np.random.default_rng(35).standard_normal(D).astype(np.float32) * 1e15
    rows[4] = np.random.default_rng(36).standard_normal(D).astype(np.float32) * 1e-15
    p = np.zeros((5 * k, D), np.float32)
    p[0::k] = rows  # slot 0 carries the row, weight 1; slots 1, 2 weight 0
    w = np.zeros((5, k), np.float32)
    w[:, 0] = 1.0
    R = np.zeros((5, D), np.float32)
    gamma = _gamma(D, 37)
    want_out, want_norm = O.combine_residual_rmsnorm(p, w, None, R, gamma, 1e-12)
    out, normed = ops.moe_combine_residual_rmsnorm(dev(p), dev(w), None, dev(R), dev(gamma), 1e-12)
    np.testing.assert_array_equal(out.cpu().numpy(), want_out)
    got = normed.cpu().numpy()
    _assert_normed(got, want_norm)
    assert not np.any(got[2])  # the zero row
    assert np.all(np.isfinite(got))


def test_combine_rmsnorm_rejects_bad_arguments(ops):
    p = dev(np.ones((4, 8), np.float32))
    w = dev(np.ones((4, 1), np.float32))
    R = dev(np.zeros((4, 8), np.float32))
    g = dev(np.ones(8, np.float32))
    for eps in (0.0, -1e-6, float("inf"), float("nan")):
        with pytest.raises(ops.MoeError):
            ops.moe_combine_residual_rmsnorm(p, w, None, R, g, eps)
    out = torch.empty((4, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(ops.MoeError):
        ops.moe_combine_residual_rmsnorm(p, w, None, R, g, 1e-6, out=out, normed=out)
    with pytest.raises(ops.MoeError):
        ops.moe_combine_residual_rmsnorm(p, w, None, R, g, 1e-6, normed=R)


@pytest.mark.parametrize("name,path", [("tiny", 0), ("olmoe", 0), ("qwen3moe_shared", 0), ("decode_n4", 0),
                                       ("tiny", 2)])
def test_layer_with_residual_rmsnorm(ops, name, path):
    """moe_ffn_prefill_residual_rmsnorm: out equals moe_ffn_prefill_residual's bit for bit (also in
    place), and normed is the RMSNorm of that out within NORM_RTOL of the oracle."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    R = np.random.default_rng(38).standard_normal((wl.N, wl.D)).astype(np.float32)
    gamma = _gamma(wl.D, 39)
    want = ops.moe_ffn_prefill_residual(layer.w, dev(inp["hidden"]), layer.routerW, layer.shexp_gate, dev(R),
                                        wl.top_k, wl.norm_topk_prob, layer.ws, path=path).cpu().numpy()
    out, normed = ops.moe_ffn_prefill_residual_rmsnorm(layer.w, dev(inp["hidden"]), layer.routerW, layer.shexp_gate,
                                                       dev(R), dev(gamma), 1e-5, wl.top_k, wl.norm_topk_prob,
                                                       layer.ws, path=path)
    assert layer.status() == 0
    np.testing.assert_array_equal(out.cpu().numpy(), want)
    ones = np.ones((wl.N, 1), np.float32)
    _, want_norm = O.combine_residual_rmsnorm(want, ones, None, np.zeros_like(want), gamma, 1e-5)
    _assert_normed(normed.cpu().numpy(), want_norm)
    r_dev = dev(R)
    ops.moe_ffn_prefill_residual_rmsnorm(layer.w, dev(inp["hidden"]), layer.routerW, layer.shexp_gate, r_dev,
                                         dev(gamma), 1e-5, wl.top_k, wl.norm_topk_prob, layer.ws, out=r_dev, path=path)
    assert layer.status() == 0
    np.testing.assert_array_equal(r_dev.cpu().numpy(), want)


# ---------------------------------------------------------- whole layer ---
@pytest.mark.parametrize("name", CONFIGS + Q4K + Q3K)
@pytest.mark.parametrize("path", [0, 1, 2])
def test_layer_parity(ops, name, path):
    """moe_ffn_prefill (the call bench.py times, path 0 = its launch configuration)."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    out = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=path)
    assert layer.status() == 0
    clear = clear_tokens(ref["logits"], wl.top_k)
    v = layer.views(wl.N)
    np.testing.assert_array_equal(v["topk_idx"].cpu().numpy()[clear], ref["topk_idx"][clear])
    rel, mx = assert_out_close(out.cpu().numpy(), ref["out"], clear, what=f"{name} layer output")
    assert clear.mean() > 0.95  # near-tied tokens are few (E=256 has the most)


@pytest.mark.parametrize("name", ["decode_n1", "decode_n4", "decode_n8", "tiny"])
@pytest.mark.parametrize("path", [1, 2])
def test_layer_routing_state(ops, name, path):
    """The routing a layer call leaves in its workspace (one fused launch for batches of at most
    8 tokens on the matvec path, the general router and bucketing otherwise): indices, weights,
    Q8_1 of x and the CSR equal the oracle's where the routing is decided."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=path)
    assert layer.status() == 0
    v = layer.views(wl.N)
    clear = clear_tokens(ref["logits"], wl.top_k)
    np.testing.assert_array_equal(v["topk_idx"].cpu().numpy()[clear], ref["topk_idx"][clear])
    np.testing.assert_allclose(v["topk_w"].cpu().numpy()[clear], ref["topk_w"][clear], rtol=W_RTOL, atol=1e-7)
    np.testing.assert_array_equal(v["x_q"].cpu().numpy(), ref["x_q"])
    np.testing.assert_array_equal(v["x_d"].cpu().numpy(), O.halves(ref["x_d16"]))
    if clear.all():
        np.testing.assert_array_equal(v["expStart"].cpu().numpy(), ref["expStart"])
        total = int(ref["expStart"][-1])
        np.testing.assert_array_equal(v["expTokI"].cpu().numpy()[:total], ref["expTokI"])
        np.testing.assert_array_equal(v["expTokK"].cpu().numpy()[:total], ref["expTokK"])
    # a second call on the same workspace (the arrival counter is back at zero) gives the same state
    idx1 = v["topk_idx"].cpu().numpy().copy()
    es1 = v["expStart"].cpu().numpy().copy()
    layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=path)
    assert layer.status() == 0
    np.testing.assert_array_equal(v["topk_idx"].cpu().numpy(), idx1)
    np.testing.assert_array_equal(v["expStart"].cpu().numpy(), es1)


@pytest.mark.parametrize("name", ["olmoe", "qwen3moe_shared", "skewed", "tiny"])
def test_layer_csr_equals_bucketing_of_its_routing(ops, name):
    """The CSR a tensor-path layer call leaves (for these shapes the router writes the bucketing's
    count table and the bucketing runs without its histogram pass): bit-exact against the oracle's
    counting sort of the routing the same call produced (integer work, every token)."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=2)
    assert layer.status() == 0
    v = layer.views(wl.N)
    idx = v["topk_idx"].cpu().numpy().astype(np.int32)
    es, ti, tk = O.bucket(idx, wl.E)
    total = int(es[-1])
    assert total == wl.N * wl.top_k
    np.testing.assert_array_equal(v["expStart"].cpu().numpy(), es)
    np.testing.assert_array_equal(v["expTokI"].cpu().numpy()[:total], ti)
    np.testing.assert_array_equal(v["expTokK"].cpu().numpy()[:total], tk)


def _random_layer(N, D, E, k, F, Fs, norm, seed):
    wl = Workload(f"rand{seed}", N=N, D=D, E=E, top_k=k, F=F, Fs=Fs, norm_topk_prob=norm, seed=seed)
    return wl, make_inputs(wl)


@pytest.mark.parametrize("N,D,E,k,F,Fs,norm", [
    (1, 256, 8, 2, 128, 0, False),      # a single token
    (3, 256, 8, 8, 128, 0, True),       # k = E: every expert selected
    (130, 256, 16, 4, 192, 64, True),   # ragged N and F, shared expert
    (77, 512, 32, 1, 64, 0, False),     # top-1
    (5, 64, 4, 2, 32, 32, False),       # minimal blocks
])
def test_layer_edge_shapes(ops, N, D, E, k, F, Fs, norm):
    wl, inp = _random_layer(N, D, E, k, F, Fs, norm, seed=N * 31 + E)
    ref = O.moe_ffn_inputs(inp, k, norm)
    layer = layer_for(ops, inp, wl)
    for path in (0, 1, 2):
        if path == 2 and not ops.moe_weights_tensor_path(layer.w):
            continue
        out = layer.prefill(dev(inp["hidden"]), k, norm, path=path)
        assert layer.status() == 0
        clear = clear_tokens(ref["logits"], k)
        assert_out_close(out.cpu().numpy(), ref["out"], clear, what=f"edge N={N} E={E} k={k}")


@pytest.mark.parametrize("name", ["tiny", "qwen3moe_shared", "decode_n4"])
def test_prefill_host_buffers_match_device_buffers(ops, name):
    """The host-buffer entry point reads hidden and writes out in place: same kernels, same bits."""
    wl, inp, ref = case(name)
    layer = layer_for(ops, inp, wl)
    want = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob).cpu().numpy()
    h_host = torch.from_numpy(inp["hidden"]).pin_memory()
    o_host = torch.full((wl.N, wl.D), float("nan"), dtype=torch.float32).pin_memory()
    ops.moe_ffn_prefill_host(layer.w, h_host, layer.routerW, layer.shexp_gate, wl.top_k, wl.norm_topk_prob,
                             layer.ws, o_host)
    torch.cuda.synchronize()
    assert layer.status() == 0
    np.testing.assert_array_equal(o_host.numpy(), want)
    assert_out_close(o_host.numpy(), ref["out"], clear_tokens(ref["logits"], wl.top_k), what=f"{name} host buffers")


def test_prefill_host_rejects_device_memory(ops):
    wl, inp, _ = case("tiny")
    layer = layer_for(ops, inp, wl)
    h_dev = dev(inp["hidden"])
    o_host = torch.empty((wl.N, wl.D), dtype=torch.float32).pin_memory()
    assert not ops.moe_host_memory_addressable(h_dev)
    rc = ops.lib().moe_ffn_prefill_host(layer.w.handle, ops._P(h_dev.data_ptr()), ops._P(layer.routerW.data_ptr()),
                                        None, wl.N, wl.top_k, int(wl.norm_topk_prob), ops._P(o_host.data_ptr()), 0,
                                        ops._P(layer.ws.data_ptr()), layer.ws.numel(),
                                        ops._P(torch.cuda.current_stream().cuda_stream))
    assert rc == -1


def test_prefill_host_pageable_memory_where_addressable(ops):
    """Pageable host memory works exactly where the device walks the host page tables."""
    wl, inp, _ = case("tiny")
    layer = layer_for(ops, inp, wl)
    h_pg = torch.from_numpy(inp["hidden"].copy())
    o_pg = torch.full((wl.N, wl.D), float("nan"), dtype=torch.float32)
    if ops.moe_host_memory_addressable(h_pg) and ops.moe_host_memory_addressable(o_pg):
        ops.moe_ffn_prefill_host(layer.w, h_pg, layer.routerW, None, wl.top_k, wl.norm_topk_prob, layer.ws, o_pg)
        torch.cuda.synchronize()
        want = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob).cpu().numpy()
        np.testing.assert_array_equal(o_pg.numpy(), want)
    else:
        with pytest.raises(ops.MoeError):
            ops.moe_ffn_prefill_host(layer.w, h_pg, layer.routerW, None, wl.top_k, wl.norm_topk_prob, layer.ws, o_pg)


def test_q4_k_weights_handle_and_shapes(ops):
    """The handle reports its format; Q4_K needs D, F, Fs multiples of 256 (UNSUPPORTED_SHAPE otherwise)."""
    wl, inp, _ = case("tiny_q4k")
    layer = layer_for(ops, inp, wl)
    assert ops.moe_weights_format(layer.w) == "q4_k"
    wl8, inp8, _ = case("tiny")
    assert ops.moe_weights_format(layer_for(ops, inp8, wl8).w) == "q8_0"
    g = torch.zeros((2, 128, 144), dtype=torch.uint8, device="cuda")  # D = 256 but F = 128
    d = torch.zeros((2, 256, 72), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MoeError) as e:
        ops.MoeWeights(g, g, d, 2, 256, 128, wfmt="q4_k")
    assert e.value.code == -2


def test_q3_k_weights_handle_and_shapes(ops):
    wl, inp, _ = case("tiny_q3k")
    assert ops.moe_weights_format(layer_for(ops, inp, wl).w) == "q3_k"
    g = torch.zeros((2, 128, 110), dtype=torch.uint8, device="cuda")  # D = 256 but F = 128
    d = torch.zeros((2, 256, 55), dtype=torch.uint8, device="cuda")
    with pytest.raises(ops.MoeError) as e:
        ops.MoeWeights(g, g, d, 2, 256, 128, wfmt="q3_k")
    assert e.value.code == -2


@pytest.mark.parametrize("path", [1, 2])
def test_q3_k_extreme_codes(ops, path):
    """Rows whose every value is q = -4 with s = -32 (s*q = 128, one past int8: the library
    stores the negated codes): block dots exact and the layer within tolerance."""
    wl = WORKLOADS["tiny_q3k"]
    inp = dict(make_inputs(wl))
    ext = np.zeros(110, np.uint8)
    ext[108:110] = np.array([np.float16(2.0 ** -12)]).view(np.uint8)
    for key in ("gate", "up", "down"):
        inp[key] = inp[key].copy()
        v = inp[key].reshape(inp[key].shape[0], inp[key].shape[1], -1, 110)
        v[:, ::5] = ext  # every fifth row of every expert
    ref = O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)
    layer = layer_for(ops, inp, wl)
    es, ti, _ = _csr(ref)
    dots = ops.moe_debug_gate_up_block_dots(layer.w, dev(ref["x_q"]), dev(O.halves(ref["x_d16"])), es, ti,
                                            wl.top_k, 1, layer.ws, path=path).cpu().numpy()
    for j in range(0, int(ref["expStart"][-1]), 7):
        e = int(np.searchsorted(ref["expStart"], j, side="right") - 1)
        t = int(ref["expTokI"][j])
        for f in (0, 5, 1, wl.F - 1):
            assert dots[j, 0, f] == -O.block_dots_q3_k(inp["gate"][e, f], ref["x_q"][t])[1]
    out = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=path)
    assert layer.status() == 0
    assert_out_close(out.cpu().numpy(), ref["out"], clear_tokens(ref["logits"], wl.top_k), what="q3_k extreme")


def test_device_host_numa_node(ops):
    """The host node the device reports exists on the host (or -1: no NUMA placement)."""
    import os
    node = ops.moe_device_host_numa_node()
    assert node >= -1
    if node >= 0 and os.path.isdir("/sys/devices/system/node"):
        assert os.path.isdir(f"/sys/devices/system/node/node{node}")


@pytest.mark.parametrize("wfmt", ["q4_k", "q3_k"])
@pytest.mark.parametrize("N", [1, 3, 8])
def test_kquant_decode_batches(ops, wfmt, N):
    """K-quant weights at decode batch sizes (the matvec kernels' narrow-chunk variants, the
    one-launch routing, the shared expert's single chunk): layer output and CSR against the oracle."""
    wl = Workload(f"{wfmt}_dec{N}", N=N, D=512, E=16, top_k=4, F=256, Fs=256, norm_topk_prob=True, seed=70 + N,
                  wfmt=wfmt)
    inp = make_inputs(wl)
    ref = O.moe_ffn_inputs(inp, wl.top_k, wl.norm_topk_prob)
    layer = layer_for(ops, inp, wl)
    clear = clear_tokens(ref["logits"], wl.top_k)
    for path in (0, 1):
        out = layer.prefill(dev(inp["hidden"]), wl.top_k, wl.norm_topk_prob, path=path)
        assert layer.status() == 0
        assert_out_close(out.cpu().numpy(), ref["out"], clear, what=f"{wfmt} N={N} path {path}")
        if clear.all():
            v = layer.views(wl.N)
            np.testing.assert_array_equal(v["expStart"].cpu().numpy(), ref["expStart"])


def test_zero_hidden_gives_zero(ops):
    wl, inp = _random_layer(16, 256, 8, 2, 128, 64, False, seed=5)
    inp["hidden"][:] = 0.0
    layer = layer_for(ops, inp, wl)
    out = layer.prefill(dev(inp["hidden"]), 2, False)
    assert layer.status() == 0
    assert torch.count_nonzero(out).item() == 0


# ---------------------------------------------------------- layer stacks ---
def _stack_layers(ops, wl, n):
    from dataclasses import replace

    inps = [make_inputs(replace(wl, seed=wl.seed + 100 * l)) for l in range(n)]
    layers = [layer_for(ops, inp, wl) for inp in inps]
    return inps, layers


@pytest.mark.parametrize("name,n", [("tiny", 3), ("olmoe", 2), ("qwen3moe_shared", 2), ("decode_n4", 3)])
def test_layer_stack_equals_sequential_calls(ops, name, n):
    """moe_ffn_prefill_stack (routers of later layers launched behind the previous combine) gives the
    same bits as n separate moe_ffn_prefill_residual calls."""
    wl = WORKLOADS[name]
    inps, layers = _stack_layers(ops, wl, n)
    h0 = dev(inps[0]["hidden"])
    h = h0.clone()
    for inp, lay in zip(inps, layers):
        h = ops.moe_ffn_prefill_residual(lay.w, h, lay.routerW, lay.shexp_gate, h, wl.top_k, wl.norm_topk_prob,
                                         lay.ws)
    hs = h0.clone()
    ops.moe_ffn_prefill_stack([l.w for l in layers], [l.routerW for l in layers], [l.shexp_gate for l in layers], hs,
                              wl.top_k, wl.norm_topk_prob, layers[0].ws)
    torch.cuda.synchronize()
    assert all(l.status() == 0 for l in layers)
    a, b = hs.cpu().numpy(), h.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), float(np.abs(a - b).max())


def test_layer_stack_against_oracle_chain(ops):
    """Three tiny layers in place against the oracle applying the same layers one after another
    (out = (routed + shared) + hidden per layer)."""
    wl = WORKLOADS["tiny"]
    inps, layers = _stack_layers(ops, wl, 3)
    h = inps[0]["hidden"].copy()
    for inp in inps:
        step = dict(inp, hidden=h)
        r = O.moe_ffn_inputs(step, wl.top_k, wl.norm_topk_prob)
        h = O.combine(r["partials"], r["topk_w"], r.get("shared_out"), h)
    hs = dev(inps[0]["hidden"])
    ops.moe_ffn_prefill_stack([l.w for l in layers], [l.routerW for l in layers], [l.shexp_gate for l in layers], hs,
                              wl.top_k, wl.norm_topk_prob, layers[0].ws)
    got = hs.cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - h) / np.linalg.norm(h)
    assert rel <= 2e-3, rel


@pytest.mark.parametrize("name", ["tiny", "olmoe"])
def test_rmsnorm_alone_against_oracle(ops, name):
    wl = WORKLOADS[name]
    x = (np.random.default_rng(40).standard_normal((wl.N, wl.D)) * 3.0).astype(np.float32)
    gamma = _gamma(wl.D, 41)
    got = ops.moe_rmsnorm(dev(x), dev(gamma), 1e-6).cpu().numpy()
    _assert_normed(got, O.rmsnorm(x, gamma, 1e-6))
    with pytest.raises(ops.MoeError):
        xd = dev(x)
        ops.moe_rmsnorm(xd, dev(gamma), 1e-6, normed=xd)


def _gammas(wl, n, final):
    gs = [dev(_gamma(wl.D, 50 + l)) for l in range(n)]
    return gs + [dev(_gamma(wl.D, 50 + n)) if final else None]


@pytest.mark.parametrize("name,n,final", [("tiny", 3, True), ("olmoe", 2, True), ("qwen3moe_shared", 2, False),
                                          ("decode_n4", 3, True)])
def test_layer_stack_rmsnorm_equals_sequential_calls(ops, name, n, final):
    """moe_ffn_prefill_stack_rmsnorm (the first norm alone, every later one fused into the previous
    layer's combine, each router launched behind the kernel that writes its input) gives the same
    bits as the public calls one after another."""
    wl = WORKLOADS[name]
    inps, layers = _stack_layers(ops, wl, n)
    gammas = _gammas(wl, n, final)
    h = dev(inps[0]["hidden"])
    normed = ops.moe_rmsnorm(h, gammas[0], 1e-5)
    for l, lay in enumerate(layers):
        if gammas[l + 1] is not None:
            ops.moe_ffn_prefill_residual_rmsnorm(lay.w, normed, lay.routerW, lay.shexp_gate, h, gammas[l + 1], 1e-5,
                                                 wl.top_k, wl.norm_topk_prob, lay.ws, out=h, normed=normed)
        else:
            ops.moe_ffn_prefill_residual(lay.w, normed, lay.routerW, lay.shexp_gate, h, wl.top_k, wl.norm_topk_prob,
                                         lay.ws, out=h)
    hs = dev(inps[0]["hidden"])
    _, ns = ops.moe_ffn_prefill_stack_rmsnorm([l.w for l in layers], [l.routerW for l in layers],
                                              [l.shexp_gate for l in layers], gammas, 1e-5, hs, wl.top_k,
                                              wl.norm_topk_prob, layers[0].ws)
    torch.cuda.synchronize()
    assert all(l.status() == 0 for l in layers)
    for a, b in ((hs, h), (ns, normed)):
        a, b = a.cpu().numpy(), b.cpu().numpy()
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), float(np.abs(a - b).max())


def test_layer_stack_rmsnorm_against_oracle_chain(ops):
    """Three tiny pre-norm layers against the oracle chain: normed = RMSNorm_l(h), h = (routed +
    shared) + h per layer, within the layer's output bar."""
    wl = WORKLOADS["tiny"]
    inps, layers = _stack_layers(ops, wl, 3)
    gam = [_gamma(wl.D, 50 + l) for l in range(4)]
    h = inps[0]["hidden"].copy()
    for l, inp in enumerate(inps):
        x = O.rmsnorm(h, gam[l], 1e-5)
        r = O.moe_ffn_inputs(dict(inp, hidden=x), wl.top_k, wl.norm_topk_prob)
        h = O.combine(r["partials"], r["topk_w"], r.get("shared_out"), h)
    want_norm = O.rmsnorm(h, gam[3], 1e-5)
    hs = dev(inps[0]["hidden"])
    _, ns = ops.moe_ffn_prefill_stack_rmsnorm([l.w for l in layers], [l.routerW for l in layers],
                                              [l.shexp_gate for l in layers], [dev(g) for g in gam], 1e-5, hs,
                                              wl.top_k, wl.norm_topk_prob, layers[0].ws)
    got = hs.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(got - h) / np.linalg.norm(h) <= 2e-3
    gn = ns.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(gn - want_norm) / np.linalg.norm(want_norm) <= 2e-3


def test_layer_stack_rejects_bad_arguments(ops):
    wl = WORKLOADS["tiny"]
    inps, layers = _stack_layers(ops, wl, 2)
    h = dev(inps[0]["hidden"])
    with pytest.raises(ops.MoeError):
        ops.moe_ffn_prefill_stack([l.w for l in layers], [layers[0].routerW, layers[1].routerW], [None, None], h,
                                  wl.top_k, wl.norm_topk_prob, layers[0].ws[:1024])
