"""Expert parallelism's device backend on one GPU: a one-rank NCCL group owns every expert, so the
exchange is a self all-to-all; the layer output must equal moe_ffn_prefill's bit for bit (the
library's kernels compute each partial row independently of the batch it sits in)."""
import os
import socket

import numpy as np
import pytest

from mixture_experts_ffn_top_gb300.workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def group():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import torch.distributed as dist

    from mixture_experts_ffn_top_gb300 import build

    build.build()
    torch.cuda.set_device(0)
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    yield dist
    dist.destroy_process_group()


# decode_n8_q4k: the single-GPU layer streams the nibble-packed Q4_K copy through the decode ring,
# the expert owner (64 single-slot rows) runs the register-loading matvecs on the int8 repack
@pytest.mark.parametrize("name", ["tiny", "olmoe", "qwen3moe_shared", "decode_n8", "decode_n8_q4k", "olmoe_q4k"])
def test_device_expert_parallel_matches_prefill(group, name):
    from mixture_experts_ffn_top_gb300 import ops
    from mixture_experts_ffn_top_gb300.expert_parallel import DeviceBackend, expert_parallel_forward

    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    hidden = torch.from_numpy(inp["hidden"]).cuda()
    layer = ops.MoeLayer.from_numpy(inp, device="cuda:0", top_k=wl.top_k, max_tokens=wl.N)
    ref = layer.prefill(hidden, wl.top_k, wl.norm_topk_prob)
    be = DeviceBackend(inp, 0, wl.E, "cuda:0", wl.top_k, wl.N)
    out = expert_parallel_forward(be, hidden, wl.E, wl.top_k, wl.norm_topk_prob)
    torch.cuda.synchronize()
    assert layer.status() == 0 and ops.moe_workspace_status(be.route_ws) == 0
    a, b = out.cpu().numpy(), ref.cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), float(np.abs(a - b).max())
