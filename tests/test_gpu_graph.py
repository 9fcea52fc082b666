"""The training calls capture into a CUDA graph as they are (the library allocates
nothing and queues only memsets and kernels on the caller's stream): a replayed step
reproduces the eager step.  Selection, index LSE and forward outputs are bit-identical;
the backward's accumulation order follows the plan's fill order, which may differ between
runs, so its outputs are compared to a rounding tolerance."""
import numpy as np
import pytest
import torch

from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import device_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "8k"])
def test_captured_step_matches_eager(name):
    cfg = synth.CONFIGS[name]
    _, d = device_inputs(cfg)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)

    def step():
        bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d)
        o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx)
        g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                        scale=cfg.scale)
        return bi, li, o, lse, g

    eager = step()
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    eager = [t.clone() if isinstance(t, torch.Tensor) else {k: v.clone() for k, v in t.items()}
             for t in eager]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # the workspace is sized before the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert ops.device_status() == 0

    bi, li, o, lse, g = out
    assert torch.equal(bi, eager[0])
    assert torch.equal(li, eager[1])
    assert torch.equal(o, eager[2])
    assert torch.equal(lse, eager[3])
    for k in ("dq", "dk", "dv", "dq_idx", "dk_idx"):
        a = g[k].float().cpu().numpy()
        b = eager[4][k].float().cpu().numpy()
        scale = max(np.abs(b).max(), 1e-30)
        assert np.abs(a - b).max() <= 1e-2 * scale, k
    assert abs(float(g["kl"]) - float(eager[4]["kl"])) <= 1e-4 * abs(float(eager[4]["kl"])) + 1e-7
