"""The torch autograd wrapper (ops.attention / ops.MSAFunction): one training step
through the C ABI, with the gradients that reach the leaf tensors compared with the
float64 oracle -- dq, dk, dv from the loss sum(dO * o), dq_idx and dk_idx from the KL
alignment term alone (teacher detached; MSA summary, 7minutos.es, "Cómo se entrena MSA"
¶1-2), and the KL value kept by the wrapper."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import host_inputs
from parity import KL_REL, O_TOL, f64, gpu_sel_rows, grad_close, to_dev, validated_gpu_sets

pytestmark = pytest.mark.gpu


def test_autograd_step_matches_oracle():
    cfg = synth.CONFIGS["tiny"].with_(name="autograd", N=1536, seed=57)
    h = host_inputs(cfg)
    leaf = {n: to_dev(h[n]).clone().requires_grad_(True) for n in ("q", "k", "v", "q_idx", "k_idx")}
    dO = to_dev(h["dO"])
    o, block_idx = ops.MSAFunction.apply(leaf["q"], leaf["k"], leaf["v"], leaf["q_idx"],
                                         leaf["k_idx"], cfg.topk, 128, cfg.scale, None,
                                         cfg.kl_coef)
    o.backward(dO)
    assert ops.device_status() == 0
    # the GPU's own selection drives this step: validated against the oracle's with the
    # near-tie rule, then the oracle reruns on exactly those sets
    rows = np.arange(cfg.B * cfg.N, dtype=np.int64)
    sets, _ = validated_gpu_sets(cfg, h, gpu_sel_rows(cfg, block_idx.cpu().numpy(), rows), rows)
    o_ref, _, _ = oracle.forward(cfg, h, sets, index=False)
    assert np.abs(f64(o.detach()).reshape(o_ref.shape) - o_ref).max() <= O_TOL
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    ref = oracle.backward(cfg, h, sets, w)
    for n, r in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("q_idx", "dq_idx"), ("k_idx", "dk_idx")):
        g = leaf[n].grad
        assert g is not None and g.dtype == torch.bfloat16, n
        grad_close(f64(g), ref[r].reshape(g.shape), r)
    kl = float(ops.MSAFunction.last_kl.cpu())
    assert abs(kl - ref["kl"]) <= KL_REL * abs(ref["kl"]) + 1e-6, (kl, ref["kl"])
