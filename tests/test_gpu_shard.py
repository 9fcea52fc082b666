"""GPU check that the path shards by GQA group with dk_idx (and the KL) as the only
exchanged values: the product's per-rank step (shard.library_step on the slice that
shard.GroupShard.take gives each group) reproduces the single call over all groups
once the per-group dk_idx and KL are summed (on the host here, as the all-reduce of
shard.exchange does across GPUs).  The groups are
independent except for the one shared index-key head (MSA summary, 7minutos.es,
"Cómo funcionan las dos ramas" ¶1).
"""
import numpy as np
import pytest
import torch

from block_sparse_gqa_topk_gb300 import shard, synth
from gpu_inputs import device_inputs
from parity import KL_REL, LSE_TOL, O_TOL, f64, grad_close

CFG = synth.CONFIGS["8k"].with_(name="8k-half", B=1, N=4096)


@pytest.mark.gpu
def test_group_sliced_calls_reproduce_the_full_call():
    from block_sparse_gqa_topk_gb300 import ops
    cfg = CFG
    _, t = device_inputs(cfg)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)

    def run(x):
        bi, li = ops.msa_index_topk(x["q_idx"], x["k_idx"], cfg.topk, H_q=x["q"].shape[2],
                                    d=cfg.d)
        o, lse = ops.msa_fwd(x["q"], x["k"], x["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx)
        g = ops.msa_bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], x["q_idx"], x["k_idx"], bi, li,
                        w, scale=cfg.scale)
        torch.cuda.synchronize()
        return bi, li, o, lse, g

    bi, li, o, lse, g = run(t)
    assert ops.device_status() == 0
    G = cfg.G
    dk_idx_sum = np.zeros(tuple(t["k_idx"].shape))
    kl_sum = 0.0
    # one "rank" per group (world = H_kv), each running the product's per-rank step on
    # the slice GroupShard.take gives it, in turn on this one GPU
    for grp in range(cfg.H_kv):
        sh = shard.GroupShard(grp, cfg.H_kv, cfg.H_kv)
        assert sh.groups == (grp, grp + 1)
        hs = slice(grp * G, (grp + 1) * G)
        x = {n: sh.take(n, t[n]) for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
        sg = shard.library_step(x, cfg.topk, cfg.scale, sh.kl_weight(cfg.B, cfg.N, cfg.kl_coef))
        torch.cuda.synchronize()
        assert ops.device_status() == 0
        # selection and index LSE are per-group computations: identical
        assert torch.equal(sg["block_idx"], sh.take("block_idx", bi))
        np.testing.assert_allclose(f64(sg["lse_idx"]), f64(sh.take("lse_idx", li)), rtol=0,
                                   atol=LSE_TOL)
        np.testing.assert_allclose(f64(sg["o"]), f64(sh.take("o", o)), rtol=0, atol=O_TOL)
        np.testing.assert_allclose(f64(sg["lse"]), f64(sh.take("lse", lse)), rtol=0, atol=LSE_TOL)
        grad_close(f64(sg["dq"]), f64(g["dq"][:, :, hs]), f"dq[{grp}]")
        grad_close(f64(sg["dk"][:, :, 0]), f64(g["dk"][:, :, grp]), f"dk[{grp}]")
        grad_close(f64(sg["dv"][:, :, 0]), f64(g["dv"][:, :, grp]), f"dv[{grp}]")
        grad_close(f64(sg["dq_idx"][:, :, 0]), f64(g["dq_idx"][:, :, grp]), f"dq_idx[{grp}]")
        dk_idx_sum += f64(sg["dk_idx"])
        kl_sum += float(sg["kl"].item())
    grad_close(dk_idx_sum, f64(g["dk_idx"]), "dk_idx (sum over group shards)")
    assert kl_sum == pytest.approx(float(g["kl"].item()), rel=KL_REL)
