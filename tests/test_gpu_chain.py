"""The whole GPU chain at full size: the GPU's own block selection feeds the GPU's
index LSE, forward and backward (msa_index_topk -> msa_fwd -> msa_bwd, as a training
step runs them), and every sampled output is compared with the float64 oracle rerun
on the GPU's sets for those rows, once the near-tie rule has accepted the sets.

Per sampled row: block sets (exact outside the 1e-3 band, valid inside it), lse_idx,
o, lse, dq, dq_idx.  The KL of the sampled rows: a second backward gets lse = +inf
outside the sample, which makes those rows' main-branch probabilities, teacher and
KL terms exactly zero.  dk and dv of the sampled rows: a third backward whose dO is
zero outside the sample and whose KL weight is 0, which the oracle's row-subset
backward computes exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import device_inputs, rows_for
from parity import KL_REL, LSE_TOL, O_TOL, f64, grad_close, validated_gpu_sets

pytestmark = pytest.mark.gpu

CASES = [("32k", 512), ("128k", 256), ("1m", 128)]


@pytest.mark.parametrize("name,n_rows", CASES)
def test_gpu_chain_matches_oracle_on_gpu_sets(name, n_rows):
    cfg = synth.CONFIGS[name]
    h, d = device_inputs(cfg)
    rows, _ = rows_for(cfg, n_rows, seed=91)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                    scale=cfg.scale)
    assert ops.device_status() == 0
    b, i = rows // cfg.N, rows % cfg.N
    bt, it = torch.from_numpy(b).cuda(), torch.from_numpy(i).cuda()
    gsel = bi[bt, :, it, :].cpu().numpy()                       # [R, H_kv, k]
    sets, n_diff = validated_gpu_sets(cfg, h, gsel, rows)
    o_ref, lse_ref, li_ref = oracle.forward(cfg, h, sets, rows=rows)
    eo = np.abs(f64(o[bt, it]) - o_ref).max()
    el = np.abs(lse[bt, :, it].cpu().numpy() - lse_ref).max()
    eli = np.abs(li[bt, :, it].cpu().numpy() - li_ref).max()
    assert eo <= O_TOL and el <= LSE_TOL and eli <= LSE_TOL, (eo, el, eli)
    ref = oracle.backward(cfg, h, sets, w, rows=rows)
    c1 = grad_close(f64(g["dq"][bt, it]), ref["dq"], "dq")
    c2 = grad_close(f64(g["dq_idx"][bt, it]), ref["dq_idx"], "dq_idx")
    del g
    # the KL of the sampled rows alone
    other = torch.ones(cfg.B, cfg.N, dtype=torch.bool, device="cuda")
    other.view(-1)[torch.from_numpy(rows).cuda()] = False
    lse_m = lse.clone().masked_fill_(other[:, None, :], float("inf"))
    g3 = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse_m, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                     scale=cfg.scale)
    assert ops.device_status() == 0
    kl = float(g3["kl"].cpu())
    assert abs(kl - ref["kl"]) <= KL_REL * abs(ref["kl"]) + 1e-6, (kl, ref["kl"])
    del g3, lse_m
    # dk, dv of the sampled rows alone
    dO_m = d["dO"].clone().view(cfg.B * cfg.N, -1)
    dO_m[other.view(-1)] = 0
    dO_m = dO_m.view_as(d["dO"])
    g2 = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, dO_m, d["q_idx"], d["k_idx"], bi, li, 0.0,
                     scale=cfg.scale)
    assert ops.device_status() == 0
    ref0 = oracle.backward(cfg, h, sets, 0.0, rows=rows)
    c3 = grad_close(f64(g2["dk"]), ref0["dk"], "dk")
    c4 = grad_close(f64(g2["dv"]), ref0["dv"], "dv")
    print(f"{name}: {len(rows)} rows, {n_diff} near-tie (row, group) sets differ; o {eo:.2e} "
          f"lse {el:.2e} lse_idx {eli:.2e}; dq {c1}, dq_idx {c2}, dk {c3}, dv {c4}; "
          f"kl {kl:.6e} vs {ref['kl']:.6e}")
