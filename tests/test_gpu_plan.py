"""One plan per step: the index call builds the inverted lists of its block_idx (for every
key block, the (query, slot) pairs that selected it) into a caller-owned buffer, and the
forward and the backward read them instead of each building their own.

The chain with the shared plan gives the same selection, index LSE, o and lse bit for
bit (every row is computed on its own, whatever tile it lands in), and the same gradients
to the rounding of the backward's accumulation order (the order of a key block's list
comes from a parallel fill), at G = 1, 4, 8 and 16.  A plan buffer that names another
problem, or holds no complete build, is reported through the device status and read as
empty lists."""
import numpy as np
import pytest
import torch

from block_sparse_gqa_topk_gb300 import _lib, ops, synth
from gpu_inputs import device_inputs

pytestmark = pytest.mark.gpu

CFG_G8 = synth.CONFIGS["8k"].with_(name="plan-g8", B=1, N=4096, H_q=16, H_kv=2, seed=81)
# G = 16 (8-query forward tiles, ragged N) and G = 1 with d = 64 (128-query tiles)
CFG_G16 = synth.CONFIGS["8k"].with_(name="plan-g16", B=1, N=3000, H_q=32, H_kv=2, topk=8, seed=82)
CFG_G1 = synth.CONFIGS["tiny"].with_(name="plan-g1", N=2200, H_q=4, H_kv=4, topk=3, seed=83)


def _step(cfg, d, plan):
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d, plan=plan)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx, plan=plan)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                    scale=cfg.scale, plan=plan)
    return bi, li, o, lse, g


def _plan_for(cfg):
    return ops.new_plan(cfg.B, cfg.N, cfg.H_q, cfg.H_kv, cfg.topk, d=cfg.d, d_idx=cfg.d_idx)


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], synth.CONFIGS["8k"], CFG_G8, CFG_G16, CFG_G1],
                         ids=["tiny", "8k", "g8", "g16", "g1_d64"])
def test_shared_plan_matches_per_call_plans(cfg):
    _, d = device_inputs(cfg)
    ref = _step(cfg, d, None)
    torch.cuda.synchronize()
    n0 = _lib.msa_kernel_launch_count()
    ref = _step(cfg, d, None)
    torch.cuda.synchronize()
    n_ref = _lib.msa_kernel_launch_count() - n0
    plan = _plan_for(cfg)
    n0 = _lib.msa_kernel_launch_count()
    got = _step(cfg, d, plan)
    torch.cuda.synchronize()
    n_got = _lib.msa_kernel_launch_count() - n0
    assert ops.device_status() == 0
    # two plan builds (count, scan, fill) give way to two header checks and one re-tiling
    assert n_ref - n_got == 3, (n_ref, n_got)
    for a, b, name in zip(got[:4], ref[:4], ("block_idx", "lse_idx", "o", "lse")):
        assert torch.equal(a, b), name
    for k in ("dq", "dk", "dv", "dq_idx", "dk_idx"):
        a = got[4][k].float().cpu().numpy()
        b = ref[4][k].float().cpu().numpy()
        assert np.abs(a - b).max() <= 1e-2 * max(np.abs(b).max(), 1e-30), k
    kl_a, kl_b = float(got[4]["kl"]), float(ref[4]["kl"])
    assert abs(kl_a - kl_b) <= 1e-5 * abs(kl_b) + 1e-7


def test_plan_of_another_problem_is_reported_and_read_as_empty():
    cfg = synth.CONFIGS["tiny"]
    _, d = device_inputs(cfg)
    plan = _plan_for(cfg)
    bi, li, o, lse, _ = _step(cfg, d, plan)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    # the first 1024 tokens as a problem of their own: the plan names N = 2048
    half = cfg.with_(name="plan-half", N=1024)
    dh = {n: t[:, :1024].contiguous() for n, t in d.items()}
    bh, lh = ops.msa_index_topk(dh["q_idx"], dh["k_idx"], half.topk, H_q=half.H_q, d=half.d)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    bad = plan.clone()
    ops.msa_fwd(dh["q"], dh["k"], dh["v"], bh, scale=half.scale, d_idx=half.d_idx, plan=bad)
    torch.cuda.synchronize()
    assert ops.device_status() == _lib.MSA_ERR_ARG
    # the refused buffer no longer holds a plan, even for the problem it was built for
    ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx, plan=bad)
    torch.cuda.synchronize()
    assert ops.device_status() == _lib.MSA_ERR_ARG
    # a buffer that holds no build is refused the same way, by the forward and the backward
    blank = torch.zeros_like(plan)
    ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx, plan=blank)
    torch.cuda.synchronize()
    assert ops.device_status() == _lib.MSA_ERR_ARG
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, 1e-3,
                    scale=cfg.scale, plan=blank)
    torch.cuda.synchronize()
    assert ops.device_status() == _lib.MSA_ERR_ARG
    # read as empty lists: no key block received any gradient
    assert not g["dk"].any() and not g["dv"].any()
    # the library is still usable, and the good plan still works
    o2, lse2 = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx,
                           plan=plan)
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    assert torch.equal(o2, o) and torch.equal(lse2, lse)


def test_autograd_step_builds_one_plan():
    cfg = synth.CONFIGS["tiny"]
    _, d = device_inputs(cfg)
    q, k, v = (d[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    q_idx, k_idx = (d[n].clone().requires_grad_(True) for n in ("q_idx", "k_idx"))
    ops.attention(q, k, v, q_idx, k_idx, cfg.topk).backward(d["dO"])  # warm the workspace
    torch.cuda.synchronize()
    n0 = _lib.msa_kernel_launch_count()
    o = ops.attention(q, k, v, q_idx, k_idx, cfg.topk, scale=cfg.scale)
    o.backward(d["dO"])
    torch.cuda.synchronize()
    assert ops.device_status() == 0
    # index (top-k, count, scan, fill, re-tile, LSE, LSE merge) + forward (check, tile
    # kernel, combine) + backward (check, preprocess, tile kernel, two slot reductions,
    # dk_idx reduction, KL out)
    assert _lib.msa_kernel_launch_count() - n0 == 17
