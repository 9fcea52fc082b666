"""GPU parity of the fused backward (msa_bwd) against the float64 oracle, through
the C ABI.  The block sets and the index LSE fed to the GPU are the oracle's own
(oracle outputs may feed the GPU; nothing from the GPU feeds the oracle).

Full workloads (every gradient and the KL): small edge cases and the 8K workload.
Large workloads (32K, 128K, 1M): dq and dq_idx on seeded sampled rows (both are
per-row quantities); dk and dv from a second backward whose dO is zero outside
the sampled rows and whose KL weight is 0, which the oracle's row-subset backward
computes exactly.  dk_idx of one whole key block at 32K, 128K and 1M: only rows at or after
the block can select it, so the oracle's sets of those rows name every (query, group)
that attends to it, and the row-subset backward over them gives its dk_idx exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import device_inputs, rows_for
from parity import KL_REL, f64, grad_close
from test_gpu_index_fwd import EDGE, cfg_of

pytestmark = pytest.mark.gpu

FULL = ["tiny", "ragged", "one_block", "k1", "k3", "dense", "odd_groups", "g1", "g2", "g2_d128",
        "g8", "g16", "g16_d128", "k8_d128", "8k"]
SAMPLED = [("32k", 512), ("128k", 256), ("1m", 128)]


def _w(cfg):
    return cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)


def _dev_sel(cfg, bi_rows, rows):
    """[R,H_kv,k] oracle sets -> device [B,H_kv,N,k]; rows None means all rows."""
    if rows is None:
        full = bi_rows.reshape(cfg.B, cfg.N, cfg.H_kv, cfg.topk).transpose(0, 2, 1, 3)
    else:
        i = np.arange(cfg.N)
        ci = i // cfg.Bk
        base = ci[:, None] - np.arange(cfg.topk)[None, ::-1]
        base = np.sort(np.where(base < 0, 1 << 30, base), axis=1)
        base = np.where(base == 1 << 30, -1, base).astype(np.int32)
        full = np.broadcast_to(base, (cfg.B, cfg.H_kv, cfg.N, cfg.topk)).copy()
        full[rows // cfg.N, :, rows % cfg.N, :] = bi_rows
    return torch.from_numpy(np.ascontiguousarray(full, dtype=np.int32)).cuda()


def _dev_lse_idx(cfg, li_rows, rows):
    full = np.zeros((cfg.B, cfg.H_kv, cfg.N), dtype=np.float32)
    if rows is None:
        full[:] = li_rows.reshape(cfg.B, cfg.N, cfg.H_kv).transpose(0, 2, 1)
    else:
        full[rows // cfg.N, :, rows % cfg.N] = li_rows
    return torch.from_numpy(full).cuda()


@pytest.mark.parametrize("name", FULL)
def test_bwd_matches_oracle_full(name):
    cfg = cfg_of(name)
    h, d = device_inputs(cfg)
    bi_ref, _, _ = oracle.select(cfg, h)
    _, _, li_ref = oracle.forward(cfg, h, bi_ref, main=False)
    block_idx = _dev_sel(cfg, bi_ref, None)
    lse_idx = _dev_lse_idx(cfg, li_ref, None)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], block_idx, scale=cfg.scale, d_idx=cfg.d_idx)
    w = _w(cfg)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], block_idx,
                    lse_idx, w, scale=cfg.scale)
    assert ops.device_status() == 0
    ref = oracle.backward(cfg, h, bi_ref, w)
    out = []
    for n in ("dq", "dk", "dv", "dq_idx", "dk_idx"):
        cos, rel = grad_close(f64(g[n]), ref[n].reshape(g[n].shape), n)
        out.append(f"{n} cos {cos:.6f} rel {rel:.2e}")
    kl = float(g["kl"].cpu())
    assert abs(kl - ref["kl"]) <= KL_REL * abs(ref["kl"]) + 1e-6, (kl, ref["kl"])
    print(f"{name}: " + "; ".join(out) + f"; kl {kl:.6e} vs {ref['kl']:.6e}")


@pytest.mark.parametrize("name,n_rows", SAMPLED)
def test_bwd_matches_oracle_sampled(name, n_rows):
    cfg = cfg_of(name)
    h, d = device_inputs(cfg)
    rows, _ = rows_for(cfg, n_rows)
    bi_ref, _, _ = oracle.select(cfg, h, rows=rows)
    _, _, li_ref = oracle.forward(cfg, h, bi_ref, rows=rows, main=False)
    block_idx = _dev_sel(cfg, bi_ref, rows)
    lse_idx = _dev_lse_idx(cfg, li_ref, rows)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], block_idx, scale=cfg.scale, d_idx=cfg.d_idx)
    w = _w(cfg)
    b, i = rows // cfg.N, rows % cfg.N
    # 1) per-row gradients with the full dO and KL weight
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], block_idx,
                    lse_idx, w, scale=cfg.scale)
    assert ops.device_status() == 0
    ref = oracle.backward(cfg, h, bi_ref, w, rows=rows)
    c1 = grad_close(f64(g["dq"])[b, i], ref["dq"], "dq")
    c2 = grad_close(f64(g["dq_idx"])[b, i], ref["dq_idx"], "dq_idx")
    # (the KL total is checked in 3): here rows outside the sample carry a placeholder
    # lse_idx, so their KL terms are not a divergence)
    del g
    # 2) key-side gradients of the sampled rows only: dO zero elsewhere, no KL
    keep = torch.zeros(cfg.B * cfg.N, dtype=torch.bool, device="cuda")
    keep[torch.from_numpy(rows).cuda()] = True
    dO_m = d["dO"].clone().view(cfg.B * cfg.N, -1)
    dO_m[~keep] = 0
    dO_m = dO_m.view_as(d["dO"])
    g2 = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, dO_m, d["q_idx"], d["k_idx"], block_idx,
                     lse_idx, 0.0, scale=cfg.scale)
    assert ops.device_status() == 0
    ref0 = oracle.backward(cfg, h, bi_ref, 0.0, rows=rows)
    c3 = grad_close(f64(g2["dk"]), ref0["dk"], "dk")
    c4 = grad_close(f64(g2["dv"]), ref0["dv"], "dv")
    del g2
    # 3) the KL of the sampled rows: lse = +inf outside the sample makes those rows'
    # main-branch probabilities, hence their teacher and their KL terms, exactly zero
    other = torch.ones(cfg.B, cfg.N, dtype=torch.bool, device="cuda")
    other.view(-1)[torch.from_numpy(rows).cuda()] = False
    lse_m = lse.clone().masked_fill_(other[:, None, :], float("inf"))
    g3 = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse_m, d["dO"], d["q_idx"], d["k_idx"],
                     block_idx, lse_idx, w, scale=cfg.scale)
    assert ops.device_status() == 0
    kl = float(g3["kl"].cpu())
    assert abs(kl - ref["kl"]) <= KL_REL * abs(ref["kl"]) + 1e-6, (kl, ref["kl"])
    print(f"{name}: dq {c1}, dq_idx {c2}, dk {c3}, dv {c4}, kl {kl:.6e} vs {ref['kl']:.6e}")


@pytest.mark.parametrize("name", ["32k", "128k", "1m"])
def test_bwd_dk_idx_of_a_key_block_full_size(name):
    cfg = cfg_of(name)
    assert cfg.B == 1
    h, d = device_inputs(cfg)
    nb = (cfg.N + cfg.Bk - 1) // cfg.Bk
    c = nb - 8  # a late block: its possible readers are the 8 blocks of rows from c on
    later = np.arange(c * cfg.Bk, cfg.N, dtype=np.int64)
    bi_later, _, _ = oracle.select(cfg, h, rows=later)
    _, _, li_later = oracle.forward(cfg, h, bi_later, rows=later, main=False)
    # rows before block c keep a local window of sets, which never holds block c
    block_idx = _dev_sel(cfg, bi_later, later)
    lse_idx = _dev_lse_idx(cfg, li_later, later)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], block_idx, scale=cfg.scale, d_idx=cfg.d_idx)
    w = _w(cfg)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], block_idx,
                    lse_idx, w, scale=cfg.scale)
    assert ops.device_status() == 0
    hit = (bi_later == c).any(axis=(1, 2))  # rows with block c in some group's set
    assert hit[:cfg.Bk].all()  # the block's own rows always hold it
    rows = later[hit]
    ref = oracle.backward(cfg, h, bi_later[hit], w, rows=rows)
    keys = slice(c * cfg.Bk, min(cfg.N, (c + 1) * cfg.Bk))
    cos, rel = grad_close(f64(g["dk_idx"])[0, keys], ref["dk_idx"][0, keys], "dk_idx")
    print(f"{name}: block {c}, {len(rows)} reading rows: dk_idx cos {cos:.6f}, rel {rel:.2e}")
