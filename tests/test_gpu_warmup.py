"""GPU parity of the indexer warm-up against the float64 oracle.

Warm-up gives both branches full attention while the indexer learns from the KL
alone (MSA summary, 7minutos.es, "Cómo se entrena MSA" ¶3).  Here that is the dense set:
topk >= the number of blocks, so every visible block is selected, the main branch is
full causal attention, and the KL runs over every visible token.  The GPU path is run
end to end through the C ABI (its own set, lse_idx, o and lse feed its backward);
the oracle computes everything from the inputs.  The set is fixed by the rule and is
compared exactly; the cases use more than 32 slots per row (up to 256).
"""
import numpy as np
import pytest

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import device_inputs
from parity import KL_REL, LSE_TOL, O_TOL, f64, grad_close

pytestmark = pytest.mark.gpu

T = synth.CONFIGS["tiny"]
E = synth.CONFIGS["8k"]
CASES = {
    # 24 blocks, ragged last block, topk = nb (the forced fill below the 32-slot limit)
    "ragged-24": T.with_(name="warm-ragged", N=3000, topk=24, seed=71),
    # 64 blocks, 64 slots
    "8k-64": E.with_(name="warm-8k", B=1, topk=64, seed=72),
    # 128 blocks, the 128-slot maximum, d = 128 with G = 4
    "16k-128": E.with_(name="warm-16k", B=1, N=16384, H_q=8, H_kv=2, topk=128, seed=73),
}


def _dense(cfg):
    i = np.arange(cfg.N)
    s = np.arange(cfg.topk)
    full = np.where(s[None, :] <= (i // cfg.Bk)[:, None], s[None, :], -1).astype(np.int32)
    return np.broadcast_to(full, (cfg.B, cfg.H_kv, cfg.N, cfg.topk))


@pytest.mark.parametrize("name", sorted(CASES))
def test_warmup_dense_matches_oracle(name):
    cfg = CASES[name]
    assert cfg.topk >= cfg.nb
    h, d = device_inputs(cfg)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                    scale=cfg.scale)
    assert ops.device_status() == 0
    # the set: every visible block, identical to the oracle's selection at this topk
    bi_ref, _, _ = oracle.select(cfg, h)
    gsel = bi.cpu().numpy()
    assert np.array_equal(gsel, _dense(cfg))
    assert np.array_equal(gsel.transpose(0, 2, 1, 3).reshape(bi_ref.shape), bi_ref)
    # index LSE over every visible token; main-branch o and lse
    o_ref, lse_ref, li_ref = oracle.forward(cfg, h, bi_ref)
    el_i = np.abs(li.cpu().numpy().transpose(0, 2, 1).reshape(li_ref.shape) - li_ref).max()
    eo = np.abs(f64(o).reshape(o_ref.shape) - o_ref).max()
    el = np.abs(lse.cpu().numpy().transpose(0, 2, 1).reshape(lse_ref.shape) - lse_ref).max()
    assert el_i <= LSE_TOL and eo <= O_TOL and el <= LSE_TOL, (el_i, eo, el)
    # every gradient and the KL over every visible token
    ref = oracle.backward(cfg, h, bi_ref, w)
    out = []
    for n in ("dq", "dk", "dv", "dq_idx", "dk_idx"):
        cos, rel = grad_close(f64(g[n]), ref[n].reshape(g[n].shape), n)
        out.append(f"{n} cos {cos:.6f} rel {rel:.2e}")
    kl = float(g["kl"].cpu())
    assert abs(kl - ref["kl"]) <= KL_REL * abs(ref["kl"]) + 1e-6, (kl, ref["kl"])
    print(f"{name}: lse_idx {el_i:.2e} o {eo:.2e} lse {el:.2e}; " + "; ".join(out)
          + f"; kl {kl:.6e} vs {ref['kl']:.6e}")


def test_selection_above_32_below_nb_is_refused():
    from block_sparse_gqa_topk_gb300 import _lib
    cfg = E.with_(name="warm-refuse", B=1, N=8192, topk=40)  # 40 slots, 64 blocks
    _, d = device_inputs(cfg, names=("q_idx", "k_idx"))
    with pytest.raises(_lib.MSAError):
        ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d)


def test_warmup_dense_32k_256_slots_sampled():
    """256 slots (every block of a 32K-token sequence): the index LSE, o, lse and the
    per-row gradients dq, dq_idx on sampled rows; dk and dv of the sampled rows alone
    from a second backward with dO zero elsewhere and no KL (the oracle's row-subset
    backward computes exactly that)."""
    import torch
    from gpu_inputs import rows_for
    from parity import LSE_TOL
    cfg = E.with_(name="warm-32k", B=1, N=32768, H_q=8, H_kv=2, topk=256, n_needle=2, seed=74)
    assert cfg.topk >= cfg.nb
    h, d = device_inputs(cfg)
    rows, _ = rows_for(cfg, 192)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d)
    o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx)
    g = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li, w,
                    scale=cfg.scale)
    assert ops.device_status() == 0
    b, i = rows // cfg.N, rows % cfg.N
    assert np.array_equal(bi.cpu().numpy(), _dense(cfg))
    bi_ref, _, _ = oracle.select(cfg, h, rows=rows)
    assert np.array_equal(bi.cpu().numpy()[b, :, i], bi_ref)
    o_ref, lse_ref, li_ref = oracle.forward(cfg, h, bi_ref, rows=rows)
    assert np.abs(li.cpu().numpy()[b, :, i] - li_ref).max() <= LSE_TOL
    assert np.abs(f64(o)[b, i] - o_ref).max() <= O_TOL
    assert np.abs(lse.cpu().numpy()[b, :, i] - lse_ref).max() <= LSE_TOL
    ref = oracle.backward(cfg, h, bi_ref, w, rows=rows)
    grad_close(f64(g["dq"])[b, i], ref["dq"], "dq")
    grad_close(f64(g["dq_idx"])[b, i], ref["dq_idx"], "dq_idx")
    del g
    keep = torch.zeros(cfg.B * cfg.N, dtype=torch.bool, device="cuda")
    keep[torch.from_numpy(rows).cuda()] = True
    dO_m = d["dO"].clone().view(cfg.B * cfg.N, -1)
    dO_m[~keep] = 0
    g2 = ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, dO_m.view_as(d["dO"]), d["q_idx"], d["k_idx"],
                     bi, li, 0.0, scale=cfg.scale)
    assert ops.device_status() == 0
    ref0 = oracle.backward(cfg, h, bi_ref, 0.0, rows=rows)
    grad_close(f64(g2["dk"]), ref0["dk"], "dk")
    grad_close(f64(g2["dv"]), ref0["dv"], "dv")
