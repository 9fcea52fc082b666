"""GPU parity of the packed variable-length entry points (cu_seqlens) against the
float64 oracle run on each sequence as its own problem (the variable-length view of
Flash-MSA, tech.kuratif.com ¶7): selection, index LSE, forward, and the fused
backward with the KL summed over sequences.  The batch mixes a long sequence, an
empty one, a ragged one and a two-block one.  The block sets and index LSE fed to the
GPU forward/backward are the oracle's own."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import host_inputs
from parity import KL_REL, LSE_TOL, O_TOL, check_selection, f64, gpu_sel_rows, grad_close, to_dev

pytestmark = pytest.mark.gpu

CFG = synth.CONFIGS["tiny"].with_(name="varlen", seed=51)  # packed T = 2048 tokens
CU = [0, 1024, 1024, 1796, 2048]                            # lengths 1024, 0, 772, 252
# G = 8, d = 128, d_idx = 64, k = 16: packed T = 4096 tokens, lengths 2560, 4, 1532
CFG8 = synth.CONFIGS["8k"].with_(name="varlen-g8", B=1, N=4096, H_q=16, H_kv=2, seed=52)
CU8 = [0, 2560, 2564, 4096]


def _seq(h, c0, c1):
    """Inputs of one sequence as a B=1 problem (host bits)."""
    return {n: np.ascontiguousarray(h[n][:, c0:c1]) for n in h}


@pytest.mark.parametrize("cfg,CU", [(CFG, CU), (CFG8, CU8)], ids=["tiny", "g8_d128"])
def test_varlen_matches_oracle_per_sequence(cfg, CU):
    h = host_inputs(cfg)
    d = {n: to_dev(h[n])[0].contiguous() for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
    H_kv, k = cfg.H_kv, cfg.topk
    w = cfg.kl_coef / (cfg.H_kv * CU[-1])
    # GPU index branch over the packed batch
    bi_gpu, li_gpu = ops.msa_index_topk_varlen(d["q_idx"], d["k_idx"], CU, k, H_q=cfg.H_q, d=cfg.d)
    assert ops.device_status() == 0
    bi_pack, li_pack, refs = [], [], []
    for s in range(len(CU) - 1):
        c0, c1 = CU[s], CU[s + 1]
        L = c1 - c0
        if L == 0:
            refs.append(None)
            continue
        cs = cfg.with_(N=L)
        hs = _seq(h, c0, c1)
        bi_ref, kth, _ = oracle.select(cs, hs)
        rows = np.arange(L, dtype=np.int64)
        gsel = gpu_sel_rows(cs, ops.varlen_view(bi_gpu, CU, s, H_kv, k).cpu().numpy()[None], rows)
        n_same, n_near, diff = check_selection(cs, hs, gsel, rows, bi_ref, kth)
        _, _, li_ref = oracle.forward(cs, hs, bi_ref, main=False)
        li = ops.varlen_view(li_gpu, CU, s, H_kv).cpu().numpy()[:, :, 0].T
        err = np.abs(li[~diff] - li_ref[~diff]).max()
        assert err <= LSE_TOL, f"seq {s}: lse_idx err {err}"
        bi_pack.append(bi_ref.transpose(1, 0, 2).reshape(-1))
        li_pack.append(li_ref.T.reshape(-1).astype(np.float32))
        refs.append((cs, hs, bi_ref))
    # forward and backward over the oracle's sets
    block_idx = torch.from_numpy(np.concatenate(bi_pack).astype(np.int32)).cuda()
    lse_idx = torch.from_numpy(np.concatenate(li_pack)).cuda()
    o, lse = ops.msa_fwd_varlen(d["q"], d["k"], d["v"], block_idx, CU, k, scale=cfg.scale,
                                d_idx=cfg.d_idx)
    g = ops.msa_bwd_varlen(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"],
                           block_idx, lse_idx, w, CU, k, scale=cfg.scale)
    assert ops.device_status() == 0
    kl_ref = 0.0
    for s, r in enumerate(refs):
        if r is None:
            continue
        cs, hs, bi_ref = r
        c0, c1 = CU[s], CU[s + 1]
        o_ref, lse_ref, _ = oracle.forward(cs, hs, bi_ref, index=False)
        eo = np.abs(f64(o[c0:c1]) - o_ref).max()
        el = np.abs(ops.varlen_view(lse, CU, s, cfg.H_q).cpu().numpy()[:, :, 0].T - lse_ref).max()
        assert eo <= O_TOL and el <= LSE_TOL, (s, eo, el)
        ref = oracle.backward(cs, hs, bi_ref, w)
        grad_close(f64(g["dq"][c0:c1]), ref["dq"], f"dq[{s}]")
        grad_close(f64(g["dk"][c0:c1]), ref["dk"][0], f"dk[{s}]")
        grad_close(f64(g["dv"][c0:c1]), ref["dv"][0], f"dv[{s}]")
        grad_close(f64(g["dq_idx"][c0:c1]), ref["dq_idx"], f"dq_idx[{s}]")
        grad_close(f64(g["dk_idx"][c0:c1]), ref["dk_idx"][0], f"dk_idx[{s}]")
        kl_ref += ref["kl"]
    kl = float(g["kl"].cpu())
    assert abs(kl - kl_ref) <= KL_REL * abs(kl_ref) + 1e-6, (kl, kl_ref)


def test_varlen_rejects_bad_offsets():
    from block_sparse_gqa_topk_gb300 import _lib
    d = {"q_idx": torch.zeros(8, 2, 32, dtype=torch.bfloat16, device="cuda"),
         "k_idx": torch.zeros(8, 32, dtype=torch.bfloat16, device="cuda")}
    with pytest.raises(_lib.MSAError):
        ops.msa_index_topk_varlen(d["q_idx"], d["k_idx"], [0, 3, 8], 4, H_q=8, d=64)  # start 3
    with pytest.raises(ValueError):
        ops.msa_index_topk_varlen(d["q_idx"], d["k_idx"], [0, 6, 4, 8], 4, H_q=8, d=64)
