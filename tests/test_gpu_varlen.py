"""GPU parity of the packed variable-length entry points (device cu_seqlens) against the
float64 oracle run on each sequence as its own problem (the variable-length view of
Flash-MSA, tech.kuratif.com ¶7).

The whole GPU chain runs over the packed batch: selection, index LSE, forward and the
fused backward with the KL summed over sequences.  Each sequence's GPU block sets are
checked by the near-tie rule, and the oracle then runs on exactly those sets, so every
row of every sequence is compared.  Batches: a mix of a long, an empty, a ragged and a
short sequence at odd token offsets; G = 16, 8 and 2 with d = 128, G = 1 with d = 64; and
64 short ragged sequences.
The number of kernel launches of a call does not depend on the number of sequences.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import _lib, ops, synth
from gpu_inputs import host_inputs
from parity import KL_REL, LSE_TOL, O_TOL, f64, grad_close, to_dev, validated_gpu_sets

pytestmark = pytest.mark.gpu

CFG = synth.CONFIGS["tiny"].with_(name="varlen", seed=51)  # packed T = 2048 tokens
CU = [0, 1021, 1021, 1795, 2048]                            # lengths 1021, 0, 774, 253
# G = 8, d = 128, d_idx = 64, k = 16: packed T = 4096 tokens, lengths 2561, 3, 1531, 1
CFG8 = synth.CONFIGS["8k"].with_(name="varlen-g8", B=1, N=4096, H_q=16, H_kv=2, seed=52)
CU8 = [0, 2561, 2564, 4095, 4096]
# 64 short ragged sequences (lengths 1 .. 700, seeded; two of them emptied), k = 4 so the
# selection is sparse in the longer ones; the packed axis ends with tokens outside every
# sequence
# G = 16, 2 and 1 (the backward's 16 G-row chunks), d = 128 and 64
CFG16 = synth.CONFIGS["8k"].with_(name="varlen-g16", B=1, N=3000, H_q=32, H_kv=2, topk=8, seed=55)
CU16 = [0, 1200, 1201, 2333, 3000]
CFG2 = synth.CONFIGS["8k"].with_(name="varlen-g2", B=1, N=2600, H_q=8, H_kv=4, topk=6, n_needle=1,
                                  seed=56)
CU2 = [0, 129, 1300, 2600]
CFG1 = synth.CONFIGS["tiny"].with_(name="varlen-g1", N=2200, H_q=4, H_kv=4, topk=3, seed=57)
CU1 = [0, 700, 700, 1957, 2150]
CFG64 = synth.CONFIGS["tiny"].with_(name="varlen-64", N=20480, seed=53)
_LENS = np.diff(synth.varlen_offsets(64, 1, 700, seed=54))
_LENS[[5, 40]] = 0
CU64 = [0] + np.cumsum(_LENS).astype(int).tolist()


def _seq(h, c0, c1):
    """Inputs of one sequence as a B=1 problem (host bits)."""
    return {n: np.ascontiguousarray(h[n][:, c0:c1]) for n in h}


def _chain(cfg, cu, d, w, max_seqlen=None):
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    k = cfg.topk
    bi, li = ops.msa_index_topk_varlen(d["q_idx"], d["k_idx"], cu_t, k, max_seqlen=max_seqlen,
                                       H_q=cfg.H_q, d=cfg.d)
    o, lse = ops.msa_fwd_varlen(d["q"], d["k"], d["v"], bi, cu_t, k, max_seqlen=max_seqlen,
                                scale=cfg.scale, d_idx=cfg.d_idx)
    g = ops.msa_bwd_varlen(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li,
                           w, cu_t, k, max_seqlen=max_seqlen, scale=cfg.scale)
    assert ops.device_status() == 0
    return bi, li, o, lse, g


@pytest.mark.parametrize("cfg,cu", [(CFG, CU), (CFG8, CU8), (CFG16, CU16), (CFG2, CU2), (CFG1, CU1),
                                    (CFG64, CU64)],
                         ids=["tiny_mix", "g8_d128", "g16_d128", "g2_d128", "g1_d64", "64_ragged"])
def test_varlen_chain_matches_oracle_per_sequence(cfg, cu):
    h = host_inputs(cfg)
    T = cu[-1]
    assert T <= cfg.N
    d = {n: to_dev(h[n])[0].contiguous() for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
    H_kv, k = cfg.H_kv, cfg.topk
    w = cfg.kl_coef / (H_kv * T)
    bi, li, o, lse, g = _chain(cfg, cu, d, w)
    kl_ref, n_diff = 0.0, 0
    # gradients are compared over the whole batch at once (the tolerance scale is the
    # batch's gradient magnitude: a one-token sequence's dq is 0 up to rounding)
    got = {n: [] for n in ("dq", "dk", "dv", "dq_idx", "dk_idx")}
    want = {n: [] for n in got}
    for s in range(len(cu) - 1):
        c0, c1 = cu[s], cu[s + 1]
        L = c1 - c0
        if L == 0:
            continue
        cs = cfg.with_(N=L)
        hs = _seq(h, c0, c1)
        rows = np.arange(L, dtype=np.int64)
        gsel = ops.varlen_view(bi, cu, s, H_kv, k).cpu().numpy().transpose(1, 0, 2)
        sets, nd = validated_gpu_sets(cs, hs, gsel, rows)
        n_diff += nd
        o_ref, lse_ref, li_ref = oracle.forward(cs, hs, sets)
        li_g = ops.varlen_view(li, cu, s, H_kv).cpu().numpy()[:, :, 0].T
        assert np.abs(li_g - li_ref).max() <= LSE_TOL, f"seq {s}: lse_idx"
        eo = np.abs(f64(o[c0:c1]) - o_ref).max()
        el = np.abs(ops.varlen_view(lse, cu, s, cfg.H_q).cpu().numpy()[:, :, 0].T - lse_ref).max()
        assert eo <= O_TOL and el <= LSE_TOL, (s, eo, el)
        ref = oracle.backward(cs, hs, sets, w)
        for n in got:
            got[n].append(f64(g[n][c0:c1]).reshape(L, -1))
            want[n].append(np.asarray(ref[n]).reshape(L, -1))
        kl_ref += ref["kl"]
    for n in got:
        grad_close(np.concatenate(got[n]), np.concatenate(want[n]), n)
    kl = float(g["kl"].cpu())
    print(f"{cfg.name}: {len(cu) - 1} sequences, {n_diff} rows on another valid set")
    assert abs(kl - kl_ref) <= KL_REL * abs(kl_ref) + 1e-6, (kl, kl_ref)


def test_launches_do_not_depend_on_the_number_of_sequences():
    cfg = CFG64
    h = host_inputs(cfg)
    d = {n: to_dev(h[n])[0].contiguous() for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
    T = CU64[-1]
    w = cfg.kl_coef / (cfg.H_kv * T)
    counts = []
    for cu in ([0, T], [0, 700, 1400, T], CU64):
        _chain(cfg, [0, T], d, w, max_seqlen=T)  # warm the workspace
        n0 = _lib.msa_kernel_launch_count()
        _chain(cfg, cu, d, w, max_seqlen=T)
        counts.append(_lib.msa_kernel_launch_count() - n0)
    assert len(set(counts)) == 1, counts


def test_bad_offsets_are_reported_by_the_device():
    cfg = CFG
    h = host_inputs(cfg)
    d = {n: to_dev(h[n])[0].contiguous() for n in ("q_idx", "k_idx")}
    bad = torch.tensor([0, 600, 400, 1000], dtype=torch.int32, device="cuda")  # decreasing
    block_idx = torch.full((cfg.H_kv * cfg.N * cfg.topk,), -7, dtype=torch.int32, device="cuda")
    lse_idx = torch.full((cfg.H_kv * cfg.N,), 3.0, dtype=torch.float32, device="cuda")
    prob = ops.make_problem(1, 1000, cfg.H_q, cfg.H_kv, cfg.d, cfg.d_idx, cfg.topk, 128, True,
                            None, None)
    nws = _lib.msa_workspace_size_varlen(prob, 3, cfg.N, _lib.MSA_WS_INDEX)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    rc = _lib.msa_index_topk_varlen(prob, bad.data_ptr(), 3, cfg.N, d["q_idx"].data_ptr(),
                                    d["k_idx"].data_ptr(), block_idx.data_ptr(),
                                    lse_idx.data_ptr(), ws.data_ptr(), nws,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.MSA_OK  # the host does not read cu_seqlens
    assert ops.device_status() == _lib.MSA_ERR_ARG
    assert (block_idx == -7).all() and (lse_idx == 3.0).all()  # nothing written
    # a sequence longer than max_seqlen is refused the same way
    long = torch.tensor([0, 1001], dtype=torch.int32, device="cuda")
    rc = _lib.msa_index_topk_varlen(prob, long.data_ptr(), 1, cfg.N, d["q_idx"].data_ptr(),
                                    d["k_idx"].data_ptr(), block_idx.data_ptr(),
                                    lse_idx.data_ptr(), ws.data_ptr(), nws,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.MSA_OK and ops.device_status() == _lib.MSA_ERR_ARG
    assert (block_idx == -7).all()
