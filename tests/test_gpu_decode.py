"""GPU parity of the decode entry point (msa_decode) against the float64 oracle: for a
cache of length L, the new token's selection, output and lse must equal row L-1 of the
training path on the cache (the oracle's select and forward on that one row; the
near-tie rule applies to the selection)."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import host_inputs, tie_inputs
from parity import LSE_TOL, O_TOL, check_selection, f64, to_dev

pytestmark = pytest.mark.gpu

T = synth.CONFIGS["tiny"]
CASES = {
    "tiny": (T.with_(name="dec-tiny", B=3, seed=61), [2048, 1300, 1]),
    "ragged": (T.with_(name="dec-ragged", B=2, N=2000, seed=62), [2000, 129]),
    "g16": (T.with_(name="dec-g16", H_q=32, H_kv=2, N=1024, B=2, seed=63), [1024, 700]),
    "8k": (synth.CONFIGS["8k"], [8192, 5001]),
    # 24 groups (two group tiles of the pooling), G = 2, d = 64 with d_idx = 64, k = 20
    "wide": (T.with_(name="dec-wide", H_q=48, H_kv=24, d_idx=64, topk=20, N=3000, B=2,
                     seed=64), [3000, 2561]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_matches_oracle_last_row(name):
    cfg, lens = CASES[name]
    h = host_inputs(cfg)
    d = {n: to_dev(h[n]) for n in ("q", "k", "v", "q_idx", "k_idx")}
    bsel = torch.arange(cfg.B, device="cuda")
    last = torch.tensor([L - 1 for L in lens], device="cuda")
    q_new = d["q"][bsel, last].contiguous()          # [B, H_q, d]
    qi_new = d["q_idx"][bsel, last].contiguous()     # [B, H_kv, d_idx]
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    bi, o, lse = ops.msa_decode(q_new, qi_new, d["k"], d["v"], d["k_idx"], lens_t, cfg.topk,
                                scale=cfg.scale)
    assert ops.device_status() == 0
    bi, o, lse = bi.cpu().numpy(), f64(o), lse.cpu().numpy()
    for b, L in enumerate(lens):
        cb = cfg.with_(B=1, N=L)
        hb = {n: np.ascontiguousarray(h[n][b:b + 1, :L]) for n in h}
        rows = np.array([L - 1], dtype=np.int64)
        bi_ref, kth, _ = oracle.select(cb, hb, rows=rows)
        check_selection(cb, hb, bi[b][None], rows, bi_ref, kth)
        # the output follows the set the GPU took (equal to the oracle's outside the
        # near-tie band, a valid set inside it): the oracle reruns on that set
        o_ref, lse_ref, _ = oracle.forward(cb, hb, bi[b][None], rows=rows, index=False)
        eo = np.abs(o[b] - o_ref[0]).max()
        el = np.abs(lse[b] - lse_ref[0]).max()
        assert eo <= O_TOL and el <= LSE_TOL, (name, b, eo, el)


def test_decode_exact_ties_keep_the_lower_block():
    """Key blocks that are block 0 scaled by 1, 2 or 4 pool to exact multiples of one
    another on the decode path's mma.sync pooling as in the oracle, so the last row sees
    runs of equal block scores longer than the k - 1 free slots: the decode selection
    (ranked on (score, -block) keys) must take the oracle's set exactly."""
    cfg = T.with_(name="dec-ties", B=2, N=4096, topk=6, seed=66)
    h, _ = tie_inputs(cfg, names=("q", "k", "v", "q_idx", "k_idx"))
    d = {n: to_dev(h[n]) for n in ("q", "k", "v", "q_idx", "k_idx")}
    lens = [4096, 3001]
    bsel = torch.arange(cfg.B, device="cuda")
    last = torch.tensor([L - 1 for L in lens], device="cuda")
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    bi, _, _ = ops.msa_decode(d["q"][bsel, last].contiguous(), d["q_idx"][bsel, last].contiguous(),
                              d["k"], d["v"], d["k_idx"], lens_t, cfg.topk, scale=cfg.scale)
    assert ops.device_status() == 0
    bi = bi.cpu().numpy()
    for b, L in enumerate(lens):
        cb = cfg.with_(B=1, N=L)
        hb = {n: np.ascontiguousarray(h[n][b:b + 1, :L]) for n in h}
        bi_ref, _, _ = oracle.select(cb, hb, rows=np.array([L - 1], dtype=np.int64))
        assert np.array_equal(bi[b], bi_ref[0]), (b, bi[b], bi_ref[0])


def test_decode_invalid_length_is_reported_and_bounded():
    """A cache length outside [1, Lmax] is recorded as MSA_ERR_ARG in the status word and
    the row is served as a one-token cache (no access past the cache)."""
    from block_sparse_gqa_topk_gb300 import _lib
    cfg = T.with_(name="dec-bad-len", B=2, N=1024, seed=65)
    h = host_inputs(cfg)
    d = {n: to_dev(h[n]) for n in ("q", "k", "v", "q_idx", "k_idx")}
    q_new = d["q"][:, 0].contiguous()
    qi_new = d["q_idx"][:, 0].contiguous()
    for bad in (0, cfg.N + 1):
        lens_t = torch.tensor([bad, 1], dtype=torch.int32, device="cuda")
        bi, o, lse = ops.msa_decode(q_new, qi_new, d["k"], d["v"], d["k_idx"], lens_t, cfg.topk,
                                    scale=cfg.scale)
        assert ops.device_status() == _lib.MSA_ERR_ARG
        bi = bi.cpu().numpy()
        assert (bi[:, :, 0] == 0).all() and (bi[:, :, 1:] == -1).all()
        # both rows: attention over token 0 alone, o = v[b, 0] of the head's group
        o = f64(o)
        for b in range(cfg.B):
            for hq in range(cfg.H_q):
                ref = f64(d["v"][b, 0, hq // cfg.G])
                assert np.abs(o[b, hq] - ref).max() <= O_TOL
    assert ops.device_status() == 0
