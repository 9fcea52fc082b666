"""msa_index_topk_noalloc: the index branch for callers that cannot allocate device
memory (it takes its scratch from an array built into the library).  Its output
must match msa_index_topk with a caller workspace, call after call.

This file is collected last so that a run stopping at the first failure has
already run every other test; it sets up its own inputs so it also passes alone.
"""
import numpy as np
import pytest

from block_sparse_gqa_topk_gb300 import _lib, synth
from parity import LSE_TOL


def test_oversized_problem_is_rejected_before_any_launch():
    cfg = synth.CONFIGS["128k"]
    prob = _lib.Problem(B=cfg.B, N=cfg.N, H_q=cfg.H_q, H_kv=cfg.H_kv, d=cfg.d, d_idx=cfg.d_idx,
                        Bk=cfg.Bk, topk=cfg.topk, causal=1, scale=cfg.scale, scale_idx=0.0)
    assert _lib.msa_workspace_size(prob, _lib.MSA_WS_INDEX) > _lib.msa_noalloc_scratch_bytes()
    rc = _lib.msa_index_topk_noalloc(prob, 256, 256, 256, 256, None)
    assert rc == _lib.MSA_ERR_WORKSPACE


def _problem(cfg):
    return _lib.Problem(B=cfg.B, N=cfg.N, H_q=cfg.H_q, H_kv=cfg.H_kv, d=cfg.d, d_idx=cfg.d_idx,
                        Bk=cfg.Bk, topk=cfg.topk, causal=1, scale=cfg.scale, scale_idx=0.0)


def _compare_twice(cfg, with_lse=True):
    """Runs the workspace entry point once and the no-alloc one twice in a row on the
    same inputs; block sets must be identical and lse_idx within the LSE tolerance."""
    import torch
    from parity import to_dev

    h = synth.make_inputs(cfg, names=("q_idx", "k_idx"))
    qi, ki = to_dev(h["q_idx"]), to_dev(h["k_idx"])
    prob = _problem(cfg)
    need = _lib.msa_workspace_size(prob, _lib.MSA_WS_INDEX)
    assert 0 < need <= _lib.msa_noalloc_scratch_bytes()
    stream = torch.cuda.current_stream().cuda_stream

    def outputs():
        bi = torch.full((cfg.B, cfg.H_kv, cfg.N, cfg.topk), -7, dtype=torch.int32, device="cuda")
        li = torch.full((cfg.B, cfg.H_kv, cfg.N), float("nan"), dtype=torch.float32, device="cuda")
        return bi, li

    # reference: the workspace entry point
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    bi_ref, li_ref = outputs()
    _lib.check(_lib.msa_index_topk(prob, qi.data_ptr(), ki.data_ptr(), bi_ref.data_ptr(),
                                   li_ref.data_ptr(), ws.data_ptr(), need, stream),
               "msa_index_topk")
    for call in range(2):
        bi, li = outputs()
        _lib.check(_lib.msa_index_topk_noalloc(prob, qi.data_ptr(), ki.data_ptr(), bi.data_ptr(),
                                               li.data_ptr() if with_lse else None, stream),
                   "msa_index_topk_noalloc")
        assert _lib.msa_get_device_status(stream) == 0
        np.testing.assert_array_equal(bi.cpu().numpy(), bi_ref.cpu().numpy(),
                                      err_msg=f"{cfg.name} call {call}")
        if with_lse:
            err = float((li - li_ref).abs().max())
            assert err <= LSE_TOL, f"{cfg.name} call {call}: lse_idx differs by {err}"
        else:  # no lse_idx asked for: the output buffer is left alone
            assert torch.isnan(li).all()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    # a large problem first, then a ragged one (N not a multiple of 128, so the shared
    # array holds the larger call's leftovers beyond the small call's lists), then the
    # block-selection-only form (lse_idx NULL, no scratch used)
    _compare_twice(synth.CONFIGS["8k"])
    _compare_twice(synth.CONFIGS["tiny"].with_(name="ragged-noalloc", N=1000, B=3, seed=71))
    _compare_twice(synth.CONFIGS["tiny"].with_(name="sel-only-noalloc", N=1500, seed=72),
                   with_lse=False)
