"""The oracle against a hand-worked example (tests/golden/hand_example.json) and
against exact ties in the block ranking."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from block_sparse_gqa_topk_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "log": math.log, "exp": math.exp}))


def test_hand_example():
    gd = json.load(open(GOLDEN))
    p = gd["problem"]
    cfg = synth.MSAConfig("hand", B=p["B"], N=p["N"], H_q=p["H_q"], H_kv=p["H_kv"], d=p["d"],
                          d_idx=p["d_idx"], Bk=p["Bk"], topk=p["topk"], causal=bool(p["causal"]))
    over = {"scale": p["scale"], "scale_idx": p["scale_idx"]}
    shp = synth.shapes(cfg)
    inp = {n: synth.f32_to_bf16_bits(np.array(v, dtype=np.float32)).reshape(shp[n])
           for n, v in gd["inputs"].items()}
    ex = gd["expected"]
    bi, _, _ = oracle.select(cfg, inp, **over)
    np.testing.assert_array_equal(bi[:, 0, :], np.array(ex["block_idx"]))
    o, lse, lse_idx = oracle.forward(cfg, inp, bi, **over)
    for name, got in (("o", o.ravel()), ("lse", lse.ravel()), ("lse_idx", lse_idx.ravel())):
        want = [_ev(s) for s in ex[name]]
        np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14, err_msg=name)
    g = oracle.backward(cfg, inp, bi, 1.0, **over)
    np.testing.assert_allclose(g["kl_rows"].ravel(), [_ev(s) for s in ex["kl_rows"]],
                               rtol=1e-12, atol=1e-14)
    assert g["kl"] == pytest.approx(sum(_ev(s) for s in ex["kl_rows"]), rel=1e-12)
    g0 = oracle.backward(cfg, inp, bi, 0.0, **over)
    for name in ("dk", "dv", "dq"):
        np.testing.assert_allclose(g0[name].ravel(), [_ev(s) for s in ex[name]],
                                   rtol=1e-14, atol=1e-14, err_msg=name)
    assert np.all(g0["dq_idx"] == 0) and np.all(g0["dk_idx"] == 0)


def test_exact_ties_rank_lower_block_first():
    """Pooled scores tie exactly: the lower block id is ranked first (reading of the
    pages, which do not fix a tie rule)."""
    cfg = synth.MSAConfig("ties", B=1, N=8 * 16, H_q=2, H_kv=1, d=8, d_idx=4, Bk=16, topk=3,
                          seed=3)
    inp = synth.make_inputs(cfg)
    one = synth.f32_to_bf16_bits(np.ones(4, dtype=np.float32))
    inp["q_idx"][:] = one
    ki = np.zeros((1, cfg.N, 4), dtype=np.float32)
    # every block has the same maximum (token 5 of each block = 1), except block 4 (=2)
    ki[0, 5::16, :] = 0.25
    ki[0, 4 * 16 + 5, :] = 0.5
    inp["k_idx"] = synth.f32_to_bf16_bits(ki)
    bi, kth, _ = oracle.select(cfg, inp)
    # last query (block 7): candidates 0..6, block 4 best, then tie among 0,1,2,3,5,6 -> 0
    assert list(bi[cfg.N - 1, 0]) == [0, 4, 7]
    # query in block 3: candidates 0,1,2 all tied -> 0, 1
    assert list(bi[3 * 16 + 2, 0]) == [0, 1, 3]
    assert kth[3 * 16 + 2, 0, 0] == kth[3 * 16 + 2, 0, 1] == 1.0
