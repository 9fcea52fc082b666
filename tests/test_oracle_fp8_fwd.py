"""Pins of the FP8 training-forward oracle (oracle/fp8.py: quantize_blocks,
attend_block_e4m3, forward_fp8) against what the format, closed forms and the float64
main oracle fix:

* the per-block quantiser is the per-row quantiser (pinned against PyTorch's float8 in
  test_oracle_fp8.py) applied to the block's values laid out as one row;
* one block's softmax with P rounded to E4M3, on a hand-worked example;
* with q = 0 every score is 0, so P = 1 exactly: o is the plain mean of the dequantised
  v over the token set and lse = log |T|, whatever the blocks;
* against the float64 main oracle on the bf16 inputs the FP8 forward stays within the
  format's error (a dropped scale or a wrong block's scale is far outside it);
* planted mistakes fail one of these pins.
"""
import numpy as np
import pytest

import oracle
from oracle import fp8
from block_sparse_gqa_topk_gb300 import synth

CFG = synth.CONFIGS["tiny"].with_(name="fp8-fwd-pin", N=700, d=128, d_idx=64, H_q=8, H_kv=2,
                                  topk=3, seed=91)


def _rows(cfg, n=24, seed=5):
    return synth.sample_rows(cfg, n, seed)


def test_quantize_blocks_is_the_row_quantiser_on_each_block():
    h = synth.make_inputs(CFG, names=("k",))
    codes, scale = fp8.quantize_blocks(h["k"], CFG.Bk)
    B, N, H, d = h["k"].shape
    nb = (N + CFG.Bk - 1) // CFG.Bk
    assert scale.shape == (B, H, nb)
    for b in range(B):
        for g in range(H):
            for c in range(nb):
                sl = slice(c * CFG.Bk, min(N, (c + 1) * CFG.Bk))
                row = np.ascontiguousarray(h["k"][b, sl, g].reshape(1, -1))  # the block as one row
                rc, rs = fp8.quantize_rows(row)
                assert rs[0] == scale[b, g, c]
                assert np.array_equal(rc[0], codes[b, sl, g].reshape(-1))


def test_quantize_blocks_zero_block_has_unit_scale():
    h = synth.make_inputs(CFG, names=("v",))
    bits = h["v"].copy()
    bits[:, 128:256, 1] = 0
    codes, scale = fp8.quantize_blocks(bits, CFG.Bk)
    assert (scale[:, 1, 1] == 1.0).all() and not codes[:, 128:256, 1].any()


def test_attend_block_hand_example():
    # scores 0 and ln 0.3: P = (1, 0.3); E4M3(0.3) = 1.25 * 2^-2 = 0.3125 (1.2 is nearer
    # 1.25 than 1.125); o = (1 * 1 + 0.3125 * 2) / 1.3 = 1.25; lse = 0 + ln 1.3
    o, lse = fp8.attend_block_e4m3(np.array([0.0, np.log(0.3)]), np.array([[1.0], [2.0]]))
    assert o[0] == pytest.approx(1.25, abs=1e-12)
    assert lse == pytest.approx(np.log(1.3), abs=1e-12)
    # a single token: P = 1, o = v, lse = s
    o, lse = fp8.attend_block_e4m3(np.array([-3.5]), np.array([[0.75, -2.0]]))
    assert np.array_equal(o, [0.75, -2.0]) and lse == -3.5


def test_forward_fp8_with_zero_q_is_the_mean_of_the_dequantised_v():
    h = dict(synth.make_inputs(CFG))
    h["q"] = np.zeros_like(h["q"])
    rows = _rows(CFG)
    bi, _, _ = oracle.select(CFG, h, rows=rows)
    o, lse = fp8.forward_fp8(h, bi, rows, CFG.scale, CFG.G, CFG.Bk)
    v8, sv = fp8.quantize_blocks(h["v"], CFG.Bk)
    vd = fp8.e4m3_decode(v8)
    N = CFG.N
    for r, row in enumerate(rows):
        b, i = int(row // N), int(row % N)
        for g in range(CFG.H_kv):
            toks = [j for c in bi[r, g] if c >= 0 for j in range(c * CFG.Bk, min((c + 1) * CFG.Bk, i + 1))]
            ref = np.mean([vd[b, j, g] * sv[b, g, j // CFG.Bk] for j in toks], axis=0)
            for h_ in range(g * CFG.G, (g + 1) * CFG.G):
                np.testing.assert_allclose(o[r, h_], ref, rtol=0, atol=1e-12)
                assert lse[r, h_] == pytest.approx(np.log(len(toks)), abs=1e-12)


def test_forward_fp8_is_close_to_the_float64_forward():
    h = synth.make_inputs(CFG)
    rows = _rows(CFG, 32, 6)
    bi, _, _ = oracle.select(CFG, h, rows=rows)
    o8, lse8 = fp8.forward_fp8(h, bi, rows, CFG.scale, CFG.G, CFG.Bk)
    o, lse, _ = oracle.forward(CFG, h, bi, rows=rows, index=False)
    # E4M3 keeps 3 mantissa bits (relative step 2^-3, error <= 2^-4): the scores move by a
    # few percent of their spread, P by up to 2^-4 of itself, o by a few 1e-2
    assert np.abs(o8 - o).max() < 0.1
    assert np.abs(lse8 - lse).max() < 0.1
    # and the error is not zero: the oracle does apply the 8-bit rounding
    assert np.abs(o8 - o).max() > 1e-4


@pytest.mark.parametrize("plant", ["v_scale_dropped", "sum_of_rounded_p", "k_scale_of_block_0"])
def test_planted_mistakes_fail_a_pin(plant, monkeypatch):
    if plant == "v_scale_dropped":
        calls = []

        def qb(x_bits, Bk=128, _orig=fp8.quantize_blocks):
            c, s = _orig(x_bits, Bk)
            calls.append(1)
            # forward_fp8 quantises k first, then v: v loses its scale
            return (c, np.ones_like(s)) if len(calls) == 2 else (c, s)
        monkeypatch.setattr(fp8, "quantize_blocks", qb)
        with pytest.raises(AssertionError):
            test_forward_fp8_with_zero_q_is_the_mean_of_the_dequantised_v()
    elif plant == "sum_of_rounded_p":
        def att(s, v):
            m = s.max()
            p8 = fp8.e4m3_decode(fp8.e4m3_encode(np.exp(s - m).astype(np.float32)))
            return (p8 @ v) / p8.sum(), m + np.log(p8.sum())
        monkeypatch.setattr(fp8, "attend_block_e4m3", att)
        with pytest.raises(AssertionError):
            test_attend_block_hand_example()
    else:
        def qb(x_bits, Bk=128, _orig=fp8.quantize_blocks):
            c, s = _orig(x_bits, Bk)
            return c, np.repeat(s[:, :, :1], s.shape[2], axis=2)  # every block takes block 0's
        monkeypatch.setattr(fp8, "quantize_blocks", qb)
        with pytest.raises(AssertionError):
            test_quantize_blocks_is_the_row_quantiser_on_each_block()
