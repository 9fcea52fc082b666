"""Pins of the FP8 (E4M3) KV-cache oracle (oracle/fp8.py) against what the format and a
library fix: PyTorch's own float8_e4m3fn type decodes and rounds every value the same
way (where it does not overflow), closed-form codes, saturation, the round trip, the
quantisation error bound, and -- for caches whose dequantised values are exactly
bf16 -- equality with the main float64 oracle's forward on the last row."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from block_sparse_gqa_topk_gb300 import synth


def _torch_codes(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_decode_table_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.e4m3_decode(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_decode_closed_forms():
    v = fp8.e4m3_decode(np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0x40, 0xB8, 0x39, 0x00],
                                 dtype=np.uint8))
    assert list(v) == [448.0, 2.0 ** -6, 7 * 2.0 ** -9, 2.0 ** -9, 1.0, 2.0, -1.0, 1.125, 0.0]
    assert np.isnan(fp8.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    assert np.signbit(fp8.e4m3_decode(np.array([0x80], dtype=np.uint8))[0])
    finite = fp8.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert len(np.unique(finite[~np.isnan(finite)])) == 253  # 254 finite codes, +0 = -0


def test_encode_matches_library_in_range():
    rng = np.random.default_rng(5)
    mags = np.exp2(rng.uniform(-13.0, np.log2(460.0), size=20000))
    pos = fp8.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[1:] + pos[:-1]) / 2          # exact ties
    near = np.concatenate([np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    x = np.concatenate([mags, pos, mids, near]).astype(np.float32)
    x = np.concatenate([x, -x, np.array([0.0, -0.0, -1e-12], dtype=np.float32)])
    x = x[np.abs(x) < 464.0]                 # the library's float8 overflows to NaN above
    assert np.array_equal(fp8.e4m3_encode(x), _torch_codes(x))


def test_ties_go_to_the_even_code_and_large_values_saturate():
    assert fp8.e4m3_encode(np.float32(1.0625))[()] == 0x38    # between 1 (0x38) and 1.125
    assert fp8.e4m3_encode(np.float32(1.1875))[()] == 0x3A    # between 1.125 and 1.25
    assert fp8.e4m3_encode(np.float32(2.0 ** -10))[()] == 0x00  # half the smallest subnormal
    big = np.array([464.0, 1000.0, 3e38, -464.0, -3e38], dtype=np.float32)
    assert list(fp8.e4m3_encode(big)) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    assert fp8.e4m3_encode(np.float32(np.nan))[()] == 0x7F


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes).astype(np.float32)), codes)


def test_quantize_rows_error_bound_and_scale():
    cfg = synth.CONFIGS["tiny"]
    h = synth.make_inputs(cfg, names=("k",))
    bits = h["k"][0, :512].copy()                      # [512, H_kv, d]
    bits[3, 1] = 0                                     # an all-zero row
    codes, s = fp8.quantize_rows(bits)
    x = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    deq = fp8.dequantize_rows(codes, s)
    assert s[3, 1] == 1.0 and not codes[3, 1].any()
    err = np.abs(deq - x)
    assert (err <= 2.0 ** -4 * np.abs(x) + s[..., None] * 2.0 ** -10).all()
    # every non-zero row uses the full range: its largest magnitude encodes to 448 and
    # dequantises back to the row's amax up to the scale's float32 rounding
    amax = np.abs(x).max(axis=-1)
    nz = amax > 0
    assert ((codes & 0x7F).max(axis=-1)[nz] == 0x7E).all()
    assert (np.abs(np.abs(deq).max(axis=-1) - amax)[nz] <= 2.0 ** -22 * amax[nz]).all()


def test_decode_attention_equals_main_oracle_on_bf16_exact_caches():
    # codes times power-of-two scales are exact bf16 values, so the fp8 decode oracle
    # must equal the float64 forward oracle's last row on the same cache
    cfg = synth.CONFIGS["tiny"].with_(name="fp8-pin", B=2, N=1300, seed=81)
    h = synth.make_inputs(cfg)
    rng = np.random.default_rng(9)
    lens = [1300, 700]
    B, L, H_kv, d = h["k"].shape
    deq = {}
    for n in ("k", "v"):
        codes = rng.integers(0, 256, size=(B, L, H_kv, d)).astype(np.uint8)
        codes = np.where((codes & 0x7F) == 0x7F, codes & 0xF0, codes).astype(np.uint8)  # no NaN
        scale = np.exp2(rng.integers(-6, 0, size=(B, L, H_kv))).astype(np.float32)
        deq[n] = fp8.dequantize_rows(codes, scale)
        bits = (deq[n].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), deq[n])
        h = dict(h, **{n: bits})
    q_new = np.stack([h["q"][b, lens[b] - 1] for b in range(B)])
    sel = np.full((B, H_kv, cfg.topk), -1, dtype=np.int32)
    for b, Lb in enumerate(lens):
        cb = cfg.with_(B=1, N=Lb)
        hb = {n: np.ascontiguousarray(h[n][b:b + 1, :Lb]) for n in h}
        rows = np.array([Lb - 1], dtype=np.int64)
        bi, _, _ = oracle.select(cb, hb, rows=rows)
        sel[b] = bi[0]
    o, lse = fp8.decode_attention(q_new, deq["k"], deq["v"], sel, lens, cfg.scale)
    for b, Lb in enumerate(lens):
        cb = cfg.with_(B=1, N=Lb)
        hb = {n: np.ascontiguousarray(h[n][b:b + 1, :Lb]) for n in h}
        rows = np.array([Lb - 1], dtype=np.int64)
        o_ref, lse_ref, _ = oracle.forward(cb, hb, sel[b][None], rows=rows, index=False)
        np.testing.assert_allclose(o[b], o_ref[0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[b], lse_ref[0], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("plant", ["no_tie_even", "no_saturate", "scale_off_by_one"])
def test_planted_mistakes_fail_a_pin(plant, monkeypatch):
    """A plausible mistake in the quantiser or codec breaks one of the pins above."""
    if plant == "no_tie_even":
        def enc(x, _orig=fp8.e4m3_encode):
            c = _orig(x)
            a = np.abs(np.asarray(x, dtype=np.float32).astype(np.float64))
            pos = fp8._POS
            hi = np.clip(np.searchsorted(pos, a), 0, len(pos) - 1)
            tie = (hi > 0) & (pos[hi] - a == a - pos[np.maximum(hi - 1, 0)])
            return np.where(tie, (c & 0x80) | hi.astype(np.uint8), c).astype(np.uint8)  # ties up
        monkeypatch.setattr(fp8, "e4m3_encode", enc)
        with pytest.raises(AssertionError):
            test_ties_go_to_the_even_code_and_large_values_saturate()
    elif plant == "no_saturate":
        def enc(x, _orig=fp8.e4m3_encode):
            c = _orig(x)
            big = np.abs(np.asarray(x, dtype=np.float32)) > 464.0
            return np.where(big, (c & 0x80) | 0x7F, c).astype(np.uint8)
        monkeypatch.setattr(fp8, "e4m3_encode", enc)
        with pytest.raises(AssertionError):
            test_ties_go_to_the_even_code_and_large_values_saturate()
    else:
        def q(x_bits, _orig=fp8.quantize_rows):
            c, s = _orig(x_bits)
            return c, (s * np.float32(1.01)).astype(np.float32)  # scale not matched to codes
        monkeypatch.setattr(fp8, "quantize_rows", q)
        with pytest.raises(AssertionError):
            test_quantize_rows_error_bound_and_scale()
