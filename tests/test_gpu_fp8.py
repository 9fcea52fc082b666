"""GPU parity of the FP8 (E4M3) KV cache against the oracle (oracle/fp8.py).

The quantiser is an encoding, so its codes and scales must equal the oracle's bit for
bit.  Decode over the FP8 cache must equal the float64 decode attention over the
oracle's own dequantised cache, with the oracle's own block selection (the index
branch stays bf16), to the forward tolerances: P is rounded to bf16 after the V row
scale is folded into it, as in the bf16 path.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import host_inputs
from parity import LSE_TOL, O_TOL, check_selection, f64, to_dev

pytestmark = pytest.mark.gpu

T = synth.CONFIGS["tiny"]
CASES = {
    "tiny": (T.with_(name="f8-tiny", B=3, seed=91), [2048, 1300, 1]),
    "ragged": (T.with_(name="f8-ragged", B=2, N=2000, seed=92), [2000, 129]),
    "g16": (T.with_(name="f8-g16", H_q=32, H_kv=2, N=1024, B=2, seed=93), [1024, 700]),
    "8k": (synth.CONFIGS["8k"], [8192, 5001]),
    # 24 groups (two group tiles of the pooling), G = 2, d = 64 with d_idx = 64, k = 20
    "wide": (T.with_(name="f8-wide", H_q=48, H_kv=24, d_idx=64, topk=20, N=3000, B=2,
                     seed=94), [3000, 2561]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_quantizer_matches_oracle_bit_for_bit(name):
    cfg, _ = CASES[name]
    h = host_inputs(cfg)
    for n in ("k", "v"):
        x8, sc = ops.msa_quantize_kv_fp8(to_dev(h[n]))
        codes, s = fp8.quantize_rows(h[n])
        assert np.array_equal(x8.cpu().numpy(), codes), n
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), s.view(np.uint32)), n


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_fp8_matches_oracle(name):
    cfg, lens = CASES[name]
    h = host_inputs(cfg)
    d = {n: to_dev(h[n]) for n in ("q", "q_idx", "k", "v", "k_idx")}
    k8, ks = ops.msa_quantize_kv_fp8(d["k"])
    v8, vs = ops.msa_quantize_kv_fp8(d["v"])
    bsel = torch.arange(cfg.B, device="cuda")
    last = torch.tensor([L - 1 for L in lens], device="cuda")
    q_new = d["q"][bsel, last].contiguous()
    qi_new = d["q_idx"][bsel, last].contiguous()
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    bi, o, lse = ops.msa_decode_fp8(q_new, qi_new, k8, v8, ks, vs, d["k_idx"], lens_t, cfg.topk,
                                    scale=cfg.scale)
    assert ops.device_status() == 0
    bi, o, lse = bi.cpu().numpy(), f64(o), lse.cpu().numpy()
    # oracle: its own quantisation of the bf16 cache, its own selection
    kq, ks_ref = fp8.quantize_rows(h["k"])
    vq, vs_ref = fp8.quantize_rows(h["v"])
    k_deq, v_deq = fp8.dequantize_rows(kq, ks_ref), fp8.dequantize_rows(vq, vs_ref)
    q_bits = np.stack([h["q"][b, L - 1] for b, L in enumerate(lens)])
    sel = np.zeros_like(bi)
    for b, L in enumerate(lens):
        cb = cfg.with_(B=1, N=L)
        hb = {n: np.ascontiguousarray(h[n][b:b + 1, :L]) for n in h}
        rows = np.array([L - 1], dtype=np.int64)
        bi_ref, kth, _ = oracle.select(cb, hb, rows=rows)
        check_selection(cb, hb, bi[b][None], rows, bi_ref, kth)
        # the output follows the set the GPU took (the oracle's outside the near-tie
        # band, a valid set inside it): the oracle's decode runs on that set
        sel[b] = bi[b]
    o_ref, lse_ref = fp8.decode_attention(q_bits, k_deq, v_deq, sel, lens, cfg.scale)
    for b in range(cfg.B):
        eo = np.abs(o[b] - o_ref[b]).max()
        el = np.abs(lse[b] - lse_ref[b]).max()
        assert eo <= O_TOL and el <= LSE_TOL, (name, b, eo, el)
