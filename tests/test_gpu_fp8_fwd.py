"""GPU parity of the FP8 (E4M3) training forward (msa_quantize_fwd_fp8 + msa_fwd_fp8)
against the oracle's FP8 forward (oracle/fp8.py, forward_fp8), through the C ABI.

The quantisers are encodings and must reproduce the oracle's codes and scales bit for
bit: q per (token, head) row, k per 128-key block (layout kept), v per block and
transposed within it.  The forward is compared on sampled rows with the oracle's
block sets as input: o within 2e-2 max-abs and lse within 1e-3 of the FP8 oracle; the
distance to the float64 bf16 forward (the FP8 error itself) is printed beside it.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from block_sparse_gqa_topk_gb300 import ops, synth
from gpu_inputs import device_inputs, rows_for
from parity import LSE_TOL, O_TOL, f64
from test_gpu_index_fwd import cfg_of

pytestmark = pytest.mark.gpu

CASES = [("k8_d128", 96), ("g16_d128", 64), ("g2_d128", 64), ("8k", 64), ("32k", 48),
         ("128k", 32), ("1m", 24)]


def _sets(cfg, h, rows):
    """Oracle block sets of the sampled rows; every other row gets a valid local window."""
    bi_ref, _, _ = oracle.select(cfg, h, rows=rows)
    i = np.arange(cfg.N)
    ci = i // cfg.Bk
    base = ci[:, None] - np.arange(cfg.topk)[None, ::-1]
    base = np.sort(np.where(base < 0, 1 << 30, base), axis=1)
    base = np.where(base == 1 << 30, -1, base).astype(np.int32)
    full = np.broadcast_to(base, (cfg.B, cfg.H_kv, cfg.N, cfg.topk)).copy()
    full[rows // cfg.N, :, rows % cfg.N, :] = bi_ref
    return bi_ref, torch.from_numpy(np.ascontiguousarray(full, dtype=np.int32)).cuda()


@pytest.mark.parametrize("name", ["k8_d128", "8k", "128k"])
def test_fp8_quantisers_are_bit_exact(name):
    cfg = cfg_of(name)
    h, d = device_inputs(cfg, names=("q", "k", "v"))
    q8, qs, k8, ks, v8t, vs = ops.msa_quantize_fwd_fp8(d["q"], d["k"], d["v"])
    assert ops.device_status() == 0
    rng = np.random.default_rng(3)
    # q: sampled tokens (every head); k, v: sampled blocks (the last, ragged or not, too)
    toks = np.unique(np.concatenate([rng.integers(0, cfg.N, 64), [0, cfg.N - 1]]))
    for b in range(cfg.B):
        rc, rs = fp8.quantize_rows(h["q"][b, toks])
        assert np.array_equal(q8[b, toks].cpu().numpy(), rc)
        assert np.array_equal(qs[b, toks].cpu().numpy(), rs)
    nb = (cfg.N + cfg.Bk - 1) // cfg.Bk
    blocks = np.unique(np.concatenate([rng.integers(0, nb, 12), [0, nb - 1]]))
    k8h, v8h = k8.cpu().numpy(), v8t.cpu().numpy()
    ksh, vsh = ks.cpu().numpy(), vs.cpu().numpy()
    for b in range(cfg.B):
        for c in blocks:
            sl = slice(c * cfg.Bk, min(cfg.N, (c + 1) * cfg.Bk))
            n = sl.stop - sl.start
            kc, kref = fp8.quantize_blocks(h["k"][b:b + 1, sl], cfg.Bk)
            vc, vref = fp8.quantize_blocks(h["v"][b:b + 1, sl], cfg.Bk)
            assert np.array_equal(k8h[b, sl], kc[0])
            assert np.array_equal(ksh[b, :, c], kref[0, :, 0])
            assert np.array_equal(vsh[b, :, c], vref[0, :, 0])
            # v8t[b, g, c] is the block's [d][128 keys] tile, keys past N are 0
            vt = v8h[b, :, c]                                 # [H_kv, d, Bk]
            assert np.array_equal(vt[:, :, :n], vc[0].transpose(1, 2, 0))
            assert not vt[:, :, n:].any()


@pytest.mark.parametrize("name,n_rows", CASES)
def test_fwd_fp8_matches_fp8_oracle(name, n_rows):
    cfg = cfg_of(name)
    h, d = device_inputs(cfg, names=("q", "k", "v"))
    rows, _ = rows_for(cfg, n_rows, seed=13)
    bi_ref, block_idx = _sets(cfg, h, rows)
    q8, qs, k8, ks, v8t, vs = ops.msa_quantize_fwd_fp8(d["q"], d["k"], d["v"])
    o, lse = ops.msa_fwd_fp8(q8, qs, k8, ks, v8t, vs, block_idx, scale=cfg.scale, d_idx=cfg.d_idx)
    assert ops.device_status() == 0
    b, i = rows // cfg.N, rows % cfg.N
    o_g = f64(o)[b, i]
    lse_g = lse.cpu().numpy()[b, :, i]
    o_ref, lse_ref = fp8.forward_fp8(h, bi_ref, rows, cfg.scale, cfg.G, cfg.Bk)
    eo = np.abs(o_g - o_ref).max()
    el = np.abs(lse_g - lse_ref).max()
    o64, lse64, _ = oracle.forward(cfg, h, bi_ref, rows=rows, index=False)
    print(f"{name}: o max-abs {eo:.3e} lse {el:.3e} (vs FP8 oracle); "
          f"FP8 vs bf16 float64 forward: o {np.abs(o_g - o64).max():.3e} "
          f"lse {np.abs(lse_g - lse64).max():.3e}")
    assert eo <= O_TOL and el <= LSE_TOL, (eo, el)
