"""Cached seeded inputs for the GPU tests (host bits + device tensors)."""
import functools

import numpy as np

from block_sparse_gqa_topk_gb300 import synth


@functools.lru_cache(maxsize=2)
def host_inputs(cfg: synth.MSAConfig):
    return synth.make_inputs(cfg)


def device_inputs(cfg, names=("q", "k", "v", "q_idx", "k_idx", "dO")):
    from parity import to_dev
    h = host_inputs(cfg)
    return h, {n: to_dev(h[n]) for n in names}


def rows_for(cfg, n_rows, seed=77):
    if n_rows is None:
        return None, np.arange(cfg.B * cfg.N, dtype=np.int64)
    r = synth.sample_rows(cfg, n_rows, seed)
    return r, r


def tie_inputs(cfg, seed=46, names=("q_idx", "k_idx")):
    """Host inputs whose key blocks are copies of block 0 scaled by 1, 2 or 4 (seeded).

    Scaling bf16 values by a power of two is exact, and so is every partial sum of the
    scores, in float32 as in float64: a query's pooled block scores are its block-0
    score times 1, 2 or 4, exactly.  Each query therefore sees runs of exactly equal
    scores, which only the lower-block tie rule orders.
    """
    h = dict(synth.make_inputs(cfg, names=tuple(names)))
    nb = cfg.N // cfg.Bk
    ki = synth.bf16_bits_to_f32(h["k_idx"]).reshape(cfg.B, nb, cfg.Bk, cfg.d_idx)
    scale = 2.0 ** np.random.default_rng(seed).integers(0, 3, size=nb)
    ki = ki[:, :1] * scale[None, :, None, None]
    h["k_idx"] = synth.f32_to_bf16_bits(ki.reshape(cfg.B, cfg.N, cfg.d_idx).astype(np.float32))
    return h, scale
