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
