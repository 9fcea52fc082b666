"""Seeded synthetic inputs for the MSA training hot path.

This module draws random numbers and rounds them to bf16; it holds none of the
method's arithmetic. Both the GPU path (tests, bench) and the float64 oracle take
their inputs from here, and from nowhere else.

Workloads follow the MSA description (MiniMax Sparse Attention summary,
7minutos.es, "Cómo funcionan las dos ramas"): GQA with H_q query heads in H_kv
groups, one index-query head per group and one shared index-key head, 128-token
blocks, k selected blocks per query and group.

Distribution: every tensor is N(0, 1) in float32. For the "needle" workloads,
n_needle distinct blocks per group, drawn uniformly from [1, nb/2) (far from the
late queries), get a +2.0 shift along a seeded unit direction u_g in k_idx and
v_g in the group's k head; every q_idx row of group g is shifted by 0.5 * u_g.
The result is rounded to bf16 (round to nearest, ties to even) and returned as
raw uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# tensor ids: each tensor draws from its own stream, spawned from the config seed
_TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "q_idx": 3, "k_idx": 4, "dO": 5}
_CHUNK_ELEMS = 1 << 22  # fixed chunking keeps the stream independent of thread count


@dataclasses.dataclass(frozen=True)
class MSAConfig:
    name: str
    B: int
    N: int
    H_q: int
    H_kv: int
    d: int
    d_idx: int
    Bk: int = 128
    topk: int = 16
    causal: bool = True
    n_needle: int = 0
    seed: int = 0
    needle_seed: int = 0
    kl_coef: float = 1.0

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv

    @property
    def nb(self) -> int:
        return (self.N + self.Bk - 1) // self.Bk

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def scale_idx(self) -> float:
        return 1.0 / float(np.sqrt(self.d_idx))

    def with_(self, **kw) -> "MSAConfig":
        return dataclasses.replace(self, **kw)


# The five workloads of the MSA training path (2K tiny .. 1M tokens); seed 1000+c,
# needle seed 2000+c for workload c.
CONFIGS = {
    "tiny": MSAConfig("tiny", B=1, N=2048, H_q=8, H_kv=2, d=64, d_idx=32, topk=4,
                      n_needle=0, seed=1000, needle_seed=2000),
    "8k": MSAConfig("8k", B=2, N=8192, H_q=16, H_kv=4, d=128, d_idx=64, topk=16,
                    n_needle=3, seed=1001, needle_seed=2001),
    "32k": MSAConfig("32k", B=1, N=32768, H_q=32, H_kv=8, d=128, d_idx=64, topk=16,
                     n_needle=8, seed=1002, needle_seed=2002),
    "128k": MSAConfig("128k", B=1, N=131072, H_q=32, H_kv=8, d=128, d_idx=64, topk=16,
                      n_needle=16, seed=1003, needle_seed=2003),
    "1m": MSAConfig("1m", B=1, N=1048576, H_q=16, H_kv=2, d=128, d_idx=64, topk=16,
                    n_needle=32, seed=1004, needle_seed=2004),
}


def shapes(cfg: MSAConfig) -> dict:
    """Tensor shapes (row-major, contiguous) of every input."""
    B, N = cfg.B, cfg.N
    return {
        "q": (B, N, cfg.H_q, cfg.d),
        "k": (B, N, cfg.H_kv, cfg.d),
        "v": (B, N, cfg.H_kv, cfg.d),
        "q_idx": (B, N, cfg.H_kv, cfg.d_idx),
        "k_idx": (B, N, cfg.d_idx),
        "dO": (B, N, cfg.H_q, cfg.d),
    }


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def needles(cfg: MSAConfig):
    """Needle blocks per group and the per-group unit directions (u_g, v_g)."""
    if cfg.n_needle == 0:
        return None
    rng = np.random.Generator(np.random.PCG64(cfg.needle_seed))
    lo, hi = 1, max(2, cfg.nb // 2)
    pool = np.arange(lo, hi)
    blocks = rng.choice(pool, size=cfg.H_kv * cfg.n_needle, replace=False)
    blocks = blocks.reshape(cfg.H_kv, cfg.n_needle)
    u = rng.standard_normal((cfg.H_kv, cfg.d_idx))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    vdir = rng.standard_normal((cfg.H_kv, cfg.d))
    vdir /= np.linalg.norm(vdir, axis=1, keepdims=True)
    block_group = np.full(cfg.nb, -1, dtype=np.int64)
    for g in range(cfg.H_kv):
        block_group[blocks[g]] = g
    return {"blocks": blocks, "u": u.astype(np.float32), "v": vdir.astype(np.float32),
            "block_group": block_group}


def _fill(name: str, cfg: MSAConfig, out: np.ndarray, ndl, chunk_rows: int, c: int):
    shape = out.shape
    row = int(np.prod(shape[2:]))  # elements per token
    n_tok = shape[0] * shape[1]
    t0 = c * chunk_rows
    t1 = min(n_tok, t0 + chunk_rows)
    ss = np.random.SeedSequence(cfg.seed, spawn_key=(_TENSOR_IDS[name], c))
    rng = np.random.Generator(np.random.PCG64(ss))
    x = rng.standard_normal((t1 - t0) * row, dtype=np.float32).reshape((t1 - t0,) + shape[2:])
    if ndl is not None:
        pos = np.arange(t0, t1) % cfg.N
        grp = ndl["block_group"][pos // cfg.Bk]
        if name == "q_idx":
            x += np.float32(0.5) * ndl["u"][None, :, :]
        elif name == "k_idx":
            hit = grp >= 0
            x[hit] += np.float32(2.0) * ndl["u"][grp[hit]]
        elif name == "k":
            hit = np.nonzero(grp >= 0)[0]
            x[hit, grp[hit], :] += np.float32(2.0) * ndl["v"][grp[hit]]
    out.reshape(n_tok, row)[t0:t1] = f32_to_bf16_bits(x.reshape(t1 - t0, row))


def make_inputs(cfg: MSAConfig, names=("q", "k", "v", "q_idx", "k_idx", "dO"),
                threads: int | None = None) -> dict:
    """Seeded bf16 inputs (uint16 bit arrays) for one workload."""
    ndl = needles(cfg)
    sh = shapes(cfg)
    res = {}
    threads = threads or min(32, os.cpu_count() or 1)
    with ThreadPoolExecutor(threads) as ex:
        futs = []
        for name in names:
            out = np.empty(sh[name], dtype=np.uint16)
            res[name] = out
            row = int(np.prod(sh[name][2:]))
            chunk_rows = max(1, _CHUNK_ELEMS // row)
            n_tok = sh[name][0] * sh[name][1]
            for c in range((n_tok + chunk_rows - 1) // chunk_rows):
                futs.append(ex.submit(_fill, name, cfg, out, ndl, chunk_rows, c))
        for f in futs:
            f.result()
    return res


def sample_rows(cfg: MSAConfig, n: int, seed: int) -> np.ndarray:
    """Seeded query-row subsample, as sorted flat ids b*N + i. Always includes the
    first and last row of every batch so the extremes of the causal range are seen."""
    rng = np.random.Generator(np.random.PCG64(seed))
    total = cfg.B * cfg.N
    n = min(n, total)
    picks = set(rng.choice(total, size=n, replace=False).tolist())
    for b in range(cfg.B):
        picks.add(b * cfg.N)
        picks.add(b * cfg.N + cfg.N - 1)
    return np.array(sorted(picks), dtype=np.int64)


def varlen_offsets(n: int, lo: int, hi: int, seed: int) -> list:
    """cu_seqlens of a packed batch of n sequences whose lengths are drawn uniformly from
    lo .. hi (inclusive, seeded): [0, L_0, L_0 + L_1, ...]."""
    lens = np.random.default_rng(seed).integers(lo, hi + 1, size=n)
    return [0] + np.cumsum(lens).astype(int).tolist()


def varlen_offsets_total(n: int, total: int, lo: int, hi: int, seed: int) -> list:
    """cu_seqlens of n sequences that fill exactly `total` tokens: seeded lengths drawn
    log-uniformly from lo .. hi, scaled to the total and rounded, the rounding remainder
    given to the last sequence."""
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))
    lens = np.maximum(1, np.floor(raw * total / raw.sum())).astype(np.int64)
    lens[-1] += total - int(lens.sum())
    return [0] + np.cumsum(lens).astype(int).tolist()
