"""Shared helpers of the GPU parity tests: seeded inputs on the device, the
selection rule for near ties, and the tolerances the tests enforce.

Tolerances (bf16 I/O, fp32 accumulation): o max-abs 2e-2; lse and lse_idx abs
1e-3; each gradient cosine >= 0.999 and max-abs <= 5e-2 * max|ref|; KL rel 1e-3
(+1e-6 abs).  Block sets must equal the oracle's wherever the oracle's
(k-1)-th and k-th best non-local pooled scores differ by more than 1e-3
relative; inside that band the GPU's set must be a valid top-k of the oracle's
pooled scores within the band.
"""
import numpy as np
import torch

import oracle
from block_sparse_gqa_topk_gb300 import synth

O_TOL = 2e-2
LSE_TOL = 1e-3
GRAD_COS = 0.999
GRAD_REL = 5e-2
KL_REL = 1e-3
GAP_REL = 1e-3


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t_or_bits) -> np.ndarray:
    if isinstance(t_or_bits, torch.Tensor):
        if t_or_bits.dtype == torch.bfloat16:
            return t_or_bits.float().cpu().numpy().astype(np.float64)
        return t_or_bits.cpu().numpy().astype(np.float64)
    return synth.bf16_bits_to_f32(t_or_bits).astype(np.float64)


def gpu_sel_rows(cfg, bi_gpu: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """[B,H_kv,N,k] -> [R,H_kv,k] for flat rows b*N+i."""
    b = rows // cfg.N
    i = rows % cfg.N
    return bi_gpu[b, :, i, :]


def check_selection(cfg, inputs, bi_gpu_rows, rows, bi_ref, kth):
    """Applies the near-tie rule; returns (n_exact_rows, n_band_rows, mismatch_mask)."""
    R, H, k = bi_ref.shape
    s1, s2 = kth[..., 0], kth[..., 1]
    with np.errstate(invalid="ignore"):
        band = GAP_REL * np.maximum(np.abs(np.where(np.isfinite(s1), s1, 0)),
                                    np.abs(np.where(np.isfinite(s2), s2, 0)))
        near = np.isfinite(s1) & np.isfinite(s2) & ((s1 - s2) <= band)
    same = np.all(bi_gpu_rows == bi_ref, axis=-1)
    bad = ~same & ~near
    assert not bad.any(), (
        f"{int(bad.sum())} rows differ outside the near-tie band, e.g. row "
        f"{rows[np.argwhere(bad)[0][0]]}: gpu {bi_gpu_rows[bad][0]} oracle {bi_ref[bad][0]}")
    diff = ~same & near
    if diff.any():
        idx = np.argwhere(diff)
        r_sub = np.unique(rows[idx[:, 0]])
        _, _, pooled = oracle.select(cfg, inputs, rows=r_sub, pooled=True)
        pos = {int(r): n for n, r in enumerate(r_sub)}
        for r, g in idx:
            i = int(rows[r] % cfg.N)
            ci = i // cfg.Bk
            gs = bi_gpu_rows[r, g]
            valid = gs[gs >= 0]
            assert ci in valid and len(valid) == min(k, ci + 1)
            assert np.all(np.diff(valid) > 0) and np.all(gs[len(valid):] == -1)
            pl = pooled[pos[int(rows[r])], g]
            for c in valid:
                if c != ci:
                    assert pl[c] >= s1[r, g] - band[r, g], (r, g, c, pl[c], s1[r, g])
    return int(same.sum()), int(near.sum()), diff


def validated_gpu_sets(cfg, inputs, bi_gpu_rows, rows):
    """The GPU's block sets of the listed rows, after the near-tie rule has accepted
    them: the oracle then reruns on exactly these sets, so a row where the GPU took
    another valid set inside the band is compared against the oracle's output for
    that set instead of being skipped.  Returns (sets [R,H_kv,k], n_differing)."""
    bi_ref, kth, _ = oracle.select(cfg, inputs, rows=rows)
    _, _, diff = check_selection(cfg, inputs, bi_gpu_rows, np.asarray(rows), bi_ref, kth)
    return np.ascontiguousarray(bi_gpu_rows, dtype=np.int32), int(diff.sum())


def grad_close(got: np.ndarray, ref: np.ndarray, name: str):
    g = got.ravel().astype(np.float64)
    r = ref.ravel().astype(np.float64)
    nr = np.linalg.norm(r)
    cos = float(g @ r / (np.linalg.norm(g) * nr)) if nr > 0 else 1.0
    mx = float(np.abs(g - r).max()) if g.size else 0.0
    ref_max = float(np.abs(r).max()) if r.size else 0.0
    assert cos >= GRAD_COS, f"{name}: cosine {cos:.6f} < {GRAD_COS}"
    assert mx <= GRAD_REL * ref_max + 1e-30, f"{name}: max-abs {mx:.3e} > {GRAD_REL} * {ref_max:.3e}"
    return cos, mx / max(ref_max, 1e-30)
