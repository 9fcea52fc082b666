"""Dense, brute-force float64 restatement of the MSA hot path, for pinning the oracle.

Written independently of oracle/msa_oracle.c and in a different shape: whole score
matrices, an explicit argsort for the block ranking, a dense token mask and masked
dense softmax.  Only used on tiny inputs.  Definitions follow the MiniMax Sparse
Attention summary (7minutos.es), "Cómo funcionan las dos ramas" and "Cómo se
entrena MSA".
"""
from __future__ import annotations

import numpy as np


def decode(x_bits):
    return (np.asarray(x_bits).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def as_f64(inputs):
    return {k: decode(v) for k, v in inputs.items()}


def select_dense(cfg, qi, ki, causal=None):
    """Selection by explicit sort.  qi [B,N,H_kv,d_idx], ki [B,N,d_idx] (float64).
    Returns sel [B,H_kv,N,topk] (ascending, -1 padded), pooled [B,H_kv,N,nb]
    (nan where not a candidate)."""
    causal = cfg.causal if causal is None else causal
    B, N, H_kv, _ = qi.shape
    Bk, k = cfg.Bk, cfg.topk
    nb = -(-N // Bk)
    sel = np.full((B, H_kv, N, k), -1, dtype=np.int64)
    pooled = np.full((B, H_kv, N, nb), np.nan)
    blk = np.arange(N) // Bk
    for b in range(B):
        for g in range(H_kv):
            Z = qi[b, :, g, :] @ ki[b].T  # [N, N] raw index logits
            Zp = np.full((N, nb * Bk), -np.inf)
            Zp[:, :N] = Z
            P = Zp.reshape(N, nb, Bk).max(axis=2)  # block max-pool
            for i in range(N):
                ci = blk[i]
                cand = np.array([c for c in range(nb) if c != ci and (c < ci or not causal)],
                                dtype=np.int64)
                pooled[b, g, i, cand] = P[i, cand]
                # rank: score descending, then block id ascending
                order = cand[np.lexsort((cand, -P[i, cand]))] if len(cand) else cand
                chosen = sorted([ci] + list(order[: k - 1]))
                sel[b, g, i, : len(chosen)] = chosen
    return sel, pooled


def token_mask(cfg, sel, causal=None):
    """mask [B,H_kv,N,N]: query i of group g sees key j."""
    causal = cfg.causal if causal is None else causal
    B, H_kv, N, k = sel.shape
    blk = np.arange(N) // cfg.Bk
    M = np.zeros((B, H_kv, N, N), dtype=bool)
    for b in range(B):
        for g in range(H_kv):
            for i in range(N):
                chosen = set(int(c) for c in sel[b, g, i] if c >= 0)
                M[b, g, i] = np.isin(blk, list(chosen))
    if causal:
        M &= np.tril(np.ones((N, N), dtype=bool))[None, None]
    return M


def _masked_softmax(S, M):
    S = np.where(M, S, -np.inf)
    m = S.max(axis=-1, keepdims=True)
    E = np.where(M, np.exp(S - m), 0.0)
    l = E.sum(axis=-1, keepdims=True)
    return E / l, (m + np.log(l))[..., 0]


def dense_forward(cfg, x, M, scale, scale_idx):
    """x: float64 q,k,v,q_idx,k_idx.  Returns dict of O [B,N,H_q,d], lse [B,N,H_q],
    P [B,H_q,N,N], lse_idx [B,N,H_kv], pI [B,H_kv,N,N], pT [B,H_kv,N,N]."""
    q, k, v, qi, ki = x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"]
    B, N, H_q, d = q.shape
    H_kv = k.shape[2]
    G = H_q // H_kv
    O = np.zeros_like(q)
    lse = np.zeros((B, N, H_q))
    P = np.zeros((B, H_q, N, N))
    lse_idx = np.zeros((B, N, H_kv))
    pI = np.zeros((B, H_kv, N, N))
    pT = np.zeros((B, H_kv, N, N))
    for b in range(B):
        for h in range(H_q):
            g = h // G
            S = scale * (q[b, :, h, :] @ k[b, :, g, :].T)
            Ph, l = _masked_softmax(S, M[b, g])
            P[b, h] = Ph
            lse[b, :, h] = l
            O[b, :, h, :] = Ph @ v[b, :, g, :]
        for g in range(H_kv):
            Zs = scale_idx * (qi[b, :, g, :] @ ki[b].T)
            pI[b, g], lse_idx[b, :, g] = _masked_softmax(Zs, M[b, g])
            pT[b, g] = P[b, g * G:(g + 1) * G].mean(axis=0)
    return {"O": O, "lse": lse, "P": P, "lse_idx": lse_idx, "pI": pI, "pT": pT}


def kl_value(pT, pI, M, w):
    """w * sum over rows of KL(p_T || p_I) over the token set."""
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(M & (pT > 0), pT * (np.log(pT) - np.log(pI)), 0.0)
    return w * t.sum()


def loss_main(cfg, x, M, dO, scale, scale_idx):
    """sum(dO * O): its gradient in q, k, v is the main-branch backward."""
    return float((dense_forward(cfg, x, M, scale, scale_idx)["O"] * dO).sum())


def loss_kl_fixed_teacher(cfg, x, M, pT, w, scale_idx):
    """KL with the teacher held fixed (detached): its gradient in q_idx, k_idx."""
    qi, ki = x["q_idx"], x["k_idx"]
    B, N, H_kv, _ = qi.shape
    tot = 0.0
    for b in range(B):
        for g in range(H_kv):
            Zs = scale_idx * (qi[b, :, g, :] @ ki[b].T)
            pI, _ = _masked_softmax(Zs, M[b, g])
            tot += kl_value(pT[b, g], pI, M[b, g], 1.0)
    return w * tot
