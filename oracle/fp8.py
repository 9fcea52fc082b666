"""FP8 (E4M3): the KV-cache quantiser and the decode attention over the dequantised
cache, and the FP8 main-branch forward for training (per-block k/v scales, P rounded
to E4M3), in plain numpy.

TEST INFRASTRUCTURE ONLY, like the rest of oracle/: imported by the tests and never by
the library under block_sparse_gqa_topk_gb300/.

The pages name FP8 only as one of the precisions the MSA attention kernels support
(Flash-MSA / fmha_sm100 paragraph of the MSA summary, 7minutos.es, "El codiseño del
kernel"); they give no quantisation recipe.  Reading taken here (the plainest one for
a KV cache):
  * format: OCP 8-bit floating point E4M3 -- 1 sign bit, 4 exponent bits (bias 7),
    3 mantissa bits; exponent 0 holds the subnormals m/8 * 2^-6; no infinities; the
    all-ones pattern S.1111.111 is NaN; largest finite magnitude 1.75 * 2^8 = 448;
  * one float32 scale per (sequence, token, KV head) row of d values:
    s = float32(amax |x| / 448), or 1 when the row is all zero;
  * code = E4M3 value nearest to float32(x / s) (ties to the even code), magnitudes
    above 448 saturate to 448, the sign is kept (a negative value that rounds to zero
    gives the code 0x80);
  * the cache value seen by attention is decode(code) * s.
The quantisation is a per-row encoding, so the GPU must reproduce the codes bit for
bit; both sides divide in float32 with IEEE rounding.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """float64 value of every E4M3 code (uint8 array), from the format's fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the 127 non-negative finite values, increasing with the code 0x00 .. 0x7E
_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each float32 value (ties to the even code), saturating at
    +-448; NaN gives 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, len(_POS) - 1)  # _POS[hi] >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS[lo]
    d_hi = _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_rows(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """x [..., d] as bf16 bit patterns (uint16) -> (codes uint8 [..., d], scale float32
    [...]) with one scale per row of d values."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    s = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32), np.float32(1.0))
    s = s.astype(np.float32)
    q = (x / s[..., None]).astype(np.float32)
    return e4m3_encode(q), s


def dequantize_rows(codes, scale) -> np.ndarray:
    """decode(code) * s in float64."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]


def decode_attention(q_bits, k_deq, v_deq, block_idx, lens, scale, Bk=128):
    """Exact softmax attention of the new token of every sequence over the causally
    visible tokens (j < lens[b]) of its group's selected blocks, on float64 caches.

    q_bits [B,H_q,d] bf16 bits; k_deq, v_deq [B,Lmax,H_kv,d] float64; block_idx
    [B,H_kv,topk] (-1 padded); lens [B].  Returns (o [B,H_q,d], lse [B,H_q])."""
    q = (np.asarray(q_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    q = q.astype(np.float64)
    B, H_q, d = q.shape
    H_kv = k_deq.shape[2]
    G = H_q // H_kv
    o = np.zeros((B, H_q, d))
    lse = np.zeros((B, H_q))
    for b in range(B):
        L = int(lens[b])
        for g in range(H_kv):
            toks = [j for c in block_idx[b, g] if c >= 0
                    for j in range(c * Bk, min((c + 1) * Bk, L))]
            K = k_deq[b, toks, g]          # [T, d]
            V = v_deq[b, toks, g]
            for h in range(g * G, (g + 1) * G):
                s = scale * (K @ q[b, h])
                m = s.max()
                e = np.exp(s - m)
                lse[b, h] = m + np.log(e.sum())
                o[b, h] = (e / e.sum()) @ V
    return o, lse


# ---------------------------------------------------------------------------
# FP8 main-branch forward for training
# ---------------------------------------------------------------------------
# Reading (the pages name FP8 among the precisions of the MSA attention kernels,
# "El codiseño del kernel", and give no recipe): q keeps one scale per (token, head)
# row (quantize_rows); k and v take one scale per (batch, head, Bk-token block) over
# the block's real tokens and all d values (quantize_blocks).  The forward is split by
# selected key block, as the KV-outer design computes it: within block c the scores
# s_j = scale * s_q * s_k(c) * (q8 . k8_j) are softmaxed against the block's own max
# m_c, P_j = exp(s_j - m_c) is rounded to E4M3 for the P V product while the row sum
# l_c uses the unrounded P, o_c = s_v(c) * sum_j E4M3(P_j) v8_j / l_c and
# lse_c = m_c + log l_c; the blocks are merged by their lse.

def quantize_blocks(x_bits, Bk: int = 128) -> tuple[np.ndarray, np.ndarray]:
    """x [B, N, H, d] as bf16 bit patterns -> (codes uint8 [B, N, H, d], scale float32
    [B, H, nb]) with one scale per (batch, head, Bk-token block) over the block's tokens
    and all d values (1 for an all-zero block); each value is coded as in
    quantize_rows."""
    x = (np.asarray(x_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    B, N, H, d = x.shape
    nb = (N + Bk - 1) // Bk
    codes = np.empty(x.shape, dtype=np.uint8)
    scale = np.empty((B, H, nb), dtype=np.float32)
    for c in range(nb):
        blk = x[:, c * Bk:(c + 1) * Bk]                      # [B, n, H, d]
        amax = np.max(np.abs(blk), axis=(1, 3))              # [B, H]
        s = np.where(amax > 0, (amax / np.float32(E4M3_MAX)).astype(np.float32),
                     np.float32(1.0)).astype(np.float32)
        scale[:, :, c] = s
        codes[:, c * Bk:(c + 1) * Bk] = e4m3_encode((blk / s[:, None, :, None]).astype(np.float32))
    return codes, scale


def attend_block_e4m3(s, v):
    """One key block's share: scores s [T] (float64), values v [T, d] (float64).
    P = exp(s - max s), rounded to E4M3 (from float32) for the product with v, summed
    unrounded.  Returns (o_c = sum E4M3(P) v / sum P, lse_c = max s + log sum P)."""
    s = np.asarray(s, dtype=np.float64)
    m = s.max()
    p = np.exp(s - m)
    p8 = e4m3_decode(e4m3_encode(p.astype(np.float32)))
    l = p.sum()
    return (p8 @ v) / l, m + np.log(l)


def forward_fp8(inputs, block_idx_rows, rows, scale: float, G: int, Bk: int = 128):
    """FP8 forward of the listed flat rows (b * N + i) over their block sets
    block_idx_rows [R, H_kv, topk] (ascending, -1 padded), causal.  inputs: bf16 bit
    arrays q [B,N,H_q,d], k, v [B,N,H_kv,d].  Returns (o [R, H_q, d], lse [R, H_q]).
    Only the rows' q and the blocks they select are quantised (each quantisation is
    local to its row or block)."""
    q_bits, k_bits, v_bits = inputs["q"], inputs["k"], inputs["v"]
    B, N, H_q, d = q_bits.shape
    H_kv = k_bits.shape[2]
    blocks_seen = {}

    def block(b, g, c):
        """Decoded k and v codes of block c of (b, g) and their two scales."""
        key = (b, g, c)
        if key not in blocks_seen:
            sl = slice(c * Bk, min(N, (c + 1) * Bk))
            kc, ks = quantize_blocks(k_bits[b:b + 1, sl, g:g + 1], Bk)
            vc, vs = quantize_blocks(v_bits[b:b + 1, sl, g:g + 1], Bk)
            blocks_seen[key] = (e4m3_decode(kc[0, :, 0]), float(ks[0, 0, 0]),
                                e4m3_decode(vc[0, :, 0]), float(vs[0, 0, 0]))
        return blocks_seen[key]

    R = len(rows)
    o = np.zeros((R, H_q, d))
    lse = np.zeros((R, H_q))
    for r, row in enumerate(np.asarray(rows, dtype=np.int64)):
        b, i = int(row // N), int(row % N)
        qc, qs = quantize_rows(q_bits[b, i])      # [H_q, d], [H_q]
        qd = e4m3_decode(qc)
        for g in range(H_kv):
            blocks = [int(c) for c in block_idx_rows[r, g] if c >= 0]
            for h in range(g * G, (g + 1) * G):
                parts, lses = [], []
                for c in blocks:
                    n = min(Bk, N - c * Bk, i + 1 - c * Bk)   # causally visible keys of block c
                    if n <= 0:
                        continue
                    kd, ks, vd, vs = block(b, g, c)
                    s = scale * float(qs[h]) * ks * (kd[:n] @ qd[h])
                    oc, lc = attend_block_e4m3(s, vs * vd[:n])
                    parts.append(oc)
                    lses.append(lc)
                lt = np.array(lses)
                mx = lt.max()
                tot = mx + np.log(np.exp(lt - mx).sum())
                w = np.exp(lt - tot)
                o[r, h] = (w[:, None] * np.array(parts)).sum(axis=0)
                lse[r, h] = tot
    return o, lse
