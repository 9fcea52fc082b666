"""FP8 (E4M3) KV cache for decode: the quantiser and the decode attention over the
dequantised cache, in plain numpy.

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
