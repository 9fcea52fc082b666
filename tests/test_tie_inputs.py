"""The tie inputs of the GPU selection test hold what that test relies on.

Key blocks that are copies of block 0 scaled by 1, 2 or 4 pool, in the oracle's float64,
to exactly that multiple of a query's block-0 score, and many rows have more candidate
blocks tied at the top score than the k - 1 free slots.  There the set is decided by the
tie rule alone.  The pages take the top k of the pooled scores (MSA summary, 7minutos.es,
"Cómo funcionan las dos ramas" ¶2) and say nothing of ties; the oracle and the kernels
rank equal scores lower block first, so the lowest tied blocks are the ones taken.
"""
import numpy as np

import oracle
from block_sparse_gqa_topk_gb300 import synth
from gpu_inputs import tie_inputs

CFG = synth.CONFIGS["tiny"].with_(name="ties", N=4096, topk=6, seed=45)


def test_tie_inputs_pool_to_exact_multiples_and_ties_decide_the_set():
    h, scale = tie_inputs(CFG)
    rows = np.arange(CFG.N, dtype=np.int64)  # batch 0, every query
    bi, _, pl = oracle.select(CFG, h, rows=rows, pooled=True)
    nb = CFG.N // CFG.Bk
    qb = rows // CFG.Bk
    for c in range(1, nb):
        vis = qb > c  # block c is a candidate of these rows (earlier blocks only)
        assert np.array_equal(pl[vis, :, c] * scale[0], pl[vis, :, 0] * scale[c]), c
    decided = 0
    for r in range(CFG.N):
        if qb[r] < 2:
            continue
        for g in range(CFG.H_kv):
            cand = pl[r, g, :qb[r]]
            top = np.flatnonzero(cand == cand.max())
            if len(top) > CFG.topk - 1:
                decided += 1
                want = sorted(top[:CFG.topk - 1].tolist() + [int(qb[r])])
                assert bi[r, g].tolist() == want, (r, g)
    assert decided >= 1000, decided
