"""Pins of the float64 oracle against things other than itself (CPU only).

 - an independent dense brute force (explicit argsort, dense masks, masked softmax);
 - the exp-free top-k invariant: ranking raw pooled scores = ranking softmax-pooled
   probabilities (MSA summary, 7minutos.es, "El codiseño del kernel" ¶2);
 - the forced local block and the k-block budget (same page, "Cómo funcionan las dos
   ramas" ¶2; "¿Qué es MSA?" ¶2);
 - k >= visible blocks reduces to dense causal GQA attention, checked against
   torch's scaled_dot_product_attention in float64;
 - KL = 0 and zero index gradients when the index branch equals the main branch
   (closed form);
 - central finite differences of the dense forward for every gradient.
"""
import math

import numpy as np
import pytest
import torch

import bruteforce as bfm
import oracle
from block_sparse_gqa_topk_gb300 import synth

PIN = synth.MSAConfig("pin", B=2, N=200, H_q=4, H_kv=2, d=16, d_idx=8, Bk=32, topk=3,
                      seed=7, needle_seed=8)


def _w(cfg):
    return cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)


def _oracle_all(cfg, inp):
    bi, kth, pooled = oracle.select(cfg, inp, pooled=True)
    o, lse, lse_idx = oracle.forward(cfg, inp, bi)
    g = oracle.backward(cfg, inp, bi, _w(cfg))
    return bi, kth, pooled, o, lse, lse_idx, g


def _reshape_sel(cfg, bi):
    # oracle rows are b*N+i: [B*N, H_kv, k] -> [B, H_kv, N, k]
    return bi.reshape(cfg.B, cfg.N, cfg.H_kv, cfg.topk).transpose(0, 2, 1, 3)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n_needle", [0, 1])
def test_oracle_matches_dense_bruteforce(causal, n_needle):
    cfg = PIN.with_(causal=causal, n_needle=n_needle)
    inp = synth.make_inputs(cfg)
    x = bfm.as_f64(inp)
    bi, kth, pooled, o, lse, lse_idx, g = _oracle_all(cfg, inp)

    sel_ref, pooled_ref = bfm.select_dense(cfg, x["q_idx"], x["k_idx"])
    np.testing.assert_array_equal(_reshape_sel(cfg, bi), sel_ref)
    pr = pooled.reshape(cfg.B, cfg.N, cfg.H_kv, -1).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(pr, pooled_ref, rtol=1e-13, atol=1e-12, equal_nan=True)

    M = bfm.token_mask(cfg, sel_ref)
    ref = bfm.dense_forward(cfg, x, M, cfg.scale, cfg.scale_idx)
    np.testing.assert_allclose(o.reshape(ref["O"].shape), ref["O"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse.reshape(ref["lse"].shape), ref["lse"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse_idx.reshape(ref["lse_idx"].shape), ref["lse_idx"],
                               rtol=1e-12, atol=1e-12)
    kl_ref = sum(bfm.kl_value(ref["pT"][b, gg], ref["pI"][b, gg], M[b, gg], 1.0)
                 for b in range(cfg.B) for gg in range(cfg.H_kv)) * _w(cfg)
    assert g["kl"] == pytest.approx(kl_ref, rel=1e-10, abs=1e-14)
    assert g["kl"] > 0.0

    # gradients in dense matrix form (catches index / transpose mistakes in the loops)
    q, k, v, qi, ki = x["q"], x["k"], x["v"], x["q_idx"], x["k_idx"]
    dO = bfm.decode(inp["dO"])
    G = cfg.G
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dqi = np.zeros_like(qi)
    dki = np.zeros_like(ki)
    w = _w(cfg)
    for b in range(cfg.B):
        for h in range(cfg.H_q):
            gg = h // G
            P = ref["P"][b, h]
            dP = dO[b, :, h, :] @ v[b, :, gg, :].T
            Dv = (dO[b, :, h, :] * ref["O"][b, :, h, :]).sum(-1, keepdims=True)
            dS = P * (dP - Dv)
            dq[b, :, h, :] = cfg.scale * dS @ k[b, :, gg, :]
            dk[b, :, gg, :] += cfg.scale * dS.T @ q[b, :, h, :]
            dv[b, :, gg, :] += P.T @ dO[b, :, h, :]
        for gg in range(cfg.H_kv):
            dz = w * (ref["pI"][b, gg] - ref["pT"][b, gg])
            dqi[b, :, gg, :] = cfg.scale_idx * dz @ ki[b]
            dki[b] += cfg.scale_idx * dz.T @ qi[b, :, gg, :]
    np.testing.assert_allclose(g["dq"].reshape(dq.shape), dq, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(g["dk"], dk, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(g["dv"], dv, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(g["dq_idx"].reshape(dqi.shape), dqi, rtol=1e-9, atol=1e-14)
    np.testing.assert_allclose(g["dk_idx"], dki, rtol=1e-9, atol=1e-14)


def test_row_subsets_agree_with_full_run():
    cfg = PIN
    inp = synth.make_inputs(cfg)
    bi, kth, _ = oracle.select(cfg, inp)
    o, lse, li = oracle.forward(cfg, inp, bi)
    rows = np.array([0, 5, 63, 64, 199, 200, 333, 399], dtype=np.int64)
    bi_s, kth_s, _ = oracle.select(cfg, inp, rows=rows)
    np.testing.assert_array_equal(bi_s, bi[rows])
    np.testing.assert_array_equal(kth_s, kth[rows])
    o_s, lse_s, li_s = oracle.forward(cfg, inp, bi_s, rows=rows)
    np.testing.assert_array_equal(o_s, o[rows])
    np.testing.assert_array_equal(li_s, li[rows])
    # backward of a row subset == backward with dO zero and kl weight zero elsewhere
    # (main part), and its dq / dq_idx rows equal the full run's rows
    full = oracle.backward(cfg, inp, bi, 0.3)
    sub = oracle.backward(cfg, inp, bi_s, 0.3, rows=rows)
    np.testing.assert_allclose(sub["dq"], full["dq"][rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(sub["dq_idx"], full["dq_idx"][rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(sub["kl_rows"], full["kl_rows"][rows], rtol=1e-12)
    dO0 = inp["dO"].copy().reshape(cfg.B * cfg.N, -1)
    keep = np.zeros(cfg.B * cfg.N, dtype=bool)
    keep[rows] = True
    dO0[~keep] = 0
    inp0 = dict(inp, dO=dO0.reshape(inp["dO"].shape))
    masked = oracle.backward(cfg, inp0, bi, 0.0)
    sub0 = oracle.backward(cfg, inp, bi_s, 0.0, rows=rows)
    np.testing.assert_allclose(sub0["dk"], masked["dk"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(sub0["dv"], masked["dv"], rtol=1e-12, atol=1e-15)


def test_local_block_budget_and_kth():
    cfg = PIN.with_(N=256, topk=4)
    inp = synth.make_inputs(cfg)
    bi, kth, pooled = oracle.select(cfg, inp, pooled=True)
    nb = cfg.nb
    for r in range(cfg.B * cfg.N):
        i = r % cfg.N
        ci = i // cfg.Bk
        for g in range(cfg.H_kv):
            s = bi[r, g]
            valid = s[s >= 0]
            assert ci in valid  # the local block is always in the set
            assert len(valid) == min(cfg.topk, ci + 1)  # budget: min(k, visible)
            assert np.all(np.diff(valid) > 0) and np.all(s[len(valid):] == -1)
            cand = pooled[r, g][~np.isnan(pooled[r, g])]
            assert len(cand) == ci
            others = [c for c in valid if c != ci]
            if others:
                assert kth[r, g, 0] == min(pooled[r, g, c] for c in others)
            left = [pooled[r, g, c] for c in range(nb) if c < ci and c not in valid]
            assert kth[r, g, 1] == (max(left) if left else -np.inf)
            if left and others:
                assert kth[r, g, 0] >= kth[r, g, 1]


@pytest.mark.parametrize("scale_idx", [0.05, 1.0, 7.0])
def test_exp_free_topk_equals_softmax_then_topk(scale_idx):
    """Softmax preserves order, so ranking pooled softmax probabilities picks the
    same blocks as ranking raw pooled scores."""
    cfg = PIN.with_(N=256, topk=4, n_needle=1)
    inp = synth.make_inputs(cfg)
    x = bfm.as_f64(inp)
    bi, _, _ = oracle.select(cfg, inp)
    sel = _reshape_sel(cfg, bi)
    N, Bk = cfg.N, cfg.Bk
    for b in range(cfg.B):
        for g in range(cfg.H_kv):
            Z = scale_idx * (x["q_idx"][b, :, g, :] @ x["k_idx"][b].T)
            for i in range(Bk, N, 7):
                ci = i // Bk
                vis = Z[i, : ci * Bk]
                p = np.exp(vis - vis.max())
                p /= p.sum()
                pb = p.reshape(ci, Bk).max(axis=1)
                order = np.lexsort((np.arange(ci), -pb))
                want = sorted([ci] + list(order[: cfg.topk - 1]))
                got = [c for c in sel[b, g, i] if c >= 0]
                assert got == want


def test_group_sharing_and_independence():
    """Every head of a group uses the group's set; another group's index query does
    not change this group's outputs."""
    cfg = PIN
    inp = synth.make_inputs(cfg)
    bi, _, _ = oracle.select(cfg, inp)
    o, lse, li = oracle.forward(cfg, inp, bi)
    inp2 = dict(inp)
    qi = inp["q_idx"].copy()
    rng = np.random.default_rng(0)
    qi[:, :, 1, :] = synth.f32_to_bf16_bits(rng.standard_normal(qi[:, :, 1, :].shape).astype(np.float32))
    inp2["q_idx"] = qi
    bi2, _, _ = oracle.select(cfg, inp2)
    np.testing.assert_array_equal(bi2[:, 0], bi[:, 0])
    assert not np.array_equal(bi2[:, 1], bi[:, 1])
    o2, lse2, _ = oracle.forward(cfg, inp2, bi2)
    G = cfg.G
    np.testing.assert_array_equal(o2[:, :G], o[:, :G])
    np.testing.assert_array_equal(lse2[:, :G], lse[:, :G])


@pytest.mark.parametrize("G", [1, 2, 4])
def test_dense_special_case_matches_sdpa(G):
    """k >= number of blocks: every visible block is selected and the main branch is
    dense causal GQA attention (torch SDPA, float64, CPU)."""
    cfg = synth.MSAConfig("dense", B=2, N=160, H_q=2 * G, H_kv=2, d=16, d_idx=8, Bk=32,
                          topk=5, seed=11)
    inp = synth.make_inputs(cfg)
    bi, _, _ = oracle.select(cfg, inp)
    for r in range(cfg.B * cfg.N):
        ci = (r % cfg.N) // cfg.Bk
        for g in range(cfg.H_kv):
            assert list(bi[r, g][: ci + 1]) == list(range(ci + 1))
    o, _, _ = oracle.forward(cfg, inp, bi)
    x = bfm.as_f64(inp)
    q = torch.from_numpy(x["q"]).permute(0, 2, 1, 3)
    k = torch.from_numpy(x["k"]).permute(0, 2, 1, 3)
    v = torch.from_numpy(x["v"]).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=cfg.scale, enable_gqa=True)
    ref = ref.permute(0, 2, 1, 3).numpy().reshape(o.shape)
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_kl_zero_when_index_equals_main():
    """G = 1, q_idx = q, k_idx = k, scale_idx = scale: p_I == p_T, so KL = 0 and the
    index gradients vanish (closed form)."""
    cfg = synth.MSAConfig("klzero", B=1, N=192, H_q=1, H_kv=1, d=16, d_idx=16, Bk=32, topk=3,
                          seed=5)
    inp = synth.make_inputs(cfg)
    inp["q_idx"] = inp["q"].copy()
    inp["k_idx"] = inp["k"].reshape(cfg.B, cfg.N, cfg.d).copy()
    bi, _, _ = oracle.select(cfg, inp)
    g = oracle.backward(cfg, inp, bi, 1.0, scale_idx=cfg.scale)
    assert abs(g["kl"]) < 1e-12
    assert np.abs(g["dq_idx"]).max() < 1e-12
    assert np.abs(g["dk_idx"]).max() < 1e-12
    # and with a different index scale the KL is strictly positive
    g2 = oracle.backward(cfg, inp, bi, 1.0, scale_idx=2 * cfg.scale)
    assert g2["kl"] > 1e-6 and np.all(g2["kl_rows"] >= -1e-15)


def _fd_check(f, x, name, analytic, coords, eps=1e-6, tol=1e-6):
    for idx in coords:
        old = x[name][idx]
        x[name][idx] = old + eps
        fp = f(x)
        x[name][idx] = old - eps
        fm = f(x)
        x[name][idx] = old
        fd = (fp - fm) / (2 * eps)
        an = analytic[idx]
        assert abs(fd - an) <= tol * max(1.0, abs(an)), (name, idx, fd, an)


@pytest.mark.parametrize("causal", [True, False])
def test_gradients_match_finite_differences(causal):
    cfg = synth.MSAConfig("fd", B=1, N=96, H_q=4, H_kv=2, d=8, d_idx=4, Bk=16, topk=3,
                          causal=causal, seed=21)
    inp = synth.make_inputs(cfg)
    bi, kth, _ = oracle.select(cfg, inp)
    x = bfm.as_f64(inp)
    dO = bfm.decode(inp["dO"])
    w = 0.37
    g = oracle.backward(cfg, inp, bi, w)
    sel = _reshape_sel(cfg, bi)
    M = bfm.token_mask(cfg, sel)
    rng = np.random.default_rng(3)

    def coords(shape, n=25):
        return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]

    def fmain(xx):
        return bfm.loss_main(cfg, xx, M, dO, cfg.scale, cfg.scale_idx)

    for name, an in (("q", g["dq"].reshape(x["q"].shape)), ("k", g["dk"]), ("v", g["dv"])):
        _fd_check(fmain, x, name, an, coords(x[name].shape))

    pT = bfm.dense_forward(cfg, x, M, cfg.scale, cfg.scale_idx)["pT"]

    def fkl(xx):
        return bfm.loss_kl_fixed_teacher(cfg, xx, M, pT, w, cfg.scale_idx)

    for name, an in (("q_idx", g["dq_idx"].reshape(x["q_idx"].shape)), ("k_idx", g["dk_idx"])):
        _fd_check(fkl, x, name, an, coords(x[name].shape), tol=1e-7)
    assert g["kl"] == pytest.approx(fkl(x), rel=1e-10)
