"""Multi-process checks of the N > 1 pieces, on CPU with the gloo backend (world size 2).

1. bench.job_rate: each rank gets the slowest rank's time and the whole-job rate
   (units of all ranks / max time), as the benchmark's torchrun mode reports it.
2. Group sharding.  Every GQA group's selection, forward and main backward are
   independent; the groups share only k_idx, whose gradient sums over groups
   (MSA summary, 7minutos.es, "Cómo funcionan las dos ramas" ¶1: one shared
   index-key head).  So a run split by group across ranks needs one exchange: an
   all-reduce (sum) of dk_idx and of the KL.  Here rank r runs the oracle on group r
   alone, the ranks all-reduce dk_idx and KL over gloo, and the result must equal
   the unsharded oracle run; every other output must equal its group's slice.
"""
import os
import socket

import numpy as np
import pytest

SHARD = dict(name="shard", B=1, N=384, H_q=8, H_kv=2, d=32, d_idx=16, Bk=64, topk=3,
             n_needle=0, seed=31, needle_seed=32)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, job, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, job(rank, world)))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, RuntimeError(repr(e))))
    finally:
        dist.destroy_process_group()


def _run(job, world=2, timeout=180):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, job, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(world):
            r, v = q.get(timeout=timeout)
            out[r] = v
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    for r, v in out.items():
        if isinstance(v, Exception):
            raise v
    return out


# ---------------------------------------------------------------- job_rate
def _rate_job(rank, world):
    import bench
    return bench.job_rate(10.0 + 5.0 * rank, 1000, world)


def test_job_rate_takes_the_slowest_rank():
    out = _run(_rate_job)
    for r in (0, 1):
        ms, v = out[r]
        assert ms == 15.0
        assert v == pytest.approx(2 * 1000 / 0.015)


# ---------------------------------------------------------------- group sharding
def _group_slice(inputs, cfg, g):
    G = cfg.H_q // cfg.H_kv
    return {
        "q": np.ascontiguousarray(inputs["q"][:, :, g * G:(g + 1) * G]),
        "dO": np.ascontiguousarray(inputs["dO"][:, :, g * G:(g + 1) * G]),
        "k": np.ascontiguousarray(inputs["k"][:, :, g:g + 1]),
        "v": np.ascontiguousarray(inputs["v"][:, :, g:g + 1]),
        "q_idx": np.ascontiguousarray(inputs["q_idx"][:, :, g:g + 1]),
        "k_idx": inputs["k_idx"],
    }


def _shard_job(rank, world):
    import torch
    import torch.distributed as dist
    import oracle
    from block_sparse_gqa_topk_gb300 import synth
    cfg = synth.MSAConfig(**SHARD)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    inputs = synth.make_inputs(cfg)
    scfg = cfg.with_(H_q=cfg.G, H_kv=1)  # this rank's group alone
    sl = _group_slice(inputs, cfg, rank)
    bi, _, _ = oracle.select(scfg, sl)
    g = oracle.backward(scfg, sl, bi, w)
    dki = torch.from_numpy(np.ascontiguousarray(g["dk_idx"]))
    kl = torch.tensor([g["kl"]], dtype=torch.float64)
    dist.all_reduce(dki)  # the one exchange step
    dist.all_reduce(kl)
    return {"bi": bi, "dq": g["dq"], "dk": g["dk"], "dv": g["dv"], "dq_idx": g["dq_idx"],
            "dk_idx": dki.numpy(), "kl": float(kl.item()), "kl_local": g["kl"]}


def test_group_sharded_oracle_with_dk_idx_allreduce_matches_unsharded():
    import oracle
    from block_sparse_gqa_topk_gb300 import synth
    oracle.build()
    cfg = synth.MSAConfig(**SHARD)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    inputs = synth.make_inputs(cfg)
    bi, _, _ = oracle.select(cfg, inputs)
    full = oracle.backward(cfg, inputs, bi, w)
    out = _run(_shard_job)
    G = cfg.G
    for r in range(cfg.H_kv):
        s = out[r]
        np.testing.assert_array_equal(s["bi"][:, 0], bi[:, r])
        np.testing.assert_allclose(s["dq"], full["dq"][:, r * G:(r + 1) * G], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dk"][:, :, 0], full["dk"][:, :, r], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dv"][:, :, 0], full["dv"][:, :, r], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dq_idx"][:, 0], full["dq_idx"][:, r], rtol=0, atol=1e-12)
        # after the all-reduce every rank holds the unsharded dk_idx and KL
        np.testing.assert_allclose(s["dk_idx"], full["dk_idx"], rtol=1e-12, atol=1e-15)
        assert s["kl"] == pytest.approx(full["kl"], rel=1e-12)
    # the exchange is needed: one group's share alone is not the answer
    assert abs(out[0]["kl_local"] - full["kl"]) > 1e-6 * abs(full["kl"])
