"""Multi-process checks of the N > 1 pieces, on CPU with the gloo backend (world size 2).

1. bench.job_rate: each rank gets the slowest rank's time and the whole-job rate
   (units of all ranks / max time), as the benchmark's torchrun mode reports it.
2. Group sharding (block_sparse_gqa_topk_gb300.shard).  Every GQA group's selection,
   forward and main backward are independent; the groups share only k_idx, whose
   gradient sums over groups (MSA summary, 7minutos.es, "Cómo funcionan las dos
   ramas" ¶1: one shared index-key head).  So a run split by group across ranks needs
   one exchange: an all-reduce (sum) of dk_idx and of the KL.  The product's
   sharded_step slices each rank's groups and runs the exchange over gloo; the
   per-rank step is injected (the oracle on CPU, where the library would run on a
   GPU).  The result must equal the unsharded oracle run; every other output must
   equal its group's slice.
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
SHARD3 = dict(SHARD, name="shard3", H_q=12, H_kv=3, seed=33, needle_seed=34)


def _oracle_compute(cfg):
    """The per-rank step of shard.sharded_step, computed by the oracle on the rank's
    slice (bf16 bits carried in int16 tensors), in place of the library on a GPU."""
    import torch
    import oracle

    def compute(x, topk, scale, w):
        ng = x["k"].shape[2]
        scfg = cfg.with_(H_q=ng * cfg.G, H_kv=ng)
        h = {n: np.ascontiguousarray(x[n].numpy().view(np.uint16)) for n in x}
        bi, _, _ = oracle.select(scfg, h)
        g = oracle.backward(scfg, h, bi, w)
        out = {n: g[n] for n in ("dq", "dk", "dv", "dq_idx")}
        out["block_idx"] = bi
        out["dk_idx"] = torch.from_numpy(np.ascontiguousarray(g["dk_idx"]))
        out["kl"] = torch.tensor(g["kl"], dtype=torch.float64)
        out["kl_local"] = g["kl"]
        return out

    return compute


def _shard_job_for(spec):
    def job(rank, world):
        import torch
        from block_sparse_gqa_topk_gb300 import shard, synth
        cfg = synth.MSAConfig(**spec)
        host = synth.make_inputs(cfg)
        full = {n: torch.from_numpy(host[n].view(np.int16)) for n in host}
        sh = shard.GroupShard(rank, world, cfg.H_kv)
        out = shard.sharded_step(sh, full, cfg.topk, scale=cfg.scale, kl_coef=cfg.kl_coef,
                                 compute=_oracle_compute(cfg))
        out["groups"] = sh.groups
        out["dk_idx"] = out["dk_idx"].numpy()
        out["kl"] = float(out["kl"])
        return out
    return job


def _shard_job(rank, world):
    return _shard_job_for(SHARD)(rank, world)


def _shard_job3(rank, world):
    return _shard_job_for(SHARD3)(rank, world)


@pytest.mark.parametrize("spec,job", [(SHARD, _shard_job), (SHARD3, _shard_job3)],
                         ids=["2-groups", "3-groups-uneven"])
def test_group_sharded_step_with_dk_idx_allreduce_matches_unsharded(spec, job):
    """shard.sharded_step (the product's sharded mode) on two gloo ranks, with the
    per-rank step computed by the oracle: every per-group output equals the unsharded
    oracle's slice, and after the one all-reduce every rank holds the unsharded
    dk_idx and KL."""
    import oracle
    from block_sparse_gqa_topk_gb300 import synth
    oracle.build()
    cfg = synth.MSAConfig(**spec)
    w = cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    inputs = synth.make_inputs(cfg)
    bi, _, _ = oracle.select(cfg, inputs)
    full = oracle.backward(cfg, inputs, bi, w)
    out = _run(job)
    G = cfg.G
    seen = []
    for r in range(2):
        s = out[r]
        g0, g1 = s["groups"]
        seen += list(range(g0, g1))
        np.testing.assert_array_equal(s["block_idx"], bi[:, g0:g1])
        np.testing.assert_allclose(s["dq"], full["dq"][:, g0 * G:g1 * G], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dk"], full["dk"][:, :, g0:g1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dv"], full["dv"][:, :, g0:g1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(s["dq_idx"], full["dq_idx"][:, g0:g1], rtol=0, atol=1e-12)
        # the exchange sums in float32
        scale = np.abs(full["dk_idx"]).max()
        np.testing.assert_allclose(s["dk_idx"], full["dk_idx"], rtol=0, atol=1e-6 * scale)
        assert s["kl"] == pytest.approx(full["kl"], rel=1e-6)
    assert sorted(seen) == list(range(cfg.H_kv))  # every group owned exactly once
    # the exchange is needed: one rank's share alone is not the answer
    assert abs(out[0]["kl_local"] - full["kl"]) > 1e-6 * abs(full["kl"])


def test_group_ranges_cover_every_group_once():
    from block_sparse_gqa_topk_gb300.shard import GroupShard
    for H_kv in (1, 2, 3, 8, 13):
        for world in (1, 2, 3, 4, 8):
            rs = [GroupShard(r, world, H_kv).groups for r in range(world)]
            assert rs[0][0] == 0 and rs[-1][1] == H_kv
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [g1 - g0 for g0, g1 in rs]
            assert max(sizes) - min(sizes) <= 1
