#!/usr/bin/env python
"""Benchmark of the MSA training hot path on GB300.

One step = the whole hot path over one batch of the 128K workload (B=1,
N=131072, H_q=32, H_kv=8, d=128, d_idx=64, Bk=128, k=16, causal; seeded
N(0,1) inputs with 16 needle blocks per group): index scoring + top-k (+ index
LSE), block-sparse forward, fused backward with the KL gradient.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  `value` is device-timed tokens/s with inputs resident in
HBM; `e2e` is the same metric through the public API with pinned host inputs
copied in and the KL read back every step; `roofline` is the dominant kernel,
timed live with CUDA events around its launches inside the timed steps;
`cpu_baseline` is the float64 oracle on a bounded row sample on the host cores;
`workloads` times the same step on each of the five seeded workloads (tiny, 8K, 32K,
128K, 1M): ms per step, per forward (index branch + sparse attention), per backward,
the index scoring + top-k kernel alone, tokens/s and each kernel's fraction of peak.
`--impl reference` times that oracle alone (the reference arm).
Under torchrun (N > 1) the ranks shard one problem by GQA group (each rank owns a
contiguous range of the groups; the step ends with the one exchange, an all-reduce
of dk_idx and the KL): strong scaling, value = the problem's tokens / max rank time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_gqa_topk_gb300 import synth  # noqa: E402

METRIC = "MSA fwd+bwd tokens/s @128K (Bk=128,k=16); % of bf16 tensor-pipe peak"
# the five seeded workloads, each timed by the default run (the 128K one is the headline)
WORKLOAD_ORDER = ("tiny", "8k", "32k", "128k", "1m")
WORKLOAD_STEPS = {"tiny": 20, "8k": 20, "32k": 10, "128k": 10, "1m": 3}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def cfg_label(cfg):
    """The workload's short name as the text writes it: 128K, 1M, tiny."""
    return cfg.name.upper() if cfg.name[:1].isdigit() else cfg.name


def workload_name(cfg):
    return (f"MSA fwd+bwd: B={cfg.B} N={cfg.N} H_q={cfg.H_q} H_kv={cfg.H_kv} d={cfg.d} "
            f"d_idx={cfg.d_idx} Bk={cfg.Bk} k={cfg.topk} causal bf16, N(0,1) + "
            f"{cfg.n_needle} needle blocks/group, seed {cfg.seed}")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "of measured"
    return dict(FALLBACK_PEAKS), "of fallback"


def job_rate(local_ms, units_per_rank, world, device=None):
    """Whole-job throughput of `world` ranks that each processed `units_per_rank`
    units in `local_ms`: the job takes as long as its slowest rank (max over ranks,
    an all-reduce on the default process group when world > 1).  Returns
    (max_ms, units of all ranks per second)."""
    ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, units_per_rank * world / (ms / 1000.0)


def decode_leg(torch, ops, d, cfg, dev, stream, hbm_peak, calls=20):
    """Decode (one new token per sequence) over 8 caches of the workload's length: mean
    device time per call with L2 flushed before each call, and the algorithmic HBM bytes
    a call must move (every cached index key, the K/V rows of the selected blocks, the
    new token's q and the output)."""
    Bd, L = 8, cfg.N
    k = d["k"].expand(Bd, -1, -1, -1).contiguous()
    v = d["v"].expand(Bd, -1, -1, -1).contiguous()
    k_idx = d["k_idx"].expand(Bd, -1, -1).contiguous()
    q_new = d["q"][0, L - 1].expand(Bd, -1, -1).contiguous()
    qi_new = d["q_idx"][0, L - 1].expand(Bd, -1, -1).contiguous()
    lens = torch.full((Bd,), L, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(3):
        ops.msa_decode(q_new, qi_new, k, v, k_idx, lens, cfg.topk, scale=cfg.scale)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(calls)]
    for a, b in evs:
        flush.zero_()
        # keep the GPU busy while the host enqueues the call, so the events bracket the
        # decode kernels only (not the host's launch latency)
        torch.cuda._sleep(1_000_000)
        a.record(stream)
        ops.msa_decode(q_new, qi_new, k, v, k_idx, lens, cfg.topk, scale=cfg.scale)
        b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    per_seq = (L * cfg.d_idx * 2 + cfg.H_kv * cfg.topk * cfg.Bk * cfg.d * 2 * 2
               + (cfg.H_q * cfg.d + cfg.H_kv * cfg.d_idx) * 2 + cfg.H_q * cfg.d * 2)
    nbytes = Bd * per_seq
    gbs = nbytes / (ms / 1000.0) / 1e9
    # the same calls over an FP8 (E4M3) cache: 1-byte K/V codes + one f32 scale per row
    k8, ks = ops.msa_quantize_kv_fp8(k)
    v8, vs = ops.msa_quantize_kv_fp8(v)
    del k, v
    for _ in range(3):
        ops.msa_decode_fp8(q_new, qi_new, k8, v8, ks, vs, k_idx, lens, cfg.topk, scale=cfg.scale)
    for a, b in evs:
        flush.zero_()
        torch.cuda._sleep(1_000_000)
        a.record(stream)
        ops.msa_decode_fp8(q_new, qi_new, k8, v8, ks, vs, k_idx, lens, cfg.topk, scale=cfg.scale)
        b.record(stream)
    torch.cuda.synchronize()
    ms8 = statistics.mean(a.elapsed_time(b) for a, b in evs)
    per_seq8 = (L * cfg.d_idx * 2 + cfg.H_kv * cfg.topk * cfg.Bk * (cfg.d + 4) * 2
                + (cfg.H_q * cfg.d + cfg.H_kv * cfg.d_idx) * 2 + cfg.H_q * cfg.d * 2)
    nbytes8 = Bd * per_seq8
    gbs8 = nbytes8 / (ms8 / 1000.0) / 1e9
    del k8, v8, ks, vs, k_idx, flush
    return {"batch": Bd, "cache_len": L, "ms_per_call": ms, "tokens_per_s": Bd / (ms / 1000.0),
            "bound": "hbm", "bytes_per_call": nbytes, "achieved_gbs": gbs, "peak_gbs": hbm_peak,
            "frac": gbs / hbm_peak, "l2": "flushed before each call",
            "timing": "CUDA events around each call, queued behind a GPU spin",
            "fp8": {"cache": "E4M3 codes + f32 scale per (token, head) row", "ms_per_call": ms8,
                    "tokens_per_s": Bd / (ms8 / 1000.0), "bytes_per_call": nbytes8,
                    "achieved_gbs": gbs8, "frac": gbs8 / hbm_peak}}


def fp8_forward_leg(torch, ops, _lib, d, cfg, stream, peak_tf, steps=5):
    """FP8 (E4M3) training forward on the workload: the quantiser (q per row, k and v per
    128-key block) and msa_fwd_fp8 over the step's block sets, each timed per call (CUDA
    events, mean of `steps` after a warm-up call), with the tensor-core kernel alone timed
    live, against msa_fwd (bf16) on the same sets.  The FP8 kernel's peak is the bf16
    measured peak times the nominal 2x ratio of E4M3 to bf16 tensor throughput."""
    bi, _ = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d,
                               with_lse=False)
    torch.cuda.synchronize()
    flops = algorithmic_flops(cfg, token_set_total(cfg, bi.cpu().numpy()))["fwd"]

    def timed(fn, kernel_events):
        fn()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for e in ev:
            for x in e:
                x.record(stream)
        torch.cuda.synchronize()
        for e in ev:
            if kernel_events:
                _lib.msa_set_kernel_events(_lib.MSA_KERNEL_FWD, e[0].cuda_event, e[1].cuda_event)
            e[2].record(stream)
            fn()
            e[3].record(stream)
        torch.cuda.synchronize()
        _lib.msa_set_kernel_events(_lib.MSA_KERNEL_FWD, None, None)
        call = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
        kern = statistics.mean(e[0].elapsed_time(e[1]) for e in ev) if kernel_events else None
        return call, kern

    bf_call, bf_kern = timed(lambda: ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale,
                                                 d_idx=cfg.d_idx), True)
    ops8 = ops.msa_quantize_fwd_fp8(d["q"], d["k"], d["v"])
    q_call, _ = timed(lambda: ops.msa_quantize_fwd_fp8(d["q"], d["k"], d["v"]), False)
    f8_call, f8_kern = timed(lambda: ops.msa_fwd_fp8(*ops8, bi, scale=cfg.scale,
                                                     d_idx=cfg.d_idx), True)
    del ops8, bi
    tf8 = flops / (f8_kern / 1000.0) / 1e12
    return {"recipe": "E4M3; q one scale per (token, head) row, k and v one per 128-key block; "
                      "P rounded to E4M3 against the block's exact max",
            "ms_quantize": q_call, "ms_forward_call": f8_call, "ms_forward_kernel": f8_kern,
            "bf16_ms_forward_call": bf_call, "bf16_ms_forward_kernel": bf_kern,
            "kernel_tflops": tf8, "peak_tflops": 2.0 * peak_tf,
            "peak_source": "bf16_tflops_sustained x 2 (nominal E4M3 / bf16 ratio)",
            "frac": tf8 / (2.0 * peak_tf), "steps": steps}


def warmup_leg(torch, ops, cfg, dev, stream, peak_tf, steps=5, warm=3):
    """Indexer warm-up (dense set, topk >= nb): the workload's heads at N = 16384 with
    topk = 128 = nb, so both branches attend every visible token and the KL runs over
    all of them.  One step = index call (dense set + lse_idx), forward, backward; mean
    device time over `steps` steps after `warm` untimed ones (inputs > L2)."""
    wc = cfg.with_(name="warmup-16k", B=1, N=16384, topk=128, n_needle=4)
    host = synth.make_inputs(wc)
    t = {n: torch.from_numpy(host[n].view(np.int16)).to(dev).view(torch.bfloat16)
         for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
    w = wc.kl_coef / (wc.B * wc.H_kv * wc.N)

    plan = ops.new_plan(wc.B, wc.N, wc.H_q, wc.H_kv, wc.topk, d=wc.d, d_idx=wc.d_idx, device=dev)

    def step():
        bi, li = ops.msa_index_topk(t["q_idx"], t["k_idx"], wc.topk, H_q=wc.H_q, d=wc.d,
                                    plan=plan)
        o, lse = ops.msa_fwd(t["q"], t["k"], t["v"], bi, scale=wc.scale, d_idx=wc.d_idx, plan=plan)
        g = ops.msa_bwd(t["q"], t["k"], t["v"], o, lse, t["dO"], t["q_idx"], t["k_idx"], bi, li,
                        w, scale=wc.scale, plan=plan)
        return bi, g

    for _ in range(warm):
        bi, _ = step()
    torch.cuda.synchronize()
    sum_T = token_set_total(wc, bi.cpu().numpy())
    f = algorithmic_flops(wc, sum_T)
    flops = f["index_lse"] + f["fwd"] + f["bwd"]  # no block scoring: the set is forced
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1000.0) / 1e12
    del t
    return {"workload": workload_name(wc) + " (dense set: every visible block)",
            "ms_per_step": ms, "tokens_per_s": wc.B * wc.N / (ms / 1000.0),
            "algorithmic_tflop_per_step": flops / 1e12, "tflops": tf, "peak_tflops": peak_tf,
            "frac": tf / peak_tf, "steps": steps}


def varlen_leg(torch, ops, _lib, d, cfg, stream, peak_tf, steps=5, warm=3):
    """Packed variable-length batch over the workload's token axis and heads: 32
    sequences whose seeded lengths are log-uniform in 512 .. 16384 tokens, scaled to fill
    the B*N tokens exactly (cu_seqlens on the device).  One step = index call (+ lse_idx),
    forward, backward through the packed entry points; mean device time over `steps`
    steps after `warm` untimed ones.  Algorithmic work = the sum of every sequence's own
    work (each is its own causal problem)."""
    T = cfg.B * cfg.N
    cu = synth.varlen_offsets_total(32, T, 512, 16384, seed=55)
    lens = [b - a for a, b in zip(cu, cu[1:])]
    L = max(lens)
    cu_t = torch.tensor(cu, dtype=torch.int32, device=d["q"].device)
    t = {n: d[n].reshape((T,) + tuple(d[n].shape[2:])) for n in d}
    w = cfg.kl_coef / (cfg.H_kv * T)
    k = cfg.topk

    def step():
        bi, li = ops.msa_index_topk_varlen(t["q_idx"], t["k_idx"], cu_t, k, max_seqlen=L,
                                           H_q=cfg.H_q, d=cfg.d)
        o, lse = ops.msa_fwd_varlen(t["q"], t["k"], t["v"], bi, cu_t, k, max_seqlen=L,
                                    scale=cfg.scale, d_idx=cfg.d_idx)
        g = ops.msa_bwd_varlen(t["q"], t["k"], t["v"], o, lse, t["dO"], t["q_idx"], t["k_idx"], bi,
                               li, w, cu_t, k, max_seqlen=L, scale=cfg.scale)
        return bi, g

    for _ in range(warm):
        bi, _ = step()
    torch.cuda.synchronize()
    bi_h = bi.cpu().numpy()
    flops = {"index": 0, "index_lse": 0, "fwd": 0, "bwd": 0}
    for s, n in enumerate(lens):
        if n == 0:
            continue
        cs = cfg.with_(B=1, N=n)
        view = bi_h[cu[s] * cfg.H_kv * k:cu[s + 1] * cfg.H_kv * k].reshape(1, cfg.H_kv, n, k)
        for key, v in algorithmic_flops(cs, token_set_total(cs, view)).items():
            flops[key] += v
    n0 = _lib.msa_kernel_launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = (_lib.msa_kernel_launch_count() - n0) // steps
    ms = e0.elapsed_time(e1) / steps
    total = sum(flops.values())
    tf = total / (ms / 1000.0) / 1e12
    return {"workload": (f"packed batch of {len(lens)} sequences ({min(lens)} .. {L} tokens, "
                         f"log-uniform, seed 55) filling {T} tokens; H_q={cfg.H_q} "
                         f"H_kv={cfg.H_kv} d={cfg.d} d_idx={cfg.d_idx} k={k}"),
            "num_seqs": len(lens), "max_seqlen": L, "ms_per_step": ms,
            "tokens_per_s": T / (ms / 1000.0), "launches_per_step": launches,
            "algorithmic_tflop_per_step": total / 1e12, "tflops": tf, "peak_tflops": peak_tf,
            "frac": tf / peak_tf, "steps": steps}


# ----------------------------------------------------------------------------
# algorithmic work (what the method must compute, not what a kernel happens to do)
# ----------------------------------------------------------------------------
def token_set_total(cfg, block_idx_np):
    """Sum over (b, g, i) of |T(b,g,i)|: selected blocks wholly before the query
    count Bk tokens, the own block counts i - Bk*c_i + 1."""
    i = np.arange(cfg.N)
    ci = i // cfg.Bk
    bi = block_idx_np
    full = ((bi >= 0) & (bi < ci[None, None, :, None])).sum(axis=-1)
    tot = full.astype(np.int64).sum() * cfg.Bk + cfg.B * cfg.H_kv * int((i - ci * cfg.Bk + 1).sum())
    return int(tot)


def algorithmic_flops(cfg, sum_T):
    nb = cfg.nb
    full_blocks = cfg.N // cfg.Bk
    idx = 2 * cfg.d_idx * cfg.Bk * cfg.Bk * (full_blocks * (full_blocks - 1) // 2) * cfg.H_kv * cfg.B
    G = cfg.G
    fwd_main = 4 * cfg.d * sum_T * G           # S = QK^T and O = PV, every head of the group
    idx_lse = 2 * cfg.d_idx * sum_T            # index logits over T, once per group
    bwd_main = 10 * cfg.d * sum_T * G          # S, dP recompute; dV, dK, dQ
    bwd_kl = 6 * cfg.d_idx * sum_T             # z recompute; dk_idx, dq_idx
    _ = nb
    return {"index": idx, "index_lse": idx_lse, "fwd": fwd_main, "bwd": bwd_main + bwd_kl}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            if gpu_id:
                cmd += ["-i", gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# the oracle on a bounded sample (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(cfg, host, n_rows, seed):
    import oracle
    rows = synth.sample_rows(cfg, n_rows, seed)
    t0 = time.perf_counter()
    bi, _, _ = oracle.select(cfg, host, rows=rows)
    oracle.forward(cfg, host, bi, rows=rows)
    oracle.backward(cfg, host, bi, cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N), rows=rows)
    dt = time.perf_counter() - t0
    return len(rows), dt


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    host = synth.make_inputs(cfg)
    rows_per_step = args.ref_rows
    for w in range(args.warmup):
        oracle_sample(cfg, host, rows_per_step, seed=500 + w)
    total_rows, total_t = 0, 0.0
    for k in range(args.steps):
        n, dt = oracle_sample(cfg, host, rows_per_step, seed=600 + k)
        total_rows += n
        total_t += dt
    v = total_rows / total_t
    cores = os.cpu_count()
    sample = (f"{rows_per_step} seeded query rows (+ first/last) of the {cfg_label(cfg)} workload per step, "
              f"all {cfg.H_kv} groups: index top-k, forward, backward in float64")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(cfg), "global_batch": cfg.B, "seq_len": cfg.N,
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# one workload: warm-up steps, then K timed steps with live per-kernel events
# ----------------------------------------------------------------------------
def timed_workload(torch, ops, _lib, cfg, d, stream, steps, warmup, barrier=None,
                   clock_gpu=False, kl_weight=None, after_bwd=None):
    """Times `steps` whole steps (index scoring + top-k + index LSE, forward, fused
    backward) of workload `cfg` on the device-resident inputs `d`, after `warmup`
    untimed steps.  Returns the mean step time, live per-kernel times (CUDA events the
    library records around its four tensor-core kernels), per-phase times, the
    algorithmic FLOPs of one step, the launch count and the clock record.  In the
    group-sharded mode `cfg` and `d` are this rank's groups, `kl_weight` uses the global
    group count and `after_bwd` is the exchange (all-reduce of dk_idx and the KL)."""
    w = kl_weight if kl_weight is not None else cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    # one plan (inverted lists of the step's block_idx) serves the index LSE, forward and
    # backward of each step: built by the index call, read by the other two
    plan = ops.new_plan(cfg.B, cfg.N, cfg.H_q, cfg.H_kv, cfg.topk, d=cfg.d, d_idx=cfg.d_idx,
                        device=d["q"].device)

    def step(t, phase_ev=None):
        if phase_ev:
            phase_ev[0].record(stream)
        bi, li = ops.msa_index_topk(t["q_idx"], t["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d,
                                    plan=plan)
        if phase_ev:
            phase_ev[1].record(stream)
        o, lse = ops.msa_fwd(t["q"], t["k"], t["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx,
                             plan=plan)
        if phase_ev:
            phase_ev[2].record(stream)
        g = ops.msa_bwd(t["q"], t["k"], t["v"], o, lse, t["dO"], t["q_idx"], t["k_idx"], bi, li, w,
                        scale=cfg.scale, plan=plan)
        if after_bwd is not None:
            g = after_bwd(g)
        if phase_ev:
            phase_ev[3].record(stream)
        return bi, g

    for _ in range(warmup):
        bi, g = step(d)
    torch.cuda.synchronize()
    st = ops.device_status()
    if st != 0:
        raise RuntimeError(f"{cfg.name}: device status after warm-up: {_lib.status_string(st)}")
    sum_T = token_set_total(cfg, bi.cpu().numpy())
    flops = algorithmic_flops(cfg, sum_T)
    del bi, g

    K = steps
    kev = {kname: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K)] for kname in ("index", "index_lse", "fwd", "bwd")}
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for lst in kev.values():  # materialise the events so their handles exist
        for a, b in lst:
            a.record(stream)
            b.record(stream)
    kid = {"index": _lib.MSA_KERNEL_INDEX, "index_lse": _lib.MSA_KERNEL_INDEX_LSE,
           "fwd": _lib.MSA_KERNEL_FWD, "bwd": _lib.MSA_KERNEL_BWD}
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    clocks = ClockSampler(clock_gpu) if clock_gpu is not False else None
    if clocks is not None:
        time.sleep(0.3)
    launches0 = _lib.msa_kernel_launch_count()
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(K):
        for kname, lst in kev.items():
            _lib.msa_set_kernel_events(kid[kname], lst[s][0].cuda_event, lst[s][1].cuda_event)
        step(d, pev[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    launches = _lib.msa_kernel_launch_count() - launches0
    clk = clocks.stop() if clocks is not None else None
    for kname in kev:
        _lib.msa_set_kernel_events(kid[kname], None, None)
    st = ops.device_status()
    if st != 0:
        raise RuntimeError(f"{cfg.name}: device status after timed steps: {_lib.status_string(st)}")
    kern_ms = {k: statistics.mean(a.elapsed_time(b) for a, b in v) for k, v in kev.items()}
    phase_ms = {
        "index": statistics.mean(e[0].elapsed_time(e[1]) for e in pev),
        "fwd": statistics.mean(e[1].elapsed_time(e[2]) for e in pev),
        "bwd": statistics.mean(e[2].elapsed_time(e[3]) for e in pev),
    }
    return {"ms": t_start.elapsed_time(t_end) / K, "kernels_ms": kern_ms, "phases_ms": phase_ms,
            "flops": flops, "sum_T": sum_T, "launches": launches, "clocks": clk, "steps": K}


def graph_step(torch, ops, cfg, d, kl_weight=None, replays=10):
    """One whole step (index scoring + top-k + index LSE, forward, fused backward) on the
    device-resident inputs `d`, captured once in a CUDA graph and replayed: the step
    without per-launch host overhead, which bounds the small workloads.  The library
    allocates nothing and queues only memsets and kernels on the caller's stream, so the
    captured calls are the eager ones.  Returns ms per replayed step."""
    w = kl_weight if kl_weight is not None else cfg.kl_coef / (cfg.B * cfg.H_kv * cfg.N)
    plan = ops.new_plan(cfg.B, cfg.N, cfg.H_q, cfg.H_kv, cfg.topk, d=cfg.d, d_idx=cfg.d_idx,
                        device=d["q"].device)

    def step():
        bi, li = ops.msa_index_topk(d["q_idx"], d["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d,
                                    plan=plan)
        o, lse = ops.msa_fwd(d["q"], d["k"], d["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx,
                             plan=plan)
        return ops.msa_bwd(d["q"], d["k"], d["v"], o, lse, d["dO"], d["q_idx"], d["k_idx"], bi, li,
                           w, scale=cfg.scale, plan=plan)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):  # the workspace is sized before the capture
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / replays
    del graph
    return ms


def workload_summary(cfg, r, peak_tf):
    """Per-workload record: ms per step, per forward (index branch + sparse attention)
    and per backward, the index scoring + top-k kernel alone, tokens/s, and each
    tensor-core kernel's algorithmic TFLOP/s and fraction of the bf16 peak."""
    ms, kern, ph, f = r["ms"], r["kernels_ms"], r["phases_ms"], r["flops"]
    ktf = {k: f[k] / (kern[k] / 1000.0) / 1e12 for k in kern}
    return {
        "workload": workload_name(cfg), "steps": r["steps"], "ms_per_step": ms,
        "tokens_per_s": cfg.B * cfg.N / (ms / 1000.0),
        "ms_forward": ph["index"] + ph["fwd"], "ms_backward": ph["bwd"],
        "ms_index_topk": kern["index"], "phases_ms": ph, "kernels_ms": kern,
        "kernel_tflops": ktf, "kernel_frac_of_peak": {k: v / peak_tf for k, v in ktf.items()},
        "algorithmic_tflop_per_step": sum(f.values()) / 1e12,
        "pct_bf16_peak_step": sum(f.values()) / (ms / 1000.0) / 1e12 / peak_tf,
    }


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def run_ours(args, cfg, rank, world):
    import torch
    import torch.distributed as dist
    from block_sparse_gqa_topk_gb300 import _lib, ops

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    _lib.load()
    host = synth.make_inputs(cfg)
    names = ("q", "k", "v", "q_idx", "k_idx", "dO")

    def to_dev(x):
        return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)

    full_cfg = cfg
    after_bwd = None
    if world > 1:
        # group-sharded mode: this rank owns a contiguous range of the GQA groups and
        # the step ends with the one exchange (all-reduce of dk_idx and the KL)
        from block_sparse_gqa_topk_gb300 import shard
        sh = shard.GroupShard(rank, world, cfg.H_kv)
        host_t = {n: sh.take(n, torch.from_numpy(host[n].view(np.int16))) for n in names}
        host = {n: host_t[n].numpy().view(np.uint16) for n in names}
        del host_t
        cfg = cfg.with_(H_q=sh.n_groups * cfg.G, H_kv=sh.n_groups)
        after_bwd = shard.exchange
    d = {n: to_dev(host[n]) for n in names}
    w = full_cfg.kl_coef / (full_cfg.B * full_cfg.H_kv * full_cfg.N)
    stream = torch.cuda.current_stream(dev)
    if args.warmup_only:  # the indexer warm-up leg alone
        peaks, _ = load_peaks()
        wu = warmup_leg(torch, ops, cfg, dev, stream, float(
            peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])))
        if ops.device_status() != 0:
            raise RuntimeError("device status after warm-up leg: "
                               + _lib.status_string(ops.device_status()))
        if rank == 0:
            print(json.dumps({"indexer_warmup": wu}), flush=True)
        return
    if args.varlen_only:  # the packed variable-length leg alone
        peaks, _ = load_peaks()
        vl = varlen_leg(torch, ops, _lib, d, cfg, stream, float(
            peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])))
        if ops.device_status() != 0:
            raise RuntimeError("device status after the varlen leg: "
                               + _lib.status_string(ops.device_status()))
        if rank == 0:
            print(json.dumps({"varlen": vl}), flush=True)
        return
    if args.decode_only:  # the decode leg alone (e.g. for a profiler's launch list)
        peaks, _ = load_peaks()
        dec = decode_leg(torch, ops, d, cfg, dev, stream,
                         float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])))
        if ops.device_status() != 0:
            raise RuntimeError("device status after decode: "
                               + _lib.status_string(ops.device_status()))
        if rank == 0:
            print(json.dumps({"decode": dec}), flush=True)
        return

    def barrier():
        if world > 1:
            dist.barrier()

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    r = timed_workload(torch, ops, _lib, cfg, d, stream, args.steps, args.warmup,
                       barrier=barrier, clock_gpu=gpu_id, kl_weight=w, after_bwd=after_bwd)
    K = args.steps
    # strong scaling: the ranks share one problem of B*N tokens
    ms, value = job_rate(r["ms"], full_cfg.B * full_cfg.N / world, world, dev)
    kern_ms, phase_ms, flops, launches, clk = (r["kernels_ms"], r["phases_ms"], r["flops"],
                                               r["launches"], r["clocks"])
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    kflops = {k: flops[k] for k in kern_ms}
    dom = max(kern_ms, key=lambda k: kern_ms[k])
    achieved = kflops[dom] / (kern_ms[dom] / 1000.0) / 1e12
    traffic = None
    tf_path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tf_path):
        try:
            with open(tf_path) as f:
                traffic = json.load(f).get(cfg.name, {}).get(dom)
        except (OSError, ValueError, AttributeError):
            traffic = None
    total_flops = sum(flops.values())

    # ---- end to end through the public API with host buffers ----
    # Every step copies its own inputs from pinned host memory (h2d bytes below) and
    # reads its KL back to the host.  Two device input sets: the copies of step s+1 run
    # while step s's backward computes, as a training loop prefetches its next batch
    # (started after the forward, they stay clear of the index kernel, which relies on
    # L2 for its key tiles).  The copies are split over two copy streams (two copy
    # engines), and each call of a step waits only for the inputs it reads (index:
    # q_idx, k_idx; forward: q, k, v; backward: dO).
    pinned = {n: torch.from_numpy(host[n].view(np.int16)).pin_memory() for n in names}
    bufs = [{n: torch.empty_like(d[n]) for n in names} for _ in range(2)]
    e2e_steps = max(1, min(K, args.e2e_steps))
    kl_host = torch.empty(e2e_steps, dtype=torch.float32).pin_memory()
    h2d = sum(pinned[n].numel() * 2 for n in names)
    copy_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    plan = ops.new_plan(cfg.B, cfg.N, cfg.H_q, cfg.H_kv, cfg.topk, d=cfg.d, d_idx=cfg.d_idx,
                        device=dev)
    lanes = {"q_idx": 0, "q": 0, "k": 0, "k_idx": 1, "v": 1, "dO": 1}  # about 1.4 GB each
    landed = [{n: torch.cuda.Event() for n in names} for _ in range(2)]  # per set, per input
    consumed = [torch.cuda.Event() for _ in range(2)]  # the step reading set i is done
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def h2d_into(i, first):
        for cs in copy_streams:
            cs.wait_event(e0 if first else consumed[i])
        for n in ("q_idx", "k_idx", "q", "k", "v", "dO"):
            cs = copy_streams[lanes[n]]
            with torch.cuda.stream(cs):
                bufs[i][n].view(torch.int16).copy_(pinned[n], non_blocking=True)
            landed[i][n].record(cs)

    fwd_done = torch.cuda.Event()

    def e2e_step(i, after_fwd=None):
        t = bufs[i]
        for n in ("q_idx", "k_idx"):
            stream.wait_event(landed[i][n])
        bi, li = ops.msa_index_topk(t["q_idx"], t["k_idx"], cfg.topk, H_q=cfg.H_q, d=cfg.d,
                                    plan=plan)
        for n in ("q", "k", "v"):
            stream.wait_event(landed[i][n])
        o, lse = ops.msa_fwd(t["q"], t["k"], t["v"], bi, scale=cfg.scale, d_idx=cfg.d_idx,
                             plan=plan)
        if after_fwd is not None:
            after_fwd()
        stream.wait_event(landed[i]["dO"])
        g = ops.msa_bwd(t["q"], t["k"], t["v"], o, lse, t["dO"], t["q_idx"], t["k_idx"], bi, li,
                        w, scale=cfg.scale, plan=plan)
        return after_bwd(g) if after_bwd is not None else g

    torch.cuda.synchronize()
    barrier()
    e0.record(stream)
    h2d_into(0, True)
    for si in range(e2e_steps):
        i = si % 2
        nxt = None
        if si + 1 < e2e_steps:
            def nxt(si=si):
                # the next step's inputs stream in while this step's backward runs
                fwd_done.record(stream)
                for cs in copy_streams:
                    cs.wait_event(fwd_done)
                h2d_into((si + 1) % 2, si == 0)
        g = e2e_step(i, nxt)
        consumed[i].record(stream)
        kl_host[si:si + 1].copy_(g["kl"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms, e2e_val = job_rate(e0.elapsed_time(e1) / e2e_steps, full_cfg.B * full_cfg.N / world,
                               world, dev)
    del pinned, bufs

    # ---- decode (inference) leg ----
    dec = None
    if not args.no_decode and world == 1:
        dec = decode_leg(torch, ops, d, cfg, dev, stream,
                         float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])))

    # ---- FP8 (E4M3) training forward leg ----
    f8 = None
    if not args.no_fp8_leg and world == 1:
        f8 = fp8_forward_leg(torch, ops, _lib, d, cfg, stream, peak_tf)
        st = ops.device_status()
        if st != 0:
            raise RuntimeError(f"device status after the FP8 leg: {_lib.status_string(st)}")

    # ---- packed variable-length batch leg ----
    vl = None
    if not args.no_varlen_leg and world == 1:
        vl = varlen_leg(torch, ops, _lib, d, cfg, stream, peak_tf)
        st = ops.device_status()
        if st != 0:
            raise RuntimeError(f"device status after the varlen leg: {_lib.status_string(st)}")

    # ---- indexer warm-up leg (dense set) ----
    wu = None
    if not args.no_warmup_leg and world == 1:
        wu = warmup_leg(torch, ops, cfg, dev, stream, peak_tf)
        st = ops.device_status()
        if st != 0:
            raise RuntimeError(f"device status after warm-up leg: {_lib.status_string(st)}")

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_rows, dt = oracle_sample(cfg, host, args.cpu_rows, seed=900)
        cpu = {"value": n_rows / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": (f"{n_rows} seeded query rows of the {cfg_label(cfg)} workload, all {cfg.H_kv} groups: "
                          f"index top-k, forward, backward in float64 ({dt:.1f} s)")}

    # ---- every other seeded workload: the same step timed on its own inputs ----
    workloads = {cfg.name: workload_summary(cfg, r, peak_tf)}
    if world == 1 and not args.no_graph:
        gms = graph_step(torch, ops, cfg, d, kl_weight=w, replays=5)
        workloads[cfg.name]["graph"] = {"ms_per_step": gms,
                                        "tokens_per_s": cfg.B * cfg.N / (gms / 1000.0)}
        st = ops.device_status()
        if st != 0:
            raise RuntimeError(f"device status after the graph replay: {_lib.status_string(st)}")
    others = [] if (args.no_workloads or world > 1) else [n for n in WORKLOAD_ORDER
                                                          if n != cfg.name]
    if others:
        del d, host
        for n in others:
            torch.cuda.empty_cache()
            wc = synth.CONFIGS[n]
            hw = synth.make_inputs(wc)
            dw = {x: to_dev(hw[x]) for x in names}
            del hw
            rw = timed_workload(torch, ops, _lib, wc, dw, stream, WORKLOAD_STEPS[n], args.warmup)
            workloads[n] = workload_summary(wc, rw, peak_tf)
            if not args.no_graph:
                gms = graph_step(torch, ops, wc, dw, replays=max(3, WORKLOAD_STEPS[n]))
                workloads[n]["graph"] = {"ms_per_step": gms,
                                         "tokens_per_s": wc.B * wc.N / (gms / 1000.0)}
                st = ops.device_status()
                if st != 0:
                    raise RuntimeError(f"{n}: device status after the graph replay: "
                                       f"{_lib.status_string(st)}")
            del dw
        ops.release_workspace()
        torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(full_cfg), "global_batch": full_cfg.B,
                       "seq_len": full_cfg.N,
                       "parallelism": (f"group-sharded x{world} ({cfg.H_kv} of {full_cfg.H_kv} "
                                       "GQA groups per rank, all-reduce of dk_idx and KL)")
                       if world > 1 else "1 GPU",
                       "l2": "inputs larger than L2 (q and dO are 1.07 GB each)"},
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": traffic,
                         "peak_source": f"bf16_tflops_sustained {peak_src}"},
            "pct_bf16_peak_step": total_flops / (ms / 1000.0) / 1e12 / peak_tf,
            "kernels_ms": kern_ms, "phases_ms": phase_ms,
            "kernel_tflops": {k: kflops[k] / (kern_ms[k] / 1000.0) / 1e12 for k in kern_ms},
            "algorithmic_tflop_per_step": total_flops / 1e12,
            "e2e": {"value": e2e_val, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": 4, "steps": e2e_steps},
            "cpu_baseline": cpu,
            "workloads": {n: workloads[n] for n in WORKLOAD_ORDER if n in workloads},
            "decode": dec,
            "fp8_forward": f8,
            "varlen": vl,
            "indexer_warmup": wu,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--config", default="128k", choices=sorted(synth.CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-rows", type=int, default=1400)
    ap.add_argument("--ref-rows", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only the --config workload (skip the other four)")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode leg")
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the decode leg and print its JSON object")
    ap.add_argument("--no-fp8-leg", action="store_true",
                    help="skip the FP8 (E4M3) forward leg")
    ap.add_argument("--no-warmup-leg", action="store_true",
                    help="skip the indexer warm-up (dense set) leg")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing of each workload")
    ap.add_argument("--no-varlen-leg", action="store_true",
                    help="skip the packed variable-length batch leg")
    ap.add_argument("--varlen-only", action="store_true",
                    help="run only the packed variable-length leg and print its JSON object")
    ap.add_argument("--warmup-only", action="store_true",
                    help="run only the indexer warm-up leg and print its JSON object")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = synth.CONFIGS[args.config]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, cfg, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
