"""Group-sharded MSA across ranks: one process per GPU, each owning a contiguous range
of GQA groups.

Every group's block selection, main attention and backward are independent: a group
has its own index-query head and its own query heads, and its block set is shared by
those heads only (MSA summary, 7minutos.es, "¿Qué es MSA?" ¶4 and "Cómo funcionan las
dos ramas" ¶1-2).  The groups share one tensor, the index-key head k_idx, so its
gradient dk_idx sums over all groups, and the KL value is a sum over groups too.  A
sharded step therefore runs the single-GPU library on the rank's groups and ends with
one exchange: an all-reduce (sum) of dk_idx and of the KL.  Every other output (o,
lse, block_idx, lse_idx, dq, dk, dv, dq_idx) stays on the rank that owns its group.

The KL weight of a row is kl_coef / (B * H_kv * N) with the GLOBAL group count, so the
sharded KL and gradients equal the unsharded ones.
"""
from __future__ import annotations

import dataclasses


@dataclasses.dataclass(frozen=True)
class GroupShard:
    """Rank `rank` of `world` owns groups [g0, g1) of H_kv (contiguous, as even as
    possible: the first H_kv % world ranks take one more group)."""

    rank: int
    world: int
    H_kv: int

    def __post_init__(self):
        if not (0 <= self.rank < self.world) or self.H_kv <= 0:
            raise ValueError(f"bad shard: rank {self.rank} of {self.world}, H_kv {self.H_kv}")

    @property
    def groups(self) -> tuple[int, int]:
        base, extra = divmod(self.H_kv, self.world)
        g0 = self.rank * base + min(self.rank, extra)
        return g0, g0 + base + (1 if self.rank < extra else 0)

    @property
    def n_groups(self) -> int:
        g0, g1 = self.groups
        return g1 - g0

    def take(self, name: str, x):
        """This rank's slice of a step input or a per-group output, contiguous.
        q, dO, o, dq [B,N,H_q,d]: the owned groups' query heads; k, v, q_idx, dk, dv,
        dq_idx [B,N,H_kv,*]: the owned groups; lse [B,H_q,N], block_idx, lse_idx
        [B,H_kv,...]: along the head axis; k_idx, dk_idx [B,N,d_idx]: whole."""
        g0, g1 = self.groups
        if name in ("k_idx", "dk_idx"):
            return x
        if name in ("q", "dO", "o", "dq"):
            G = x.shape[2] // self.H_kv
            return x[:, :, g0 * G:g1 * G].contiguous()
        if name in ("k", "v", "q_idx", "dk", "dv", "dq_idx"):
            return x[:, :, g0:g1].contiguous()
        if name == "lse":
            G = x.shape[1] // self.H_kv
            return x[:, g0 * G:g1 * G].contiguous()
        if name in ("block_idx", "lse_idx"):
            return x[:, g0:g1].contiguous()
        raise KeyError(name)

    def kl_weight(self, B: int, N: int, kl_coef: float) -> float:
        return kl_coef / float(B * self.H_kv * N)


def exchange(grads: dict, group=None) -> dict:
    """The step's one exchange: dk_idx and the KL summed over ranks (in float32; the
    bf16 dk_idx of each rank is widened before the sum and rounded once after it).
    `grads` holds this rank's msa_bwd outputs; returns it with both replaced."""
    import torch
    import torch.distributed as dist

    dki = grads["dk_idx"]
    acc = dki.float()
    dist.all_reduce(acc, op=dist.ReduceOp.SUM, group=group)
    kl = grads["kl"].reshape(1).float().clone()
    dist.all_reduce(kl, op=dist.ReduceOp.SUM, group=group)
    out = dict(grads)
    out["dk_idx"] = acc.to(dki.dtype)
    out["kl"] = kl.reshape(grads["kl"].shape)
    return out


def sharded_step(shard: GroupShard, inputs: dict, topk: int, *, scale=None, kl_coef: float = 1.0,
                 compute=None, group=None) -> dict:
    """One MSA training step (index branch, forward, fused backward) over this rank's
    groups, followed by the exchange.  `inputs` holds the FULL tensors q, k, v, q_idx,
    k_idx, dO (each rank slices its own); `compute(x, topk, scale, w)` runs the step on
    a slice and returns block_idx, lse_idx, o, lse and the gradients (default: the
    library's msa_index_topk, msa_fwd, msa_bwd on the current CUDA stream).  Returns
    the rank's outputs with dk_idx and kl summed over ranks."""
    x = {n: shard.take(n, inputs[n]) for n in ("q", "k", "v", "q_idx", "k_idx", "dO")}
    B, N = x["q"].shape[0], x["q"].shape[1]
    w = shard.kl_weight(B, N, kl_coef)
    out = (compute or library_step)(x, topk, scale, w)
    return exchange(out, group=group)


def library_step(x: dict, topk: int, scale, w: float) -> dict:
    """The single-GPU step on one rank's slice through the C ABI."""
    from . import ops

    H_q, d = x["q"].shape[2], x["q"].shape[3]
    bi, li = ops.msa_index_topk(x["q_idx"], x["k_idx"], topk, H_q=H_q, d=d)
    o, lse = ops.msa_fwd(x["q"], x["k"], x["v"], bi, scale=scale, d_idx=x["q_idx"].shape[3])
    g = ops.msa_bwd(x["q"], x["k"], x["v"], o, lse, x["dO"], x["q_idx"], x["k_idx"], bi, li, w,
                    scale=scale)
    out = dict(g)
    out.update(block_idx=bi, lse_idx=li, o=o, lse=lse)
    return out
