"""PyTorch-facing wrappers of the C ABI (device memory and streams only).

Each function checks dtypes/shapes, allocates outputs and a workspace with torch,
and calls the same-named entry point of libmsa.so on the current CUDA stream.
There is no fallback: without the built library or a CUDA device these raise.

Layouts (contiguous): q, o [B,N,H_q,d]; k, v [B,N,H_kv,d]; q_idx [B,N,H_kv,d_idx];
k_idx [B,N,d_idx]; lse [B,H_q,N] f32; lse_idx [B,H_kv,N] f32;
block_idx [B,H_kv,N,topk] int32.
"""
from __future__ import annotations

import math

import torch

from . import _lib

_WS = {}


def _workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    """Per-device scratch buffer, grown on demand (256-byte aligned by torch)."""
    key = (device.type, device.index)
    buf = _WS.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = buf
    return buf


def release_workspace() -> None:
    _WS.clear()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def make_problem(B, N, H_q, H_kv, d, d_idx, topk, Bk=128, causal=True, scale=None,
                 scale_idx=None) -> _lib.Problem:
    return _lib.Problem(B=B, N=N, H_q=H_q, H_kv=H_kv, d=d, d_idx=d_idx, Bk=Bk, topk=topk,
                        causal=int(bool(causal)),
                        scale=float(scale if scale is not None else 1.0 / math.sqrt(d)),
                        scale_idx=float(scale_idx if scale_idx is not None else 0.0))


def new_plan(B, N, H_q, H_kv, topk, *, d=128, d_idx=64, Bk: int = 128, causal: bool = True,
             device="cuda") -> torch.Tensor:
    """A buffer for one step's inverted lists ("plan").  Pass it as `plan=` to
    msa_index_topk, which builds it, then to msa_fwd and msa_bwd of the same step, which
    read it instead of each building their own (see include/msa.h)."""
    prob = make_problem(B, N, H_q, H_kv, d, d_idx, topk, Bk, causal, None, None)
    n = _lib.msa_plan_size(prob)
    if n == 0:
        raise ValueError("invalid problem for a plan")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _plan_arg(plan):
    if plan.dtype != torch.uint8 or not plan.is_cuda or not plan.is_contiguous():
        raise ValueError("plan must be a contiguous uint8 CUDA tensor from new_plan")
    return _ptr(plan), plan.numel()


def msa_index_topk(q_idx: torch.Tensor, k_idx: torch.Tensor, topk: int = 16, *, H_q=None, d=None,
                   Bk: int = 128, causal: bool = True, scale_idx=None, with_lse: bool = True,
                   plan=None):
    """Index branch: returns (block_idx [B,H_kv,N,topk] int32, lse_idx [B,H_kv,N] f32 or None).
    With `plan` (from new_plan) it also builds the step's shared plan there."""
    _need(q_idx, "q_idx", ndim=4)
    _need(k_idx, "k_idx", ndim=3)
    B, N, H_kv, d_idx = q_idx.shape
    if tuple(k_idx.shape) != (B, N, d_idx):
        raise ValueError(f"k_idx must be {(B, N, d_idx)}, got {tuple(k_idx.shape)}")
    prob = make_problem(B, N, H_q or H_kv, H_kv, d or 128, d_idx, topk, Bk, causal, None, scale_idx)
    dev = q_idx.device
    block_idx = torch.empty((B, H_kv, N, topk), dtype=torch.int32, device=dev)
    lse_idx = torch.empty((B, H_kv, N), dtype=torch.float32, device=dev) if with_lse else None
    nws = _lib.msa_workspace_size(prob, _lib.MSA_WS_INDEX) if with_lse else 0
    ws = _workspace(nws, dev) if with_lse else None
    if plan is None:
        rc = _lib.msa_index_topk(prob, _ptr(q_idx), _ptr(k_idx), _ptr(block_idx), _ptr(lse_idx),
                                 _ptr(ws), nws, _stream(dev))
    else:
        pp, pn = _plan_arg(plan)
        rc = _lib.msa_index_topk_plan(prob, _ptr(q_idx), _ptr(k_idx), _ptr(block_idx),
                                      _ptr(lse_idx), pp, pn, _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_index_topk")
    return block_idx, lse_idx


def msa_fwd(q, k, v, block_idx, *, scale=None, Bk: int = 128, causal: bool = True, d_idx=64,
            plan=None):
    """Main branch forward: returns (o [B,N,H_q,d] bf16, lse [B,H_q,N] f32).  With `plan`
    it reads the step's shared plan (built by msa_index_topk for this block_idx)."""
    _need(q, "q", ndim=4)
    _need(k, "k", ndim=4)
    _need(v, "v", ndim=4)
    _need(block_idx, "block_idx", torch.int32, ndim=4)
    B, N, H_q, d = q.shape
    H_kv = k.shape[2]
    topk = block_idx.shape[3]
    if tuple(k.shape) != (B, N, H_kv, d) or tuple(v.shape) != (B, N, H_kv, d):
        raise ValueError("k, v must be [B,N,H_kv,d] matching q")
    if tuple(block_idx.shape) != (B, H_kv, N, topk):
        raise ValueError("block_idx must be [B,H_kv,N,topk]")
    prob = make_problem(B, N, H_q, H_kv, d, d_idx, topk, Bk, causal, scale, None)
    dev = q.device
    o = torch.empty_like(q)
    lse = torch.empty((B, H_q, N), dtype=torch.float32, device=dev)
    nws = _lib.msa_workspace_size(prob, _lib.MSA_WS_FWD)
    ws = _workspace(nws, dev)
    if plan is None:
        rc = _lib.msa_fwd(prob, _ptr(q), _ptr(k), _ptr(v), _ptr(block_idx), _ptr(o), _ptr(lse),
                          _ptr(ws), nws, _stream(dev))
    else:
        pp, pn = _plan_arg(plan)
        rc = _lib.msa_fwd_plan(prob, _ptr(q), _ptr(k), _ptr(v), _ptr(block_idx), pp, pn, _ptr(o),
                               _ptr(lse), _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_fwd")
    return o, lse


def msa_bwd(q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight: float, *,
            scale=None, scale_idx=None, Bk: int = 128, causal: bool = True, plan=None):
    """Fused backward: returns dict dq, dk, dv, dq_idx, dk_idx (bf16) and kl (f32 [1]).
    With `plan` it reads the step's shared plan (built by msa_index_topk)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (q_idx, "q_idx")):
        _need(t, n, ndim=4)
    _need(k_idx, "k_idx", ndim=3)
    _need(lse, "lse", torch.float32, ndim=3)
    _need(lse_idx, "lse_idx", torch.float32, ndim=3)
    _need(block_idx, "block_idx", torch.int32, ndim=4)
    B, N, H_q, d = q.shape
    H_kv = k.shape[2]
    d_idx = q_idx.shape[3]
    topk = block_idx.shape[3]
    prob = make_problem(B, N, H_q, H_kv, d, d_idx, topk, Bk, causal, scale, scale_idx)
    dev = q.device
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
           "dq_idx": torch.empty_like(q_idx), "dk_idx": torch.empty_like(k_idx),
           "kl": torch.empty(1, dtype=torch.float32, device=dev)}
    nws = _lib.msa_workspace_size(prob, _lib.MSA_WS_BWD)
    ws = _workspace(nws, dev)
    outs = (_ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dq_idx"]),
            _ptr(out["dk_idx"]), _ptr(out["kl"]), _ptr(ws), nws, _stream(dev))
    ins = (prob, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(q_idx), _ptr(k_idx),
           _ptr(block_idx), _ptr(lse_idx))
    if plan is None:
        rc = _lib.msa_bwd(*ins, kl_weight, *outs)
    else:
        rc = _lib.msa_bwd_plan(*ins, *_plan_arg(plan), kl_weight, *outs)
    _lib.check(rc, "msa_bwd")
    return out


def device_status() -> int:
    """Reads and clears the current device's status word (after syncing the stream)."""
    return _lib.msa_get_device_status(_stream(torch.device("cuda", torch.cuda.current_device())))


class MSAFunction(torch.autograd.Function):
    """o = MSA(q, k, v, q_idx, k_idx).  Backward returns dq, dk, dv from dO and the
    KL-alignment gradients for q_idx, k_idx (teacher detached).  The KL value of
    the last backward is kept in ctx-free storage `MSAFunction.last_kl`."""

    last_kl = None

    @staticmethod
    def forward(ctx, q, k, v, q_idx, k_idx, topk, Bk, scale, scale_idx, kl_coef):
        B, N, H_q, d = q.shape
        # one plan (inverted lists of block_idx) serves the index LSE, forward and backward
        plan = new_plan(B, N, H_q, k.shape[2], topk, d=d, d_idx=q_idx.shape[3], Bk=Bk,
                        device=q.device)
        block_idx, lse_idx = msa_index_topk(q_idx, k_idx, topk, H_q=H_q, d=d, Bk=Bk,
                                            scale_idx=scale_idx, with_lse=True, plan=plan)
        o, lse = msa_fwd(q, k, v, block_idx, scale=scale, Bk=Bk, d_idx=q_idx.shape[3], plan=plan)
        ctx.save_for_backward(q, k, v, q_idx, k_idx, o, lse, block_idx, lse_idx, plan)
        ctx.cfg = (Bk, scale, scale_idx, kl_coef)
        ctx.mark_non_differentiable(block_idx)
        return o, block_idx

    @staticmethod
    def backward(ctx, dO, _dblock):
        q, k, v, q_idx, k_idx, o, lse, block_idx, lse_idx, plan = ctx.saved_tensors
        Bk, scale, scale_idx, kl_coef = ctx.cfg
        B, N, H_q, _ = q.shape
        H_kv = k.shape[2]
        w = kl_coef / float(B * H_kv * N)
        g = msa_bwd(q, k, v, o, lse, dO.contiguous(), q_idx, k_idx, block_idx, lse_idx, w,
                    scale=scale, scale_idx=scale_idx, Bk=Bk, plan=plan)
        MSAFunction.last_kl = g["kl"]
        return g["dq"], g["dk"], g["dv"], g["dq_idx"], g["dk_idx"], None, None, None, None, None


def attention(q, k, v, q_idx, k_idx, topk: int = 16, Bk: int = 128, scale=None, scale_idx=None,
              kl_coef: float = 1.0):
    """MSA attention for training: returns o; backward also trains the index heads.
    Stopping the gradient at the index-branch input is the caller's job (feed the
    projections a detached hidden state)."""
    o, _ = MSAFunction.apply(q, k, v, q_idx, k_idx, topk, Bk, scale, scale_idx, kl_coef)
    return o


# ---------------------------------------------------------------------------
# Packed variable-length batches (cu_seqlens on the device): each sequence is its own
# causal problem; token axes are packed, per-sequence outputs are stored one sequence
# after another in the single-sequence layout (see include/msa.h).  Every call runs a
# fixed number of kernels whatever the number of sequences; cu_seqlens is checked on
# the device (a bad batch writes nothing and sets the device status).
# ---------------------------------------------------------------------------
def _cu_dev(cu_seqlens, dev):
    if not isinstance(cu_seqlens, torch.Tensor):
        cu_seqlens = torch.tensor([int(x) for x in cu_seqlens], dtype=torch.int32)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.ndim != 1 or cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor of num_seqs + 1 offsets")
    return cu_seqlens.to(dev).contiguous()


def _max_len(cu, max_seqlen):
    """max_seqlen as given, else read from cu_seqlens (one device-to-host copy)."""
    if max_seqlen is not None:
        return int(max_seqlen)
    return int((cu[1:] - cu[:-1]).max()) if cu.numel() > 1 else 0


def varlen_view(flat: torch.Tensor, cu_seqlens, s: int, heads: int, per_row: int = 1):
    """Sequence s of a packed per-sequence output: [heads, L_s, per_row] (block_idx:
    heads = H_kv, per_row = topk; lse_idx: H_kv, 1; lse: H_q, 1)."""
    cu = cu_seqlens.tolist() if isinstance(cu_seqlens, torch.Tensor) else list(cu_seqlens)
    a, b = cu[s] * heads * per_row, cu[s + 1] * heads * per_row
    return flat[a:b].view(heads, cu[s + 1] - cu[s], per_row)


def msa_index_topk_varlen(q_idx, k_idx, cu_seqlens, topk: int = 16, *, max_seqlen=None, H_q=None,
                          d=None, Bk: int = 128, causal: bool = True, scale_idx=None,
                          with_lse: bool = True):
    """q_idx [T,H_kv,d_idx], k_idx [T,d_idx], cu_seqlens (int32, num_seqs + 1) -> packed
    block_idx (int32, H_kv*T*topk) and lse_idx (f32, H_kv*T) or None."""
    _need(q_idx, "q_idx", ndim=3)
    _need(k_idx, "k_idx", ndim=2)
    T, H_kv, d_idx = q_idx.shape
    if tuple(k_idx.shape) != (T, d_idx):
        raise ValueError("q_idx and k_idx must share the token axis")
    dev = q_idx.device
    cu = _cu_dev(cu_seqlens, dev)
    n = cu.numel() - 1
    prob = make_problem(1, _max_len(cu, max_seqlen), H_q or H_kv, H_kv, d or 128, d_idx, topk, Bk,
                        causal, None, scale_idx)
    block_idx = torch.empty(H_kv * T * topk, dtype=torch.int32, device=dev)
    lse_idx = torch.empty(H_kv * T, dtype=torch.float32, device=dev) if with_lse else None
    nws = _lib.msa_workspace_size_varlen(prob, n, T, _lib.MSA_WS_INDEX)
    ws = _workspace(nws, dev)
    rc = _lib.msa_index_topk_varlen(prob, _ptr(cu), n, T, _ptr(q_idx), _ptr(k_idx),
                                    _ptr(block_idx), _ptr(lse_idx), _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_index_topk_varlen")
    return block_idx, lse_idx


def msa_fwd_varlen(q, k, v, block_idx, cu_seqlens, topk: int, *, max_seqlen=None, scale=None,
                   Bk: int = 128, causal: bool = True, d_idx=64):
    """q [T,H_q,d], k, v [T,H_kv,d], packed block_idx -> o [T,H_q,d], packed lse (H_q*T)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, ndim=3)
    _need(block_idx, "block_idx", torch.int32, ndim=1)
    T, H_q, d = q.shape
    H_kv = k.shape[1]
    if block_idx.numel() != H_kv * T * topk:
        raise ValueError("block_idx must hold H_kv*T*topk entries")
    dev = q.device
    cu = _cu_dev(cu_seqlens, dev)
    n = cu.numel() - 1
    prob = make_problem(1, _max_len(cu, max_seqlen), H_q, H_kv, d, d_idx, topk, Bk, causal, scale,
                        None)
    o = torch.empty_like(q)
    lse = torch.empty(H_q * T, dtype=torch.float32, device=dev)
    nws = _lib.msa_workspace_size_varlen(prob, n, T, _lib.MSA_WS_FWD)
    ws = _workspace(nws, dev)
    rc = _lib.msa_fwd_varlen(prob, _ptr(cu), n, T, _ptr(q), _ptr(k), _ptr(v), _ptr(block_idx),
                             _ptr(o), _ptr(lse), _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_fwd_varlen")
    return o, lse


def msa_bwd_varlen(q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight: float,
                   cu_seqlens, topk: int, *, max_seqlen=None, scale=None, scale_idx=None,
                   Bk: int = 128, causal: bool = True):
    """Fused backward over a packed batch: dict dq, dk, dv, dq_idx, dk_idx and kl (sum over
    every row of every sequence)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dO, "dO"), (q_idx, "q_idx")):
        _need(t, n, ndim=3)
    _need(k_idx, "k_idx", ndim=2)
    _need(lse, "lse", torch.float32, ndim=1)
    _need(lse_idx, "lse_idx", torch.float32, ndim=1)
    _need(block_idx, "block_idx", torch.int32, ndim=1)
    T, H_q, d = q.shape
    H_kv = k.shape[1]
    d_idx = q_idx.shape[2]
    dev = q.device
    cu = _cu_dev(cu_seqlens, dev)
    n = cu.numel() - 1
    prob = make_problem(1, _max_len(cu, max_seqlen), H_q, H_kv, d, d_idx, topk, Bk, causal, scale,
                        scale_idx)
    out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
           "dq_idx": torch.empty_like(q_idx), "dk_idx": torch.empty_like(k_idx),
           "kl": torch.empty(1, dtype=torch.float32, device=dev)}
    nws = _lib.msa_workspace_size_varlen(prob, n, T, _lib.MSA_WS_BWD)
    ws = _workspace(nws, dev)
    rc = _lib.msa_bwd_varlen(prob, _ptr(cu), n, T, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                             _ptr(dO), _ptr(q_idx), _ptr(k_idx), _ptr(block_idx), _ptr(lse_idx),
                             kl_weight, _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
                             _ptr(out["dq_idx"]), _ptr(out["dk_idx"]), _ptr(out["kl"]), _ptr(ws),
                             nws, _stream(dev))
    _lib.check(rc, "msa_bwd_varlen")
    return out


# ---------------------------------------------------------------------------
# Decode: one new token per sequence against its KV cache (see include/msa.h).
# ---------------------------------------------------------------------------
def msa_decode(q, q_idx, k, v, k_idx, lens, topk: int = 16, *, scale=None, Bk: int = 128):
    """q [B,H_q,d], q_idx [B,H_kv,d_idx] (new token); k, v [B,Lmax,H_kv,d] and
    k_idx [B,Lmax,d_idx] (caches); lens int32 [B] on the device (cache lengths including
    the new token).  Returns (block_idx [B,H_kv,topk] int32, o [B,H_q,d] bf16,
    lse [B,H_q] f32)."""
    _need(q, "q", ndim=3)
    _need(q_idx, "q_idx", ndim=3)
    _need(k, "k", ndim=4)
    _need(v, "v", ndim=4)
    _need(k_idx, "k_idx", ndim=3)
    _need(lens, "lens", torch.int32, ndim=1)
    B, H_q, d = q.shape
    _, Lmax, H_kv, _ = k.shape
    d_idx = q_idx.shape[2]
    if tuple(v.shape) != tuple(k.shape) or tuple(k_idx.shape) != (B, Lmax, d_idx) or lens.numel() != B:
        raise ValueError("cache shapes must agree: k, v [B,Lmax,H_kv,d], k_idx [B,Lmax,d_idx], lens [B]")
    prob = make_problem(B, Lmax, H_q, H_kv, d, d_idx, topk, Bk, True, scale, None)
    dev = q.device
    block_idx = torch.empty((B, H_kv, topk), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    nws = _lib.msa_decode_workspace_size(prob)
    ws = _workspace(nws, dev)
    rc = _lib.msa_decode(prob, _ptr(q), _ptr(q_idx), _ptr(k), _ptr(v), _ptr(k_idx), _ptr(lens),
                         _ptr(block_idx), _ptr(o), _ptr(lse), _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_decode")
    return block_idx, o, lse


def msa_quantize_kv_fp8(x, *, Bk: int = 128):
    """x [B,Lmax,H_kv,d] bf16 (a k or v cache) -> (codes [B,Lmax,H_kv,d] uint8 E4M3,
    scale [B,Lmax,H_kv] f32): one scale amax/448 per (sequence, token, head) row."""
    _need(x, "x", ndim=4)
    B, Lmax, H_kv, d = x.shape
    prob = make_problem(B, Lmax, H_kv, H_kv, d, 64, 1, Bk, True, None, None)
    x8 = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scale = torch.empty((B, Lmax, H_kv), dtype=torch.float32, device=x.device)
    rc = _lib.msa_quantize_kv_fp8(prob, _ptr(x), _ptr(x8), _ptr(scale), _stream(x.device))
    _lib.check(rc, "msa_quantize_kv_fp8")
    return x8, scale


def msa_decode_fp8(q, q_idx, k8, v8, k_scale, v_scale, k_idx, lens, topk: int = 16, *,
                   scale=None, Bk: int = 128):
    """msa_decode over an FP8 cache: k8, v8 [B,Lmax,H_kv,d] uint8 codes and k_scale,
    v_scale [B,Lmax,H_kv] f32 from msa_quantize_kv_fp8.  Returns (block_idx [B,H_kv,topk]
    int32, o [B,H_q,d] bf16, lse [B,H_q] f32)."""
    _need(q, "q", ndim=3)
    _need(q_idx, "q_idx", ndim=3)
    _need(k8, "k8", torch.uint8, ndim=4)
    _need(v8, "v8", torch.uint8, ndim=4)
    _need(k_scale, "k_scale", torch.float32, ndim=3)
    _need(v_scale, "v_scale", torch.float32, ndim=3)
    _need(k_idx, "k_idx", ndim=3)
    _need(lens, "lens", torch.int32, ndim=1)
    B, H_q, d = q.shape
    _, Lmax, H_kv, _ = k8.shape
    d_idx = q_idx.shape[2]
    if (tuple(v8.shape) != tuple(k8.shape) or tuple(k_scale.shape) != (B, Lmax, H_kv)
            or tuple(v_scale.shape) != (B, Lmax, H_kv) or tuple(k_idx.shape) != (B, Lmax, d_idx)
            or lens.numel() != B):
        raise ValueError("cache shapes must agree: k8, v8 [B,Lmax,H_kv,d], scales [B,Lmax,H_kv], "
                         "k_idx [B,Lmax,d_idx], lens [B]")
    prob = make_problem(B, Lmax, H_q, H_kv, d, d_idx, topk, Bk, True, scale, None)
    dev = q.device
    block_idx = torch.empty((B, H_kv, topk), dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    nws = _lib.msa_decode_workspace_size(prob)
    ws = _workspace(nws, dev)
    rc = _lib.msa_decode_fp8(prob, _ptr(q), _ptr(q_idx), _ptr(k8), _ptr(v8), _ptr(k_scale),
                             _ptr(v_scale), _ptr(k_idx), _ptr(lens), _ptr(block_idx), _ptr(o),
                             _ptr(lse), _ptr(ws), nws, _stream(dev))
    _lib.check(rc, "msa_decode_fp8")
    return block_idx, o, lse


# ---------------------------------------------------------------------------
# FP8 (E4M3) main-branch forward for training (d = 128); see include/msa.h.
# ---------------------------------------------------------------------------
def msa_quantize_fwd_fp8(q, k, v, *, Bk: int = 128):
    """bf16 q [B,N,H_q,d], k, v [B,N,H_kv,d] -> the FP8 forward's operands:
    q8 [B,N,H_q,d] uint8 + q_scale [B,N,H_q] (one scale per row), k8 [B,N,H_kv,d] +
    k_scale [B,H_kv,nb] and v8t [B,H_kv,nb,d,Bk] (v transposed per block) + v_scale
    [B,H_kv,nb] (one scale per Bk-key block)."""
    _need(q, "q", ndim=4)
    _need(k, "k", ndim=4)
    _need(v, "v", ndim=4)
    B, N, H_q, d = q.shape
    H_kv = k.shape[2]
    if tuple(k.shape) != (B, N, H_kv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k, v must be [B, N, H_kv, d] with q's B, N, d")
    nb = (N + Bk - 1) // Bk
    prob = make_problem(B, N, H_q, H_kv, d, 64, 1, Bk, True, None, None)
    dev = q.device
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=dev)
    q_scale = torch.empty((B, N, H_q), dtype=torch.float32, device=dev)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=dev)
    k_scale = torch.empty((B, H_kv, nb), dtype=torch.float32, device=dev)
    v8t = torch.empty((B, H_kv, nb, d, Bk), dtype=torch.uint8, device=dev)
    v_scale = torch.empty((B, H_kv, nb), dtype=torch.float32, device=dev)
    rc = _lib.msa_quantize_fwd_fp8(prob, _ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(q_scale),
                                   _ptr(k8), _ptr(k_scale), _ptr(v8t), _ptr(v_scale), _stream(dev))
    _lib.check(rc, "msa_quantize_fwd_fp8")
    return q8, q_scale, k8, k_scale, v8t, v_scale


def msa_fwd_fp8(q8, q_scale, k8, k_scale, v8t, v_scale, block_idx, *, scale=None, Bk: int = 128,
                d_idx: int = 64):
    """FP8 forward over the operands of msa_quantize_fwd_fp8 and the block sets
    block_idx [B,H_kv,N,topk]: returns (o [B,N,H_q,d] bf16, lse [B,H_q,N] f32)."""
    _need(q8, "q8", torch.uint8, ndim=4)
    _need(k8, "k8", torch.uint8, ndim=4)
    _need(v8t, "v8t", torch.uint8, ndim=5)
    _need(q_scale, "q_scale", torch.float32, ndim=3)
    _need(k_scale, "k_scale", torch.float32, ndim=3)
    _need(v_scale, "v_scale", torch.float32, ndim=3)
    _need(block_idx, "block_idx", torch.int32, ndim=4)
    B, N, H_q, d = q8.shape
    H_kv = k8.shape[2]
    topk = block_idx.shape[3]
    nb = (N + Bk - 1) // Bk
    if (tuple(k8.shape) != (B, N, H_kv, d) or tuple(v8t.shape) != (B, H_kv, nb, d, Bk)
            or tuple(q_scale.shape) != (B, N, H_q) or tuple(k_scale.shape) != (B, H_kv, nb)
            or tuple(v_scale.shape) != (B, H_kv, nb) or tuple(block_idx.shape[:3]) != (B, H_kv, N)):
        raise ValueError("operand shapes must be those of msa_quantize_fwd_fp8")
    prob = make_problem(B, N, H_q, H_kv, d, d_idx, topk, Bk, True, scale, None)
    dev = q8.device
    o = torch.empty((B, N, H_q, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H_q, N), dtype=torch.float32, device=dev)
    nws = _lib.msa_workspace_size(prob, _lib.MSA_WS_FWD)
    ws = _workspace(nws, dev)
    rc = _lib.msa_fwd_fp8(prob, _ptr(q8), _ptr(q_scale), _ptr(k8), _ptr(k_scale), _ptr(v8t),
                          _ptr(v_scale), _ptr(block_idx), _ptr(o), _ptr(lse), _ptr(ws), nws,
                          _stream(dev))
    _lib.check(rc, "msa_fwd_fp8")
    return o, lse
