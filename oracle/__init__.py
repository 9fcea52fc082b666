"""float64 CPU oracle of the MSA training hot path (ctypes wrapper of msa_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check and by
the CPU-baseline leg of the benchmark.  The library under
block_sparse_gqa_topk_gb300/ never imports it; the two share no code.

fp8.py holds the FP8 (E4M3) KV-cache quantiser and the decode attention over the
dequantised cache (numpy).

All arrays in and out are numpy.  Inputs are bf16 bit patterns (uint16) from
block_sparse_gqa_topk_gb300.synth; outputs are float64 (int32 for block ids).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


class _Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "N", "H_q", "H_kv", "d", "d_idx", "Bk", "topk", "causal")] + \
               [("scale", ctypes.c_double), ("scale_idx", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11, -O2, IEEE arithmetic)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def load(path=None):
    """Load the oracle library (the built one by default); returns the ctypes handle."""
    global _lib
    lib = ctypes.CDLL(path or build())
    _declare(lib)
    _lib = lib
    return lib


def _get():
    if _lib is None:
        load()
    return _lib


def _declare(lib):
    P = ctypes.POINTER
    vp = ctypes.c_void_p
    lib.oracle_select.argtypes = [P(_Problem), vp, vp, vp, ctypes.c_int64, vp, vp, vp,
                                  ctypes.c_int]
    lib.oracle_forward.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp,
                                   vp, vp, vp, ctypes.c_int]
    lib.oracle_backward.argtypes = [P(_Problem), vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64,
                                    vp, ctypes.c_double, vp, vp, vp, vp, vp, vp, vp,
                                    ctypes.c_int]
    for f in (lib.oracle_select, lib.oracle_forward, lib.oracle_backward):
        f.restype = ctypes.c_int


def problem(cfg, **over) -> _Problem:
    """Build the C problem struct from an MSAConfig (fields may be overridden)."""
    f = {n: getattr(cfg, n) for n in ("B", "N", "H_q", "H_kv", "d", "d_idx", "Bk", "topk")}
    f["causal"] = int(bool(cfg.causal))
    f["scale"] = cfg.scale
    f["scale_idx"] = cfg.scale_idx
    f.update(over)
    return _Problem(**f)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(rows):
    if rows is None:
        return None, None
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    return rows, len(rows)


def _u16(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.uint16)


def select(cfg, inputs, rows=None, pooled=False, n_threads=0, **over):
    """Block sets: (block_idx [R,H_kv,topk] int32, kth [R,H_kv,2], pooled [R,H_kv,nb]|None)."""
    p = problem(cfg, **over)
    rows, R = _rows(rows)
    if R is None:
        R = p.B * p.N
    nb = (p.N + p.Bk - 1) // p.Bk
    bi = np.empty((R, p.H_kv, p.topk), dtype=np.int32)
    kth = np.empty((R, p.H_kv, 2), dtype=np.float64)
    pl = np.empty((R, p.H_kv, nb), dtype=np.float64) if pooled else None
    qi, ki = _u16(inputs["q_idx"]), _u16(inputs["k_idx"])
    rc = _get().oracle_select(ctypes.byref(p), _ptr(qi), _ptr(ki), _ptr(rows), R, _ptr(bi),
                              _ptr(kth), _ptr(pl), n_threads)
    if rc:
        raise RuntimeError(f"oracle_select failed ({rc})")
    return bi, kth, pl


def forward(cfg, inputs, block_idx, rows=None, n_threads=0, main=True, index=True, **over):
    """(o [R,H_q,d], lse [R,H_q], lse_idx [R,H_kv]) over the given block sets; main=False
    skips o/lse (None), index=False skips lse_idx (None)."""
    p = problem(cfg, **over)
    rows, R = _rows(rows)
    if R is None:
        R = p.B * p.N
    o = np.empty((R, p.H_q, p.d)) if main else None
    lse = np.empty((R, p.H_q)) if main else None
    lse_idx = np.empty((R, p.H_kv)) if index else None
    bi = np.ascontiguousarray(block_idx, dtype=np.int32).reshape(R, p.H_kv, p.topk)
    want = (("q", "k", "v") if main else ()) + (("q_idx", "k_idx") if index else ())
    ins = [_u16(inputs[n]) if n in want else None for n in ("q", "k", "v", "q_idx", "k_idx")]
    rc = _get().oracle_forward(ctypes.byref(p), *[_ptr(a) for a in ins], _ptr(rows), R,
                               _ptr(bi), _ptr(o), _ptr(lse), _ptr(lse_idx), n_threads)
    if rc:
        raise RuntimeError(f"oracle_forward failed ({rc})")
    return o, lse, lse_idx


def backward(cfg, inputs, block_idx, kl_weight, rows=None, n_threads=0, **over):
    """Gradients of the listed rows (see msa_oracle.c, oracle_backward)."""
    p = problem(cfg, **over)
    rows, R = _rows(rows)
    if R is None:
        R = p.B * p.N
    out = {
        "dq": np.empty((R, p.H_q, p.d)),
        "dk": np.empty((p.B, p.N, p.H_kv, p.d)),
        "dv": np.empty((p.B, p.N, p.H_kv, p.d)),
        "dq_idx": np.empty((R, p.H_kv, p.d_idx)),
        "dk_idx": np.empty((p.B, p.N, p.d_idx)),
        "kl_rows": np.empty((R, p.H_kv)),
    }
    kl = ctypes.c_double(0.0)
    bi = np.ascontiguousarray(block_idx, dtype=np.int32).reshape(R, p.H_kv, p.topk)
    ins = [_u16(inputs[n]) for n in ("q", "k", "v", "q_idx", "k_idx", "dO")]
    rc = _get().oracle_backward(ctypes.byref(p), *[_ptr(a) for a in ins], _ptr(rows), R,
                                _ptr(bi), float(kl_weight), _ptr(out["dq"]), _ptr(out["dk"]),
                                _ptr(out["dv"]), _ptr(out["dq_idx"]), _ptr(out["dk_idx"]),
                                _ptr(out["kl_rows"]), ctypes.byref(kl), n_threads)
    if rc:
        raise RuntimeError(f"oracle_backward failed ({rc})")
    out["kl"] = kl.value
    return out
