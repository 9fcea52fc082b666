"""ctypes binding of libmsa.so, the C ABI declared in include/msa.h.

Names match the C entry points.  Marshalling only: pointers, sizes and the
stream handle go through unchanged; every step of the computation runs in the
library's CUDA kernels.  Loading fails loudly if the library was not built.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

MSA_OK = 0
MSA_ERR_ARG = -1
MSA_ERR_SHAPE = -2
MSA_ERR_UNSUPPORTED = -3
MSA_ERR_WORKSPACE = -4
MSA_ERR_CUDA = -5
MSA_ERR_DEVICE_TIMEOUT = -6

MSA_WS_INDEX = 0
MSA_WS_FWD = 1
MSA_WS_BWD = 2

# every symbol include/msa.h declares
EXPORTS = ("msa_workspace_size", "msa_index_topk", "msa_fwd", "msa_bwd",
           "msa_get_device_status", "msa_status_string", "msa_debug_set",
           "msa_set_kernel_events", "msa_kernel_launch_count", "msa_index_topk_noalloc",
           "msa_noalloc_scratch_bytes", "msa_version", "msa_workspace_size_varlen",
           "msa_index_topk_varlen", "msa_fwd_varlen", "msa_bwd_varlen",
           "msa_decode_workspace_size", "msa_decode", "msa_quantize_kv_fp8",
           "msa_decode_fp8", "msa_quantize_fwd_fp8", "msa_fwd_fp8", "msa_plan_size",
           "msa_index_topk_plan", "msa_fwd_plan", "msa_bwd_plan")

MSA_KERNEL_INDEX = 0
MSA_KERNEL_FWD = 1
MSA_KERNEL_BWD = 2
MSA_KERNEL_INDEX_LSE = 3

MSA_DEBUG_WITHHOLD_LOAD = 1


class Problem(ctypes.Structure):
    """msa_problem_t"""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "N", "H_q", "H_kv", "d", "d_idx", "Bk", "topk", "causal")] + \
               [("scale", ctypes.c_float), ("scale_idx", ctypes.c_float)]


class MSAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    vp, sz, i32, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float
    P = ctypes.POINTER(Problem)
    lib.msa_workspace_size.argtypes = [P, i32]
    lib.msa_workspace_size.restype = sz
    lib.msa_index_topk.argtypes = [P, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_index_topk.restype = i32
    lib.msa_fwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_fwd.restype = i32
    lib.msa_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp,
                            vp, vp, sz, vp]
    lib.msa_bwd.restype = i32
    lib.msa_plan_size.argtypes = [P]
    lib.msa_plan_size.restype = sz
    lib.msa_index_topk_plan.argtypes = [P, vp, vp, vp, vp, vp, sz, vp, sz, vp]
    lib.msa_index_topk_plan.restype = i32
    lib.msa_fwd_plan.argtypes = [P, vp, vp, vp, vp, vp, sz, vp, vp, vp, sz, vp]
    lib.msa_fwd_plan.restype = i32
    lib.msa_bwd_plan.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, f32, vp, vp,
                                 vp, vp, vp, vp, vp, sz, vp]
    lib.msa_bwd_plan.restype = i32
    lib.msa_get_device_status.argtypes = [vp, ctypes.POINTER(i32)]
    lib.msa_get_device_status.restype = i32
    lib.msa_status_string.argtypes = [i32]
    lib.msa_status_string.restype = ctypes.c_char_p
    lib.msa_debug_set.argtypes = [ctypes.c_uint64, i32]
    lib.msa_debug_set.restype = i32
    lib.msa_set_kernel_events.argtypes = [i32, vp, vp]
    lib.msa_set_kernel_events.restype = i32
    lib.msa_kernel_launch_count.argtypes = []
    lib.msa_kernel_launch_count.restype = ctypes.c_uint64
    lib.msa_index_topk_noalloc.argtypes = [P, vp, vp, vp, vp, vp]
    lib.msa_index_topk_noalloc.restype = i32
    lib.msa_noalloc_scratch_bytes.argtypes = []
    lib.msa_noalloc_scratch_bytes.restype = sz
    lib.msa_version.argtypes = []
    lib.msa_version.restype = i32
    lib.msa_workspace_size_varlen.argtypes = [P, i32, i32, i32]
    lib.msa_workspace_size_varlen.restype = sz
    lib.msa_index_topk_varlen.argtypes = [P, vp, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_index_topk_varlen.restype = i32
    lib.msa_fwd_varlen.argtypes = [P, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_fwd_varlen.restype = i32
    lib.msa_bwd_varlen.argtypes = [P, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, f32, vp,
                                   vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_bwd_varlen.restype = i32
    lib.msa_decode_workspace_size.argtypes = [P]
    lib.msa_decode_workspace_size.restype = sz
    lib.msa_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_decode.restype = i32
    lib.msa_quantize_kv_fp8.argtypes = [P, vp, vp, vp, vp]
    lib.msa_quantize_kv_fp8.restype = i32
    lib.msa_decode_fp8.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_decode_fp8.restype = i32
    lib.msa_quantize_fwd_fp8.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.msa_quantize_fwd_fp8.restype = i32
    lib.msa_fwd_fp8.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.msa_fwd_fp8.restype = i32
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().msa_status_string(int(code)).decode()


def check(code: int, where: str) -> None:
    if code != MSA_OK:
        raise MSAError(code, where)


def msa_workspace_size(prob: Problem, which: int) -> int:
    return int(load().msa_workspace_size(ctypes.byref(prob), which))


def msa_index_topk(prob, q_idx, k_idx, block_idx, lse_idx, ws, ws_bytes, stream) -> int:
    return load().msa_index_topk(ctypes.byref(prob), q_idx, k_idx, block_idx, lse_idx, ws,
                                 ws_bytes, stream)


def msa_fwd(prob, q, k, v, block_idx, o, lse, ws, ws_bytes, stream) -> int:
    return load().msa_fwd(ctypes.byref(prob), q, k, v, block_idx, o, lse, ws, ws_bytes, stream)


def msa_bwd(prob, q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, kl_weight, dq, dk, dv,
            dq_idx, dk_idx, kl_out, ws, ws_bytes, stream) -> int:
    return load().msa_bwd(ctypes.byref(prob), q, k, v, o, lse, dO, q_idx, k_idx, block_idx,
                          lse_idx, float(kl_weight), dq, dk, dv, dq_idx, dk_idx, kl_out, ws,
                          ws_bytes, stream)


def msa_plan_size(prob) -> int:
    return int(load().msa_plan_size(ctypes.byref(prob)))


def msa_index_topk_plan(prob, q_idx, k_idx, block_idx, lse_idx, plan, plan_bytes, ws, ws_bytes,
                        stream) -> int:
    return load().msa_index_topk_plan(ctypes.byref(prob), q_idx, k_idx, block_idx, lse_idx, plan,
                                      plan_bytes, ws, ws_bytes, stream)


def msa_fwd_plan(prob, q, k, v, block_idx, plan, plan_bytes, o, lse, ws, ws_bytes, stream) -> int:
    return load().msa_fwd_plan(ctypes.byref(prob), q, k, v, block_idx, plan, plan_bytes, o, lse,
                               ws, ws_bytes, stream)


def msa_bwd_plan(prob, q, k, v, o, lse, dO, q_idx, k_idx, block_idx, lse_idx, plan, plan_bytes,
                 kl_weight, dq, dk, dv, dq_idx, dk_idx, kl_out, ws, ws_bytes, stream) -> int:
    return load().msa_bwd_plan(ctypes.byref(prob), q, k, v, o, lse, dO, q_idx, k_idx, block_idx,
                               lse_idx, plan, plan_bytes, float(kl_weight), dq, dk, dv, dq_idx,
                               dk_idx, kl_out, ws, ws_bytes, stream)


def msa_index_topk_noalloc(prob, q_idx, k_idx, block_idx, lse_idx, stream) -> int:
    """msa_index_topk with the library's built-in scratch instead of a workspace."""
    return load().msa_index_topk_noalloc(ctypes.byref(prob), q_idx, k_idx, block_idx, lse_idx,
                                         stream)


def msa_noalloc_scratch_bytes() -> int:
    return int(load().msa_noalloc_scratch_bytes())


def msa_get_device_status(stream) -> int:
    st = ctypes.c_int(0)
    check(load().msa_get_device_status(stream, ctypes.byref(st)), "msa_get_device_status")
    return st.value


def msa_debug_set(wait_limit_ns: int, flags: int) -> int:
    return load().msa_debug_set(int(wait_limit_ns), int(flags))


def msa_set_kernel_events(kernel: int, start, stop) -> int:
    """start/stop: cudaEvent_t handles (torch.cuda.Event().cuda_event) or None."""
    return load().msa_set_kernel_events(int(kernel), start, stop)


def msa_kernel_launch_count() -> int:
    return int(load().msa_kernel_launch_count())


def msa_workspace_size_varlen(prob: Problem, num_seqs: int, total_tokens: int, which: int) -> int:
    return int(load().msa_workspace_size_varlen(ctypes.byref(prob), num_seqs, total_tokens, which))


def msa_index_topk_varlen(prob, cu_seqlens, num_seqs, total_tokens, q_idx, k_idx, block_idx,
                          lse_idx, ws, ws_bytes, stream) -> int:
    """cu_seqlens: device pointer to num_seqs + 1 int32."""
    return load().msa_index_topk_varlen(ctypes.byref(prob), cu_seqlens, num_seqs, total_tokens,
                                        q_idx, k_idx, block_idx, lse_idx, ws, ws_bytes, stream)


def msa_fwd_varlen(prob, cu_seqlens, num_seqs, total_tokens, q, k, v, block_idx, o, lse, ws,
                   ws_bytes, stream) -> int:
    return load().msa_fwd_varlen(ctypes.byref(prob), cu_seqlens, num_seqs, total_tokens, q, k, v,
                                 block_idx, o, lse, ws, ws_bytes, stream)


def msa_bwd_varlen(prob, cu_seqlens, num_seqs, total_tokens, q, k, v, o, lse, dO, q_idx, k_idx,
                   block_idx, lse_idx, kl_weight, dq, dk, dv, dq_idx, dk_idx, kl_out, ws, ws_bytes,
                   stream) -> int:
    return load().msa_bwd_varlen(ctypes.byref(prob), cu_seqlens, num_seqs, total_tokens, q, k, v, o,
                                 lse, dO, q_idx, k_idx, block_idx, lse_idx, float(kl_weight), dq, dk,
                                 dv, dq_idx, dk_idx, kl_out, ws, ws_bytes, stream)


def msa_decode_workspace_size(prob: Problem) -> int:
    return int(load().msa_decode_workspace_size(ctypes.byref(prob)))


def msa_decode(prob, q, q_idx, k, v, k_idx, lens, block_idx, o, lse, ws, ws_bytes, stream) -> int:
    return load().msa_decode(ctypes.byref(prob), q, q_idx, k, v, k_idx, lens, block_idx, o, lse,
                             ws, ws_bytes, stream)


def msa_quantize_kv_fp8(prob, x, x8, scale, stream) -> int:
    return load().msa_quantize_kv_fp8(ctypes.byref(prob), x, x8, scale, stream)


def msa_decode_fp8(prob, q, q_idx, k8, v8, k_scale, v_scale, k_idx, lens, block_idx, o, lse, ws,
                   ws_bytes, stream) -> int:
    return load().msa_decode_fp8(ctypes.byref(prob), q, q_idx, k8, v8, k_scale, v_scale, k_idx,
                                 lens, block_idx, o, lse, ws, ws_bytes, stream)


def msa_quantize_fwd_fp8(prob, q, k, v, q8, q_scale, k8, k_scale, v8t, v_scale, stream) -> int:
    return load().msa_quantize_fwd_fp8(ctypes.byref(prob), q, k, v, q8, q_scale, k8, k_scale, v8t,
                                       v_scale, stream)


def msa_fwd_fp8(prob, q8, q_scale, k8, k_scale, v8t, v_scale, block_idx, o, lse, ws, ws_bytes,
                stream) -> int:
    return load().msa_fwd_fp8(ctypes.byref(prob), q8, q_scale, k8, k_scale, v8t, v_scale, block_idx,
                              o, lse, ws, ws_bytes, stream)


def msa_version() -> int:
    return load().msa_version()
