"""The C ABI library on the CPU: it loads, exports every entry point that
include/msa.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from block_sparse_gqa_topk_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("msa_index_topk", "msa_fwd", "msa_bwd", "msa_workspace_size"):
        assert want in names
    assert set(names) == set(_lib.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def _prob(**kw):
    base = dict(B=1, N=2048, H_q=8, H_kv=2, d=64, d_idx=32, Bk=128, topk=4, causal=1, scale=0.125,
                scale_idx=0.0)
    base.update(kw)
    return _lib.Problem(**base)


def test_status_strings_and_version():
    for code in range(0, -7, -1):
        assert _lib.status_string(code)
    assert "unknown" in _lib.status_string(-99)
    assert _lib.msa_version() >= 10000


@pytest.mark.parametrize("kw,code", [
    (dict(H_q=6, H_kv=4), _lib.MSA_ERR_SHAPE),
    (dict(N=-1), _lib.MSA_ERR_SHAPE),
    (dict(topk=0), _lib.MSA_ERR_SHAPE),
    (dict(Bk=64), _lib.MSA_ERR_UNSUPPORTED),
    (dict(d=96), _lib.MSA_ERR_UNSUPPORTED),
    (dict(d_idx=16), _lib.MSA_ERR_UNSUPPORTED),
    (dict(topk=257), _lib.MSA_ERR_UNSUPPORTED),
    (dict(N=(1 << 23) + 1), _lib.MSA_ERR_UNSUPPORTED),
    (dict(causal=0), _lib.MSA_ERR_UNSUPPORTED),
    (dict(scale=0.0), _lib.MSA_ERR_ARG),
    (dict(scale=float("nan")), _lib.MSA_ERR_ARG),
])
def test_bad_problems_are_rejected_on_the_host(kw, code):
    p = _prob(**kw)
    assert _lib.msa_workspace_size(p, _lib.MSA_WS_FWD) == 0
    assert _lib.msa_index_topk(p, 16, 16, 16, None, None, 0, None) == code
    assert _lib.msa_fwd(p, 16, 16, 16, 16, 16, 16, None, 0, None) == code


def test_more_than_32_slots_only_for_the_dense_set():
    # selection keeps at most 32 blocks: topk = 33 < nb = 64 is refused by the index
    # entry point on the host, while the forward accepts any caller-given set
    p = _prob(N=8192, topk=33)
    assert _lib.msa_index_topk(p, 16, 16, 16, None, None, 0, None) == _lib.MSA_ERR_UNSUPPORTED
    assert _lib.msa_workspace_size(p, _lib.MSA_WS_FWD) > 0
    # topk >= nb (every visible block): a valid problem for every entry point
    p = _prob(N=8192, topk=64)
    for which in (_lib.MSA_WS_INDEX, _lib.MSA_WS_FWD, _lib.MSA_WS_BWD):
        assert _lib.msa_workspace_size(p, which) > 0


def test_null_and_misaligned_pointers_are_rejected():
    p = _prob()
    assert _lib.msa_index_topk(p, None, 16, 16, None, None, 0, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_index_topk(p, 18, 16, 16, None, None, 0, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_fwd(p, 16, 16, 16, 16, 16, 16, None, 0, None) == _lib.MSA_ERR_WORKSPACE
    assert _lib.msa_fwd(p, 16, 16, None, 16, 16, 16, 256, 1 << 40, None) == _lib.MSA_ERR_ARG
    small = _lib.msa_workspace_size(p, _lib.MSA_WS_FWD) - 1
    assert _lib.msa_fwd(p, 16, 16, 16, 16, 16, 16, 256, small, None) == _lib.MSA_ERR_WORKSPACE


def test_decode_and_fp8_entry_points_reject_bad_arguments_on_the_host():
    p = _prob()
    ws = _lib.msa_decode_workspace_size(p)
    assert ws > 0
    # decode: null / misaligned pointers, missing FP8 scales, too many slots to select
    assert _lib.msa_decode(p, None, 16, 16, 16, 16, 16, 16, 16, 16, 256, ws, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_decode(p, 16, 16, 24, 16, 16, 16, 16, 16, 16, 256, ws, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_decode_fp8(p, 16, 16, 16, 16, None, 16, 16, 16, 16, 16, 16, 256, ws,
                               None) == _lib.MSA_ERR_ARG
    assert _lib.msa_decode(_prob(topk=40), 16, 16, 16, 16, 16, 16, 16, 16, 16, 256, 1 << 30,
                           None) == _lib.MSA_ERR_UNSUPPORTED
    # quantiser: only the cache sizes matter; d must be 64 or 128, pointers aligned
    assert _lib.msa_quantize_kv_fp8(_prob(d=96), 16, 16, 16, None) == _lib.MSA_ERR_UNSUPPORTED
    assert _lib.msa_quantize_kv_fp8(p, 16, None, 16, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_quantize_kv_fp8(p, 16, 20, 16, None) == _lib.MSA_ERR_ARG
    assert _lib.msa_quantize_kv_fp8(_prob(N=0), None, None, None, None) == _lib.MSA_OK
    assert _lib.msa_quantize_kv_fp8(_prob(H_kv=0, H_q=0), 16, 16, 16, None) == _lib.MSA_ERR_SHAPE


def test_varlen_arguments_are_checked_on_the_host():
    # cu_seqlens lives on the device and is checked there; the host checks what it is
    # given: sizes, pointers and the workspace.  p.N is the batch's max_seqlen.
    p = _prob(N=4096)
    assert _lib.msa_workspace_size_varlen(p, -1, 100, _lib.MSA_WS_FWD) == 0
    assert _lib.msa_workspace_size_varlen(p, 2, -5, _lib.MSA_WS_FWD) == 0
    assert _lib.msa_workspace_size_varlen(p, 2, 100, 7) == 0
    assert _lib.msa_workspace_size_varlen(_prob(N=(1 << 21) + 128), 1, 100, _lib.MSA_WS_FWD) == 0
    # the workspace grows with the packed tokens, not with num_seqs x max_seqlen
    for which in (_lib.MSA_WS_INDEX, _lib.MSA_WS_FWD, _lib.MSA_WS_BWD):
        packed = _lib.msa_workspace_size_varlen(p, 8, 8192, which)
        fixed = _lib.msa_workspace_size(_prob(B=2, N=4096), which)
        assert packed > 0 and packed < fixed + (1 << 20)
        assert _lib.msa_workspace_size_varlen(p, 8, 16384, which) > packed
    # empty batches are no-ops; a null or misaligned cu_seqlens is refused
    assert _lib.msa_index_topk_varlen(p, None, 0, 100, None, None, None, None, None, 0, None) == \
        _lib.MSA_OK
    assert _lib.msa_fwd_varlen(p, None, 2, 0, None, None, None, None, None, None, None, 0,
                               None) == _lib.MSA_OK
    assert _lib.msa_index_topk_varlen(p, None, 2, 100, 16, 16, 16, None, 256, 1 << 20, None) == \
        _lib.MSA_ERR_ARG
    assert _lib.msa_index_topk_varlen(p, 18, 2, 100, 16, 16, 16, None, 256, 1 << 20, None) == \
        _lib.MSA_ERR_ARG
    # the index call needs the workspace head even without lse_idx
    assert _lib.msa_index_topk_varlen(p, 16, 2, 100, 16, 16, 16, None, None, 0, None) == \
        _lib.MSA_ERR_WORKSPACE
    assert _lib.msa_fwd_varlen(p, 16, 2, 100, 16, 16, 16, 16, 16, 16, 256, 16, None) == \
        _lib.MSA_ERR_WORKSPACE
    assert _lib.msa_fwd_varlen(p, 16, 2, 100, 16, 16, 16, 16, 16, 16, 128, 1 << 30, None) == \
        _lib.MSA_ERR_ARG  # workspace not 256-byte aligned


def test_plan_arguments_are_checked_on_the_host():
    # the shared plan's size grows with the problem; a null, short or misaligned plan
    # buffer is refused before anything is queued (its contents are checked on the device)
    small, big = _prob(N=1024), _prob(N=4096)
    assert _lib.msa_plan_size(small) > 0
    assert _lib.msa_plan_size(big) > _lib.msa_plan_size(small)
    assert _lib.msa_plan_size(_prob(N=1024, H_q=24, H_kv=16)) == 0  # H_q % H_kv != 0
    n = _lib.msa_plan_size(small)
    ws = 1 << 34
    assert _lib.msa_index_topk_plan(small, 16, 16, 16, None, None, n, None, 0, None) == \
        _lib.MSA_ERR_ARG
    assert _lib.msa_index_topk_plan(small, 16, 16, 16, None, 256, n - 1, None, 0, None) == \
        _lib.MSA_ERR_WORKSPACE
    assert _lib.msa_index_topk_plan(small, 16, 16, 16, None, 128, n, None, 0, None) == \
        _lib.MSA_ERR_ARG  # not 256-byte aligned
    assert _lib.msa_fwd_plan(small, 16, 16, 16, 16, None, n, 16, 16, 256, ws, None) == \
        _lib.MSA_ERR_ARG
    assert _lib.msa_fwd_plan(small, 16, 16, 16, 16, 256, n - 256, 16, 16, 256, ws, None) == \
        _lib.MSA_ERR_WORKSPACE
    args = [16] * 10
    assert _lib.msa_bwd_plan(small, *args, None, n, 1.0, 16, 16, 16, 16, 16, None, 256, ws,
                             None) == _lib.MSA_ERR_ARG
    assert _lib.msa_bwd_plan(small, *args, 256, 16, 1.0, 16, 16, 16, 16, 16, None, 256, ws,
                             None) == _lib.MSA_ERR_WORKSPACE
    # empty problems are no-ops with or without a plan
    p0 = _prob(N=0)
    assert _lib.msa_index_topk_plan(p0, None, None, None, None, None, 0, None, 0, None) == \
        _lib.MSA_OK
    assert _lib.msa_fwd_plan(p0, None, None, None, None, None, 0, None, None, None, 0, None) == \
        _lib.MSA_OK


def test_empty_problem_is_a_no_op():
    p = _prob(N=0)
    assert _lib.msa_index_topk(p, None, None, None, None, None, 0, None) == _lib.MSA_OK
    assert _lib.msa_fwd(p, None, None, None, None, None, None, None, 0, None) == _lib.MSA_OK


def test_workspace_sizes_grow_with_the_problem():
    a = [_lib.msa_workspace_size(_prob(N=n), w) for n in (1024, 4096) for w in range(3)]
    assert all(x > 0 for x in a)
    assert a[3] > a[0] and a[4] > a[1] and a[5] > a[2]


def test_product_code_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "block_sparse_gqa_topk_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "liboracle" not in text and "msa_oracle" not in text, f


def test_fp8_forward_entry_points_check_arguments_on_the_host():
    """The FP8 training forward takes d = 128 only and rejects null or misaligned
    pointers before anything is enqueued."""
    lib = _lib.load()
    p64 = _prob()  # d = 64
    p128 = _prob(d=128, d_idx=64)
    z = None
    assert lib.msa_quantize_fwd_fp8(ctypes.byref(p64), 256, 256, 256, 256, 256, 256, 256, 256,
                                    256, None) == _lib.MSA_ERR_UNSUPPORTED
    assert lib.msa_quantize_fwd_fp8(ctypes.byref(p128), z, 256, 256, 256, 256, 256, 256, 256,
                                    256, None) == _lib.MSA_ERR_ARG
    assert lib.msa_fwd_fp8(ctypes.byref(p64), 256, 256, 256, 256, 256, 256, 256, 256, 256, 256,
                           1 << 20, None) == _lib.MSA_ERR_UNSUPPORTED
    assert lib.msa_fwd_fp8(ctypes.byref(p128), 256, 256, 264, 256, 256, 256, 256, 256, 256, 256,
                           1 << 20, None) == _lib.MSA_ERR_ARG  # k8 not 16-byte aligned
    assert lib.msa_fwd_fp8(ctypes.byref(p128), 256, 256, 256, 256, 256, 256, 256, 256, 256, 256,
                           16, None) == _lib.MSA_ERR_WORKSPACE
