"""The C-ABI library loads, exports every entry point include/fa2.h declares,
and rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import tiled_exact_attention_fa2_gb300 as fa2
from tiled_exact_attention_fa2_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fa2.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa2.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa2_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fa2_fwd", "fa2_bwd", "fa2_bwd_workspace_bytes", "fa2_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    for name in declared_functions():
        assert name in fa2._SIGNATURES, name


def test_status_strings(lib):
    for s in range(10):
        assert fa2.fa2_status_string(s)
    assert fa2.fa2_status_string(0) == "ok"
    assert "unknown" in fa2.fa2_status_string(12345)
    assert fa2.fa2_abi_version() == 101


def test_workspace_bytes(lib):
    # D (fp32 per row) + dQ accumulator (fp32 per element), 256-byte rounded
    assert fa2.fa2_bwd_workspace_bytes(2, 16, 4096, 128) == 2 * 16 * 4096 * 4 + 2 * 16 * 4096 * 128 * 4
    assert fa2.fa2_bwd_workspace_bytes(1, 1, 1, 16) == 256 + 256
    assert fa2.fa2_bwd_workspace_bytes(0, 1, 1, 16) == 0
    assert fa2.fa2_bwd_workspace_bytes(1, 1, 1, 48) == 0


def test_splitkv_suggested_splits(lib):
    f = lib.fa2_fwd_splitkv_suggest_splits
    # 8 sequences x 8 K/V heads (4 query heads each, one query): 64 units per
    # key range, so two ranges reach 0.8 x 152 SMs
    assert f(152, 8, 32, 8, 1, 16384) == 2
    # one sequence x 8 K/V heads against 128K keys: 8 units per range -> 16
    assert f(152, 1, 32, 8, 1, 131072) == 16
    # at most one range per 128-key tile
    assert f(152, 1, 8, 8, 1, 256) == 2
    assert f(152, 1, 8, 8, 1, 1) == 1
    # enough units without splitting
    assert f(152, 64, 64, 32, 1, 16384) == 1
    # up to 256 packed rows per K/V head are one pair of 128-row tiles; 300 rows are two
    assert f(152, 2, 200, 1, 1, 65536) == f(152, 2, 1, 1, 1, 65536) == 61
    assert f(152, 2, 300, 1, 1, 65536) == 31
    # invalid arguments
    for args in ((0, 1, 1, 1, 1, 1), (152, 0, 1, 1, 1, 1), (152, 1, 6, 4, 1, 1), (152, 1, 1, 1, 0, 1),
                 (152, 1, 1, 1, 1, 0)):
        assert f(*args) == 0


A = 1 << 20  # a fake, 16-byte aligned "device" address; never dereferenced


def fwd(lib, q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, H=1, N=128, d=64, scale=0.125, causal=1):
    return lib.fa2_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def bwd(lib, ptrs=None, B=1, H=1, N=128, d=64, scale=0.125):
    p = ptrs or [A * (i + 1) for i in range(9)]
    return lib.fa2_bwd(*p, B, H, N, d, scale, 1, None)


def test_fwd_rejects_bad_arguments(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, lse=None) == 1
    assert fwd(lib, B=0) == 2
    assert fwd(lib, N=0) == 2
    assert fwd(lib, H=-1) == 2
    for d in (0, 8, 48, 96, 256):
        assert fwd(lib, d=d) == 3
    assert fwd(lib, q=A + 8) == 4
    assert fwd(lib, o=4 * A + 2) == 4
    assert fwd(lib, lse=5 * A + 2) == 4
    for s in (0.0, -0.1, float("inf"), float("nan")):
        assert fwd(lib, scale=s) == 5
    assert fwd(lib, o=A) == 9            # o aliases q
    assert fwd(lib, lse=3 * A + 64) == 9  # lse inside v
    assert lib.fa2_fwd(A, 2 * A, 3 * A, 4 * A, 5 * A, 1, 1, (1 << 30) + 1, 64, 0.1, 1, None) == 2


def test_bwd_rejects_bad_arguments(lib):
    p = [A * (i + 1) for i in range(9)]
    for i in range(9):
        q = list(p)
        q[i] = None
        assert bwd(lib, q) == 1
    assert bwd(lib, B=0) == 2
    assert bwd(lib, d=24) == 3
    q = list(p)
    q[6] = 7 * A + 4  # dq misaligned
    assert bwd(lib, q) == 4
    assert bwd(lib, scale=float("nan")) == 5
    q = list(p)
    q[7] = q[6]  # dk == dq
    assert bwd(lib, q) == 9
    q = list(p)
    q[8] = q[0]  # dv == q
    assert bwd(lib, q) == 9


def test_bwd_ws_rejects_bad_workspace(lib):
    p = [A * (i + 1) for i in range(9)]
    need = fa2.fa2_bwd_workspace_bytes(1, 1, 128, 64)
    ws = 64 * A
    assert lib.fa2_bwd_ws(*p, 1, 1, 128, 64, 0.125, 1, None, need, None) == 8
    assert lib.fa2_bwd_ws(*p, 1, 1, 128, 64, 0.125, 1, ws, need - 1, None) == 8
    assert lib.fa2_bwd_ws(*p, 1, 1, 128, 64, 0.125, 1, ws + 16, need, None) == 8


def test_device_status_null(lib):
    assert lib.fa2_device_status(None, 0) == 1


def test_python_binding_checks_metadata():
    import torch
    q = torch.zeros(1, 1, 4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa2.fa2_fwd(q, q, q)  # CPU tensors are refused before any call
    with pytest.raises(ValueError):
        fa2.fa2_fwd(q.float(), q, q)


def fwd_varlen(lib, q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, cuq=6 * A, cuk=7 * A, B=2, H=2, Hkv=1,
               tq=300, tk=400, mq=200, mk=300, d=64, scale=0.125, causal=1):
    return lib.fa2_fwd_varlen(q, k, v, o, lse, cuq, cuk, B, H, Hkv, tq, tk, mq, mk, d, scale, causal, None)


def test_fwd_varlen_rejects_bad_arguments(lib):
    assert fwd_varlen(lib, B=0) == 2
    assert fwd_varlen(lib, Hkv=3) == 2           # H not a multiple of H_kv
    assert fwd_varlen(lib, mq=301) == 2          # a sequence longer than the packed total
    assert fwd_varlen(lib, mq=0) == 2            # queries exist but the maximum length is 0
    assert fwd_varlen(lib, tq=-1) == 2
    assert fwd_varlen(lib, tq=(1 << 30) + 1, mq=5) == 2
    assert fwd_varlen(lib, d=48) == 3
    assert fwd_varlen(lib, scale=0.0) == 5
    assert fwd_varlen(lib, cuq=None) == 1
    assert fwd_varlen(lib, k=None) == 1
    assert fwd_varlen(lib, cuk=7 * A + 2) == 4   # offsets must be 4-byte aligned
    assert fwd_varlen(lib, q=A + 8) == 4
    assert fwd_varlen(lib, o=A) == 9             # o aliases q
    assert fwd_varlen(lib, lse=6 * A) == 9       # lse over the query offsets
    # no query rows: valid, nothing to do (returns before any CUDA call)
    assert fwd_varlen(lib, q=None, o=None, lse=None, tq=0, mq=0) == 0


def test_bwd_varlen_rejects_bad_arguments(lib):
    p = [A * (i + 1) for i in range(9)]
    cu = [10 * A, 11 * A]
    need = lib.fa2_bwd_varlen_workspace_bytes(2, 300, 64)
    assert need >= 300 * 2 * 4 + 300 * 2 * 64 * 4
    ws = 64 * A

    def call(ptrs=p, cus=cu, wsp=ws, wsb=need, **kw):
        a = dict(B=2, H=2, Hkv=1, tq=300, tk=400, mq=200, mk=300, d=64)
        a.update(kw)
        return lib.fa2_bwd_varlen(*ptrs, *cus, a["B"], a["H"], a["Hkv"], a["tq"], a["tk"], a["mq"], a["mk"],
                                  a["d"], 0.125, 1, wsp, wsb, None)

    assert call(B=0) == 2
    assert call(d=24) == 3
    assert call(cus=[None, 11 * A]) == 1
    for i in range(9):
        q = list(p)
        q[i] = None
        assert call(q) == 1
    q = list(p)
    q[7] = q[6]  # dk == dq
    assert call(q) == 9
    assert call(wsp=None) == 8
    assert call(wsb=need - 1) == 8
    assert call(wsp=ws + 16) == 8


def _round256(x):
    return (x + 255) // 256 * 256


def test_fwd_workspace_bytes(lib):
    # fp16 copy of V, then a 64-bit flag and an fp32 scale per K/V head,
    # each part 256-byte rounded
    B, Hkv, N, d = 2, 4, 300, 64
    heads = B * Hkv
    assert fa2.fa2_fwd_workspace_bytes(B, Hkv, N, d) == (_round256(heads * N * d * 2) + _round256(heads * 8) +
                                                         _round256(heads * 4))
    assert fa2.fa2_fwd_workspace_bytes(1, 1, 1, 48) == 0
    assert fa2.fa2_fwd_workspace_bytes(0, 1, 1, 16) == 0


def test_fwd_ws_rejects_bad_workspace(lib):
    need = fa2.fa2_fwd_workspace_bytes(1, 1, 128, 64)
    args = (A, 2 * A, 3 * A, 4 * A, 5 * A, 1, 1, 128, 64, 0.125, 1)
    ws = 64 * A
    assert lib.fa2_fwd_ws(*args, None, need, None) == 8
    assert lib.fa2_fwd_ws(*args, ws, need - 1, None) == 8
    assert lib.fa2_fwd_ws(*args, ws + 16, need, None) == 8
    for p in (A, 2 * A, 3 * A, 4 * A, 5 * A):  # over q, k, v, o, lse
        assert lib.fa2_fwd_ws(*args, p, need, None) == 9


def test_bwd_ws_rejects_overlapping_workspace(lib):
    p = [A * (i + 1) for i in range(9)]
    need = fa2.fa2_bwd_workspace_bytes(1, 1, 128, 64)
    for i in range(9):  # over each of q, k, v, o, dO, lse, dq, dk, dv
        assert lib.fa2_bwd_ws(*p, 1, 1, 128, 64, 0.125, 1, p[i], need, None) == 9


def test_dq_partials_and_deterministic_workspace_bytes(lib):
    f = lib.fa2_bwd_dq_partials_bytes
    # one 128 x d fp32 slot per (query tile, key tile) pair; causal: the
    # pairs on or below the diagonal.  N = 300: 3 tiles.
    assert f(2, 3, 300, 128, 1) == 2 * 3 * 6 * 128 * 128 * 4
    assert f(2, 3, 300, 128, 0) == 2 * 3 * 9 * 128 * 128 * 4
    assert f(1, 1, 300, 64, 1) == 0
    g = lib.fa2_bwd_deterministic_workspace_bytes
    assert g(2, 3, 300, 128, 1) == _round256(2 * 3 * 300 * 4) + _round256(f(2, 3, 300, 128, 1))
    assert g(1, 1, 128, 64, 1) == 0


def test_bwd_main_dq_rejects_bad_modes(lib):
    p = [A * (i + 1) for i in range(9)]  # q, k, v, dO, lse, D, dq buffer, dk, dv
    f = lib.fa2_bwd_main_dq
    assert f(*p, 1, 1, 128, 128, 0.125, 1, 3, None) == 2  # unknown mode
    assert f(*p, 1, 1, 128, 64, 0.125, 1, 1, None) == 3   # register reductions: d = 128 only
    assert f(*p, 1, 1, 128, 64, 0.125, 1, 2, None) == 3   # split partials: d = 128 only
    q = list(p)
    q[8] = q[7]  # dv == dk
    assert f(*q, 1, 1, 128, 128, 0.125, 1, 1, None) == 9


def test_bwd_deterministic_and_dq_reduce_reject_bad_arguments(lib):
    p = [A * (i + 1) for i in range(9)]
    need = lib.fa2_bwd_deterministic_workspace_bytes(1, 1, 256, 128, 1)
    f = lib.fa2_bwd_deterministic
    assert f(*p, 1, 1, 256, 64, 0.125, 1, 64 * A, 1 << 30, None) == 3  # d = 128 only
    assert f(*p, 1, 1, 256, 128, 0.125, 1, None, need, None) == 8
    assert f(*p, 1, 1, 256, 128, 0.125, 1, 64 * A, need - 1, None) == 8
    assert f(*p, 1, 1, 256, 128, 0.125, 1, p[6], need, None) == 9  # workspace over dq
    r = lib.fa2_bwd_dq_reduce
    assert r(None, A, 1, 1, 256, 128, 0.125, 1, None) == 1
    assert r(A, 2 * A, 1, 1, 256, 64, 0.125, 1, None) == 3
    assert r(A + 8, 2 * A, 1, 1, 256, 128, 0.125, 1, None) == 4
    assert r(A, A, 1, 1, 256, 128, 0.125, 1, None) == 9


def test_step_from_host_rejects_bad_arguments_before_any_cuda_call(lib):
    f, ws_bytes = lib.fa2_step_from_host, lib.fa2_step_from_host_workspace_bytes
    I = ctypes.c_int
    plan = (I * 3)(1, 2, 5)
    need = ws_bytes(2, 4, 256, 64, None, 0, 2)
    assert need > 8 * 2 * 4 * 256 * 64 * 2  # the ten tensors plus two streams' scratch
    # an explicit plan: the largest group sets the per-stream scratch
    assert ws_bytes(2, 4, 256, 64, plan, 3, 1) > 0
    assert ws_bytes(2, 4, 256, 64, plan, 2, 1) == 0        # 1 + 2 != 8 heads
    assert ws_bytes(2, 4, 256, 64, (I * 2)(8, 0), 2, 1) == 0  # empty group
    assert ws_bytes(2, 4, 256, 64, None, 0, 0) == 0        # stream count
    assert ws_bytes(2, 4, 256, 64, None, 0, 5) == 0
    assert ws_bytes(2, 4, 256, 48, None, 0, 2) == 0
    good = dict(B=2, H=4, N=256, d=64, scale=0.125, plan=None, n=0, streams=2, ws=A, nbytes=need)

    def call(ptr=A, **kw):
        a = dict(good, **kw)
        return f(ptr, A, A, A, A, A, A, A, A, a["B"], a["H"], a["N"], a["d"], a["scale"], 1, a["plan"], a["n"],
                 a["streams"], a["ws"], a["nbytes"], None)

    assert call(ptr=None) == 1                       # FA2_ERR_NULL
    assert call(d=48) == 3                           # FA2_ERR_HEADDIM
    assert call(N=0) == 2                            # FA2_ERR_SHAPE
    assert call(scale=float("nan")) == 5             # FA2_ERR_SCALE
    assert call(streams=0) == 2
    assert call(plan=plan, n=2) == 2                 # plan does not sum to B * H
    assert call(ws=None) == 8                        # FA2_ERR_WORKSPACE
    assert call(ws=A + 16) == 8                      # not 256-byte aligned
    assert call(nbytes=need - 1) == 8
