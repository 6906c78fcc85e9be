"""GB300 (sm_103a) FlashAttention-2: thin Python binding of the C ABI in include/fa2.h.

Every step of the computation runs in the CUDA kernels of
``libfa2_gb300.so``; this module only checks tensor metadata, allocates
outputs with torch and passes raw pointers, sizes and the current CUDA stream.
There is no fallback: if the shared library is missing, every call raises.

Build the library with ``python -c "import __graft_entry__ as g; g.build()"``
(or ``python tiled_exact_attention_fa2_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

from . import _build

__all__ = [
    "FA2Error", "load_library", "fa2_fwd", "fa2_fwd_ws", "fa2_fwd_workspace_bytes", "fa2_bwd", "fa2_bwd_ws", "fa2_bwd_workspace_bytes",
    "fa2_status_string", "fa2_device_status", "fa2_abi_version", "fa2_step_from_host",
    "fa2_step_from_host_workspace_bytes",
    "fa2_bwd_stages", "fa2_bwd_noalloc", "fa2_fwd_gqa", "fa2_bwd_gqa", "fa2_fwd_splitkv",
    "fa2_fwd_varlen", "fa2_bwd_varlen", "prepared_step", "FA2_OK",
]

FA2_OK = 0
_LIB: Optional[ctypes.CDLL] = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

_SIGNATURES = {
    "fa2_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_fwd_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa2_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa2_fwd_gqa_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa2_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa2_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa2_status_string": (ctypes.c_char_p, [_i]),
    "fa2_device_status": (_i, [ctypes.POINTER(_i), _i]),
    "fa2_abi_version": (_i, []),
    "fa2_bwd_preprocess": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "fa2_bwd_main": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_dq_convert": (_i, [_vp, _vp, _i, _i, _i, _i, _f, _vp]),
    "fa2_bwd_main_dq": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "fa2_bwd_dq_partials_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa2_bwd_dq_reduce": (_i, [_vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_deterministic_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa2_bwd_deterministic": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _sz,
                                   _vp]),
    "fa2_last_error_detail": (ctypes.c_char_p, []),
    "fa2_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_noalloc_scratch_capacity": (_sz, []),
    "fa2_step_from_host_workspace_bytes": (_sz, [_i, _i, _i, _i, ctypes.POINTER(_i), _i, _i]),
    "fa2_step_from_host": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i,
                                ctypes.POINTER(_i), _i, _i, _vp, _sz, _vp]),
    "fa2_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_gqa_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz,
                            _vp]),
    "fa2_check_wait_timeout": (_i, [_i, ctypes.POINTER(_i)]),
    "fa2_fwd_splitkv_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa2_fwd_splitkv_suggest_splits": (_i, [_i, _i, _i, _i, _i, _i]),
    "fa2_fwd_splitkv": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "fa2_fwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa2_bwd_varlen_workspace_bytes": (_sz, [_i, _i, _i]),
    "fa2_bwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i,
                            _f, _i, _vp, _sz, _vp]),
}


class FA2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = load_library().fa2_last_error_detail().decode() if status in (6, 7) else ""
        super().__init__(f"{fn} failed with status {status}: {fa2_status_string(status)}"
                         + (f" [{detail}]" if detail else ""))


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libfa2_gb300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{os.path.basename(path)} is not built; run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB_PATH:
        _LIB = lib
    return lib


def fa2_status_string(status: int) -> str:
    return load_library().fa2_status_string(int(status)).decode()


def fa2_abi_version() -> int:
    return load_library().fa2_abi_version()


def fa2_device_status(reset: bool = False) -> int:
    """Device status word of the kernels (0 = every internal wait completed)."""
    v = _i(0)
    rc = load_library().fa2_device_status(ctypes.byref(v), 1 if reset else 0)
    if rc != FA2_OK:
        raise FA2Error("fa2_device_status", rc)
    return v.value


def fa2_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return load_library().fa2_bwd_workspace_bytes(B, H, N, d)


def _shape(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, d], got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return tuple(t.shape)


def _stream(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def fa2_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, scale: Optional[float] = None, causal: bool = True,
            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O [B,H,N,d] bf16 and LSE [B,H,N] fp32 of softmax(scale Q K^T) V."""
    lib = load_library()
    B, H, N, d = _shape(q, "q")
    if _shape(k, "k") != (B, H, N, d) or _shape(v, "v") != (B, H, N, d):
        raise ValueError("q, k and v must have the same shape")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    _shape(o, "o")
    rc = lib.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                     _scale(scale, d), 1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_fwd", rc)
    return o, lse


def fa2_fwd_workspace_bytes(B: int, H_kv: int, N: int, d: int) -> int:
    return load_library().fa2_fwd_workspace_bytes(B, H_kv, N, d)


def fa2_fwd_ws(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, workspace: torch.Tensor,
               o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, scale: Optional[float] = None,
               causal: bool = True, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """fa2_fwd with caller-owned scratch (a CUDA byte tensor of fa2_fwd_workspace_bytes bytes)."""
    lib = load_library()
    B, H, N, d = _shape(q, "q")
    if _shape(k, "k") != (B, H, N, d) or _shape(v, "v") != (B, H, N, d):
        raise ValueError("q, k and v must have the same shape")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    _shape(o, "o")
    rc = lib.fa2_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
                        _scale(scale, d), 1 if causal else 0, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_fwd_ws", rc)
    return o, lse


def _bwd_common(q, k, v, o, dO, lse, dq, dk, dv):
    B, H, N, d = _shape(q, "q")
    for name, t in (("k", k), ("v", v), ("o", o), ("dO", dO)):
        if _shape(t, name) != (B, H, N, d):
            raise ValueError(f"{name} must have q's shape")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _shape(t, name)
    return (B, H, N, d), dq, dk, dv


def fa2_bwd(q, k, v, o, dO, lse, dq=None, dk=None, dv=None, scale: Optional[float] = None,
            causal: bool = True, stream=None):
    """dQ, dK, dV (bf16) of L with dL/dO = dO; scratch is allocated stream-ordered inside the library."""
    lib = load_library()
    (B, H, N, d), dq, dk, dv = _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    rc = lib.fa2_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                     dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, _scale(scale, d),
                     1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd", rc)
    return dq, dk, dv


def fa2_bwd_ws(q, k, v, o, dO, lse, workspace: torch.Tensor, dq=None, dk=None, dv=None,
               scale: Optional[float] = None, causal: bool = True, stream=None):
    """fa2_bwd with caller-owned scratch (a CUDA byte tensor of fa2_bwd_workspace_bytes bytes)."""
    lib = load_library()
    (B, H, N, d), dq, dk, dv = _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    rc = lib.fa2_bwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, _scale(scale, d),
                        1 if causal else 0, workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_ws", rc)
    return dq, dk, dv


def prepared_step(q, k, v, o, lse, dO, dq, dk, dv, fwd_workspace: torch.Tensor, bwd_workspace: torch.Tensor,
                  scale: Optional[float] = None, causal: bool = True, stream=None):
    """A callable that enqueues fa2_fwd_ws then fa2_bwd_ws on fixed buffers.

    Every argument is checked and converted to its C type once, here; each
    call of the returned function makes the two C calls with those values
    (which still validate their arguments).  For loops that run the same
    small problem many times, where marshalling arguments in Python would
    take as long as the kernels.  The tensors must stay alive (and in place)
    for as long as the callable is used.
    """
    lib = load_library()
    B, H, N, d = _shape(q, "q")
    if _shape(k, "k") != (B, H, N, d) or _shape(v, "v") != (B, H, N, d):
        raise ValueError("q, k and v must have the same shape")
    _shape(o, "o")
    _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    vp, ci, cf, cs = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sc, cz, st = cf(_scale(scale, d)), ci(1 if causal else 0), vp(_stream(stream, q.device))
    dims = (ci(B), ci(H), ci(N), ci(d))
    fargs = (vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()), vp(lse.data_ptr()), *dims,
             sc, cz, vp(fwd_workspace.data_ptr()), cs(fwd_workspace.numel() * fwd_workspace.element_size()), st)
    bargs = (vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()), vp(dO.data_ptr()),
             vp(lse.data_ptr()), vp(dq.data_ptr()), vp(dk.data_ptr()), vp(dv.data_ptr()), *dims, sc, cz,
             vp(bwd_workspace.data_ptr()), cs(bwd_workspace.numel() * bwd_workspace.element_size()), st)
    fwd, bwd = lib.fa2_fwd_ws, lib.fa2_bwd_ws

    def step():
        rc = fwd(*fargs)
        if rc != FA2_OK:
            raise FA2Error("fa2_fwd_ws", rc)
        rc = bwd(*bargs)
        if rc != FA2_OK:
            raise FA2Error("fa2_bwd_ws", rc)

    return step


def _gqa_shapes(q, k, v):
    B, H, N, d = _shape(q, "q")
    Bk, Hkv, Nk, dk_ = _shape(k, "k")
    if (Bk, Nk, dk_) != (B, N, d) or _shape(v, "v") != (B, Hkv, N, d):
        raise ValueError("k and v must be [B, H_kv, N, d] with q's B, N and d")
    return B, H, Hkv, N, d


def fa2_fwd_gqa(q, k, v, o=None, lse=None, scale: Optional[float] = None, causal: bool = True, stream=None):
    """Grouped-query forward: q [B,H,N,d], k/v [B,H_kv,N,d]; query head h reads K/V head h // (H // H_kv)."""
    lib = load_library()
    B, H, Hkv, N, d = _gqa_shapes(q, k, v)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _shape(o, "o")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    rc = lib.fa2_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d,
                         _scale(scale, d), 1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_fwd_gqa", rc)
    return o, lse


def fa2_bwd_gqa(q, k, v, o, dO, lse, dq=None, dk=None, dv=None, scale: Optional[float] = None,
                causal: bool = True, stream=None):
    """Grouped-query backward: dk/dv [B,H_kv,N,d] are sums over each group of query heads."""
    lib = load_library()
    B, H, Hkv, N, d = _gqa_shapes(q, k, v)
    for name, t in (("o", o), ("dO", dO)):
        if _shape(t, name) != (B, H, N, d):
            raise ValueError(f"{name} must have q's shape")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    rc = lib.fa2_bwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, N, d, _scale(scale, d),
                         1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_gqa", rc)
    return dq, dk, dv


def fa2_fwd_splitkv(q, k, v, num_splits: Optional[int] = None, o=None, lse=None, workspace=None,
                    scale: Optional[float] = None, causal: bool = True, stream=None):
    """Split-KV forward for Nq <= Nk (decoding): q [B,H,Nq,d], k/v [B,H_kv,Nk,d].

    Returns (o [B,H,Nq,d] bf16, lse [B,H,Nq] fp32).  ``num_splits`` defaults
    to fa2_fwd_splitkv_suggest_splits for q's device.  ``workspace`` (a CUDA
    byte tensor) is allocated here when not given."""
    lib = load_library()
    B, H, Nq, d = _shape(q, "q")
    Bk, Hkv, Nk, dk_ = _shape(k, "k")
    if (Bk, dk_) != (B, d) or _shape(v, "v") != (B, Hkv, Nk, d):
        raise ValueError("k and v must be [B, H_kv, Nk, d] with q's B and d")
    if num_splits is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        num_splits = max(1, lib.fa2_fwd_splitkv_suggest_splits(sms, B, H, Hkv, Nq, Nk))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = lib.fa2_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wptr = workspace.data_ptr() if workspace is not None else None
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.fa2_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, Nq,
                             Nk, d, _scale(scale, d), 1 if causal else 0, num_splits, wptr, wbytes,
                             _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_fwd_splitkv", rc)
    return o, lse


def _packed(t, name: str):
    if t.dim() != 3:
        raise ValueError(f"{name} must be packed [total, heads, d], got {tuple(t.shape)}")
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    return tuple(t.shape)


def _cu(t, name: str):
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 1 or t.numel() < 2:
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor of B + 1 offsets")
    return t.numel() - 1


def _ptr(t):
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _varlen_shapes(q, k, v, cu_seqlens_q, cu_seqlens_k):
    tq, H, d = _packed(q, "q")
    tk, Hkv, dk_ = _packed(k, "k")
    if dk_ != d or _packed(v, "v") != (tk, Hkv, d):
        raise ValueError("k and v must be [total_k, H_kv, d] with q's d")
    B = _cu(cu_seqlens_q, "cu_seqlens_q")
    if _cu(cu_seqlens_k, "cu_seqlens_k") != B:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    return B, H, Hkv, tq, tk, d


def _max_len(cu, given):
    if given is not None:
        return int(given)
    return int((cu[1:] - cu[:-1]).max().item()) if cu.numel() > 1 else 0


def fa2_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: Optional[int] = None,
                   max_seqlen_k: Optional[int] = None, o=None, lse=None, scale: Optional[float] = None,
                   causal: bool = True, stream=None):
    """Variable-length forward on packed sequences: q [total_q,H,d], k/v [total_k,H_kv,d],
    cu_seqlens_* CUDA int32 [B+1].  Returns (o [total_q,H,d] bf16, lse [H,total_q] fp32).
    The maximum lengths are read from the offsets (a device sync) when not given."""
    lib = load_library()
    B, H, Hkv, tq, tk, d = _varlen_shapes(q, k, v, cu_seqlens_q, cu_seqlens_k)
    mq, mk = _max_len(cu_seqlens_q, max_seqlen_q), _max_len(cu_seqlens_k, max_seqlen_k)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((H, tq), dtype=torch.float32, device=q.device) if lse is None else lse
    if _packed(o, "o") != (tq, H, d):
        raise ValueError("o must have q's shape")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (H, tq):
        raise ValueError("lse must be a contiguous fp32 [H, total_q] tensor")
    rc = lib.fa2_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), cu_seqlens_q.data_ptr(),
                            cu_seqlens_k.data_ptr(), B, H, Hkv, tq, tk, mq, mk, d, _scale(scale, d),
                            1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_fwd_varlen", rc)
    return o, lse


def fa2_bwd_varlen(q, k, v, o, dO, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: Optional[int] = None,
                   max_seqlen_k: Optional[int] = None, dq=None, dk=None, dv=None, workspace=None,
                   scale: Optional[float] = None, causal: bool = True, stream=None):
    """Variable-length backward: returns (dq [total_q,H,d], dk, dv [total_k,H_kv,d]); dk, dv
    sum over each group of query heads.  ``workspace`` is allocated here when not given."""
    lib = load_library()
    B, H, Hkv, tq, tk, d = _varlen_shapes(q, k, v, cu_seqlens_q, cu_seqlens_k)
    mq, mk = _max_len(cu_seqlens_q, max_seqlen_q), _max_len(cu_seqlens_k, max_seqlen_k)
    for name, t in (("o", o), ("dO", dO)):
        if _packed(t, name) != (tq, H, d):
            raise ValueError(f"{name} must have q's shape")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (H, tq):
        raise ValueError("lse must be a contiguous fp32 [H, total_q] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = lib.fa2_bwd_varlen_workspace_bytes(H, tq, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.fa2_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                            cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H, Hkv, tq, tk, mq, mk, d,
                            _scale(scale, d), 1 if causal else 0, workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_varlen", rc)
    return dq, dk, dv


def fa2_bwd_noalloc(q, k, v, o, dO, lse, dq=None, dk=None, dv=None, scale: Optional[float] = None,
                    causal: bool = True, stream=None):
    """fa2_bwd for callers that cannot allocate device memory: the library's
    scratch comes from a fixed 64 MiB device array shared by all calls (see
    include/fa2.h); concurrent calls on one device race."""
    lib = load_library()
    (B, H, N, d), dq, dk, dv = _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    rc = lib.fa2_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
                             lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                             _scale(scale, d), 1 if causal else 0, _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_noalloc", rc)
    return dq, dk, dv


FA2_DQ_REDUCE, FA2_DQ_ATOMIC, FA2_DQ_SPLIT = 0, 1, 2


def fa2_bwd_deterministic(q, k, v, o, dO, lse, dq=None, dk=None, dv=None, workspace=None,
                          scale: Optional[float] = None, causal: bool = True, stream=None):
    """Bitwise-reproducible backward (d = 128): dQ summed over key tiles in a
    fixed order.  ``workspace`` (CUDA byte tensor) is allocated here when not given."""
    lib = load_library()
    (B, H, N, d), dq, dk, dv = _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    need = lib.fa2_bwd_deterministic_workspace_bytes(B, H, N, d, 1 if causal else 0)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.fa2_bwd_deterministic(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(),
                                   lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                   _scale(scale, d), 1 if causal else 0, workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(), _stream(stream, q.device))
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_deterministic", rc)
    return dq, dk, dv


def fa2_bwd_stages(q, k, v, o, dO, lse, Dvec, dq_acc, dq, dk, dv, scale: Optional[float] = None,
                   causal: bool = True, stream=None, hook=None, dq_mode: int = FA2_DQ_REDUCE):
    """fa2_bwd_ws as its three C-ABI stages; ``hook(i)`` is called before stage i
    (0: preprocess, 1: main, 2: dQ convert) and with i = 3 after the last, so a
    caller can record CUDA events between them."""
    lib = load_library()
    (B, H, N, d), dq, dk, dv = _bwd_common(q, k, v, o, dO, lse, dq, dk, dv)
    sc, st = _scale(scale, d), _stream(stream, q.device)
    hook = hook or (lambda i: None)
    hook(0)
    # (split mode: D only, the partial slots are written whole)
    acc0 = None if dq_mode == FA2_DQ_SPLIT else dq_acc.data_ptr()
    rc = lib.fa2_bwd_preprocess(o.data_ptr(), dO.data_ptr(), Dvec.data_ptr(), acc0, B, H, N, d, st)
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_preprocess", rc)
    hook(1)
    rc = lib.fa2_bwd_main_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), dO.data_ptr(), lse.data_ptr(),
                             Dvec.data_ptr(), dq_acc.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, sc,
                             1 if causal else 0, dq_mode, st)
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_main_dq", rc)
    hook(2)
    if dq_mode == FA2_DQ_SPLIT:
        rc = lib.fa2_bwd_dq_reduce(dq_acc.data_ptr(), dq.data_ptr(), B, H, N, d, sc, 1 if causal else 0, st)
    else:
        rc = lib.fa2_bwd_dq_convert(dq_acc.data_ptr(), dq.data_ptr(), B, H, N, d, sc, st)
    if rc != FA2_OK:
        raise FA2Error("fa2_bwd_dq_convert", rc)
    hook(3)
    return dq, dk, dv


def _group_plan(BH: int, chunks: Optional[int], groups):
    """Head counts per group for fa2_step_from_host: `groups` as given,
    `chunks` equal groups, or None for the library's default plan."""
    if groups is not None:
        sizes = [int(x) for x in groups]
        if sum(sizes) != BH or min(sizes) < 1:
            raise ValueError(f"groups must be positive head counts summing to B * H = {BH}")
        return sizes
    if chunks is not None:
        n = max(1, min(BH, int(chunks)))
        return [BH * (i + 1) // n - BH * i // n for i in range(n)]
    return None


def fa2_step_from_host_workspace_bytes(B: int, H: int, N: int, d: int, groups=None, compute_streams: int = 2) -> int:
    arr, n = _int_array(groups)
    return load_library().fa2_step_from_host_workspace_bytes(B, H, N, d, arr, n, compute_streams)


def _int_array(values):
    if values is None:
        return None, 0
    return (ctypes.c_int * len(values))(*values), len(values)


def fa2_step_from_host(host: dict, causal: bool = True, scale: Optional[float] = None, stream=None,
                       chunks: Optional[int] = None, groups=None, compute_streams: int = 2,
                       workspace: Optional[torch.Tensor] = None) -> dict:
    """One forward + backward pass on host tensors (C ABI fa2_step_from_host).

    ``host`` holds CPU tensors (page-locked for overlap): bf16 q, k, v, dO
    [B, H, N, d] and outputs o, dq, dk, dv (bf16, same shape) and lse (fp32
    [B, H, N]).  The library pipelines the copies and kernels over groups of
    heads (``groups`` head counts, ``chunks`` equal groups, or its default
    plan) on ``compute_streams`` compute streams.  ``workspace`` is a CUDA
    uint8 tensor of at least fa2_step_from_host_workspace_bytes(...) bytes
    (allocated here when omitted).  Everything is enqueued on ``stream``
    (default: the current stream); synchronise it before reading ``host``.
    """
    q = host["q"]
    if q.dim() != 4 or q.dtype != torch.bfloat16 or q.is_cuda:
        raise ValueError("host['q'] must be a CPU bfloat16 [B, H, N, d] tensor")
    B, H, N, d = q.shape
    for name in ("k", "v", "dO", "o", "dq", "dk", "dv"):
        t = host[name]
        if t.shape != q.shape or t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous():
            raise ValueError(f"host['{name}'] must be a contiguous CPU bfloat16 tensor shaped like q")
    lse = host["lse"]
    if tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32 or lse.is_cuda or not lse.is_contiguous():
        raise ValueError("host['lse'] must be a contiguous CPU float32 [B, H, N] tensor")
    plan = _group_plan(B * H, chunks, groups)
    arr, n = _int_array(plan)
    lib = load_library()
    need = lib.fa2_step_from_host_workspace_bytes(B, H, N, d, arr, n, compute_streams)
    if need == 0:
        raise FA2Error("fa2_step_from_host_workspace_bytes", 2)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=torch.cuda.current_device())
    st = _stream(stream, workspace.device)
    rc = lib.fa2_step_from_host(q.data_ptr(), host["k"].data_ptr(), host["v"].data_ptr(), host["dO"].data_ptr(),
                                host["o"].data_ptr(), lse.data_ptr(), host["dq"].data_ptr(), host["dk"].data_ptr(),
                                host["dv"].data_ptr(), B, H, N, d, _scale(scale, d), 1 if causal else 0, arr, n,
                                compute_streams, workspace.data_ptr(), workspace.numel(), st)
    if rc != FA2_OK:
        raise FA2Error("fa2_step_from_host", rc)
    return host
