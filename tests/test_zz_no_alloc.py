"""fa2_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (the scratch comes from the library's fixed device array).

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  The GPU test calls the entry
point through the C ABI three times in a row on different problems (the
middle one with scratch just under the array's 64 MiB, so the tail of the
array is used) and checks each result against fa2_bwd, which allocates its
scratch itself: dK and dV must be bit-identical (both are deterministic),
dQ (an fp32 reduction whose order varies) within 1e-3 relative.  Each result
is also checked against the fp64 oracle with the parity tolerances.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_grad, rel_fro, to_np

FA2_ERR_NULL = 1
FA2_ERR_SCALE = 5
FA2_ERR_SCRATCH_CAPACITY = 10


def _largest_n_that_fits(lib, B, H, d, cap):
    lo, hi = 1, 1 << 20
    assert lib.fa2_bwd_workspace_bytes(B, H, lo, d) <= cap < lib.fa2_bwd_workspace_bytes(B, H, hi, d)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if lib.fa2_bwd_workspace_bytes(B, H, mid, d) <= cap:
            lo = mid
        else:
            hi = mid
    return lo


def test_capacity_and_oversize_rejection():
    lib = fa2.load_library()
    cap = lib.fa2_noalloc_scratch_capacity()
    assert cap == 64 << 20
    assert "fixed array" in fa2.fa2_status_string(FA2_ERR_SCRATCH_CAPACITY)
    # B=1, H=32, N=16384, d=128 needs ~270 MB of scratch.  Arguments are
    # checked first, as fa2_bwd checks them: NULL pointers give FA2_ERR_NULL
    # even for an oversize problem; with valid (never dereferenced) pointers
    # the oversize problem is rejected on the host before any CUDA call.
    need = lib.fa2_bwd_workspace_bytes(1, 32, 16384, 128)
    assert need > cap
    null = [None] * 9
    assert lib.fa2_bwd_noalloc(*null, 1, 32, 16384, 128, 0.088, 1, None) == FA2_ERR_NULL
    p = [(i + 1) << 30 for i in range(9)]
    assert lib.fa2_bwd_noalloc(*p, 1, 32, 16384, 128, 0.088, 1, None) == FA2_ERR_SCRATCH_CAPACITY
    # The boundary: one more row than the largest problem that fits is
    # rejected (the largest one itself runs in the GPU test below).
    n_fit = _largest_n_that_fits(lib, 1, 8, 128, cap)
    assert lib.fa2_bwd_workspace_bytes(1, 8, n_fit, 128) <= cap < lib.fa2_bwd_workspace_bytes(1, 8, n_fit + 1, 128)
    assert lib.fa2_bwd_noalloc(*p, 1, 8, n_fit + 1, 128, 0.088, 1, None) == FA2_ERR_SCRATCH_CAPACITY
    # a bad scale is reported as such, also for an oversize problem
    assert lib.fa2_bwd_noalloc(*p, 1, 8, n_fit + 1, 128, -1.0, 1, None) == FA2_ERR_SCALE


@pytest.mark.gpu
def test_noalloc_matches_fa2_bwd_on_calls_in_a_row():
    lib = fa2.load_library()
    cap = lib.fa2_noalloc_scratch_capacity()
    dev = torch.device("cuda:0")
    n_big = _largest_n_that_fits(lib, 1, 8, 128, cap)
    # (B, H, N, d, causal, seed); the middle problem's scratch is within a
    # fraction of a row tile of the array's end.
    cases = [(2, 3, 333, 128, True, 11), (1, 8, n_big, 128, True, 13), (1, 4, 520, 64, False, 12)]
    assert cap - lib.fa2_bwd_workspace_bytes(1, 8, n_big, 128) < 8 * 128 * 4 * 2
    prepared = []
    for B, H, N, d, causal, seed in cases:
        x = workloads.make_inputs(B, H, N, d, seed=seed)
        g = {k: t.to(dev) for k, t in x.items()}
        scale = 1.0 / np.sqrt(d)
        o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
        want = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
        prepared.append((x, g, o, lse, scale, want))
    torch.cuda.synchronize()
    # The calls back to back on one stream, results read afterwards.
    s = torch.cuda.current_stream().cuda_stream
    outs = []
    for (B, H, N, d, causal, _), (x, g, o, lse, scale, _) in zip(cases, prepared):
        out = [torch.empty_like(g["q"]) for _ in range(3)]
        rc = lib.fa2_bwd_noalloc(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), o.data_ptr(),
                                 g["dO"].data_ptr(), lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                                 out[2].data_ptr(), B, H, N, d, ctypes.c_float(scale), 1 if causal else 0, s)
        assert rc == 0, fa2.fa2_status_string(rc)
        outs.append(out)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    for (B, H, N, d, causal, _), (x, g, o, lse, scale, want), got in zip(cases, prepared, outs):
        tag = f"B={B} H={H} N={N} d={d}"
        assert torch.equal(got[1], want[1]), f"dK differs from fa2_bwd ({tag})"
        assert torch.equal(got[2], want[2]), f"dV differs from fa2_bwd ({tag})"
        assert rel_fro(to_np(got[0]), to_np(want[0])) < 1e-3, f"dQ differs from fa2_bwd ({tag})"
        heads = [(0, 0)] if N > 4096 else None
        ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], scale, causal, heads=heads)
        for name, t in zip(("dQ", "dK", "dV"), got):
            if heads is None:
                check_grad(to_np(t), ref[name], f"{name} noalloc")
            else:
                check_grad(to_np(t[0, 0]), ref[name][0, 0], f"{name} noalloc head0")
