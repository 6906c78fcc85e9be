"""fa2_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (the scratch comes from the library's fixed device array).

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test.  The GPU test calls the entry
point through the C ABI twice in a row, on different inputs, and checks each
result against fa2_bwd (which allocates its scratch itself) within the
gradient tolerance the parity tests use.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import GRAD_REL_TOL, rel_fro, to_np

FA2_ERR_SCRATCH_CAPACITY = 10


def test_capacity_and_oversize_rejection():
    lib = fa2.load_library()
    cap = lib.fa2_noalloc_scratch_capacity()
    assert cap == 64 << 20
    assert "fixed array" in fa2.fa2_status_string(FA2_ERR_SCRATCH_CAPACITY)
    # B=1, H=32, N=16384, d=128 needs ~270 MB of scratch: rejected on the host,
    # before any pointer is touched or anything is enqueued.
    need = lib.fa2_bwd_workspace_bytes(1, 32, 16384, 128)
    assert need > cap
    p = [(i + 1) << 20 for i in range(9)]
    assert lib.fa2_bwd_noalloc(*p, 1, 32, 16384, 128, 0.088, 1, None) == FA2_ERR_SCRATCH_CAPACITY


@pytest.mark.gpu
def test_noalloc_matches_fa2_bwd_on_two_calls_in_a_row():
    lib = fa2.load_library()
    dev = torch.device("cuda:0")
    cases = [(2, 3, 333, 128, True, 11), (1, 4, 520, 64, False, 12)]
    for B, H, N, d, causal, seed in cases:
        x = workloads.make_inputs(B, H, N, d, seed=seed)
        g = {k: t.to(dev) for k, t in x.items()}
        scale = 1.0 / np.sqrt(d)
        o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
        ref = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
        out = [torch.empty_like(g["q"]) for _ in range(3)]
        s = torch.cuda.current_stream().cuda_stream
        rc = lib.fa2_bwd_noalloc(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), o.data_ptr(),
                                 g["dO"].data_ptr(), lse.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                                 out[2].data_ptr(), B, H, N, d, ctypes.c_float(scale), 1 if causal else 0, s)
        assert rc == 0, fa2.fa2_status_string(rc)
        torch.cuda.synchronize()
        assert fa2.fa2_device_status(reset=True) == 0
        for name, got, want in zip(("dQ", "dK", "dV"), out, ref):
            err = rel_fro(to_np(got), to_np(want))
            assert err <= GRAD_REL_TOL, f"{name} (B={B} H={H} N={N} d={d}): {err:.3e}"
