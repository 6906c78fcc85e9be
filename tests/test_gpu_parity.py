"""CUDA path vs the fp64 oracle on identical seeded bf16 inputs (GPU only).

Tolerances: O max-abs <= 1e-2 (one bf16 ulp where |O| >= 4), LSE max-abs
<= 2e-3, dQ/dK/dV relative Frobenius <= 2e-2 per whole tensor.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_grad, check_lse, check_o, rel_fro, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# (B, H, N, d, causal, qk_mult): the small workloads plus ragged / degenerate shapes.
CASES = [
    (1, 2, 64, 16, True, 1.0),      # tiny
    (1, 2, 64, 16, False, 1.0),     # tiny, non-causal
    (8, 4, 256, 32, True, 1.0),     # small GPT layer
    (4, 16, 1024, 64, True, 1.0),   # medium GPT layer
    (4, 16, 1024, 64, False, 1.0),  # medium, non-causal
    (1, 1, 1, 16, True, 1.0),       # single row
    (1, 1, 1, 128, False, 1.0),
    (1, 1, 63, 32, True, 1.0),      # one partial tile
    (1, 1, 65, 64, False, 1.0),
    (1, 2, 129, 128, True, 1.0),    # full tile + 1-row tail
    (2, 3, 200, 128, False, 1.0),
    (2, 3, 200, 128, True, 3.0),    # sharp softmax, ragged
    (1, 1, 300, 16, True, 1.0),
    (1, 2, 384, 64, True, 3.0),
]


def _ids(c):
    B, H, N, d, causal, m = c
    return f"B{B}H{H}N{N}d{d}{'c' if causal else 'n'}{'x3' if m != 1 else ''}"


def _run(x, scale, causal):
    g = {k: t.to(DEV) for k, t in x.items()}
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    return g, o, lse, dq, dk, dv


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_fwd_bwd_chained(case):
    B, H, N, d, causal, mult = case
    x = workloads.make_inputs(B, H, N, d, seed=100 + N + d, qk_mult=mult)
    scale = 1.0 / np.sqrt(d)
    _, o, lse, dq, dk, dv = _run(x, scale, causal)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], scale, causal)
    check_o(to_np(o), ref["O"])
    check_lse(to_np(lse), ref["LSE"])
    check_grad(to_np(dq), ref["dQ"], "dQ")
    check_grad(to_np(dk), ref["dK"], "dK")
    check_grad(to_np(dv), ref["dV"], "dV")


@pytest.mark.parametrize("case", [CASES[2], CASES[4], CASES[10], CASES[11]], ids=_ids)
def test_bwd_isolated_from_fwd(case):
    # The backward fed the oracle's O (rounded to bf16) and LSE (fp32), so its
    # error is measured apart from the forward's.
    B, H, N, d, causal, mult = case
    x = workloads.make_inputs(B, H, N, d, seed=200 + N + d, qk_mult=mult)
    scale = 1.0 / np.sqrt(d)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], scale, causal)
    g = {k: t.to(DEV) for k, t in x.items()}
    o = torch.from_numpy(ref["O"]).to(torch.bfloat16).to(DEV).contiguous()
    lse = torch.from_numpy(ref["LSE"]).to(torch.float32).to(DEV).contiguous()
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        check_grad(to_np(got), ref[name], name)


def test_workload_tiny_both_masks():
    w = workloads.WORKLOADS["tiny"]
    x = workloads.workload_inputs(w)
    for causal in w.causal:
        _, o, lse, dq, dk, dv = _run(x, w.scale, causal)
        ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], w.scale, causal)
        check_o(to_np(o), ref["O"])
        check_lse(to_np(lse), ref["LSE"])
        for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
            check_grad(to_np(got), ref[name], name)


def test_determinism():
    # O, LSE, dK, dV are bitwise reproducible; dQ sums fp32 atomics whose
    # order may vary, so it is only required to agree closely.
    x = workloads.make_inputs(2, 2, 333, 64, seed=5)
    runs = [_run(x, 0.125, True) for _ in range(2)]
    for idx in (1, 2, 4, 5):
        assert torch.equal(runs[0][idx], runs[1][idx])
    assert rel_fro(to_np(runs[0][3]), to_np(runs[1][3])) < 1e-3


def test_workspace_entry_point_matches():
    x = workloads.make_inputs(1, 2, 256, 128, seed=9)
    g, o, lse, dq, dk, dv = _run(x, 1 / np.sqrt(128), True)
    nbytes = fa2.fa2_bwd_workspace_bytes(1, 2, 256, 128)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    dq2, dk2, dv2 = fa2.fa2_bwd_ws(g["q"], g["k"], g["v"], o, g["dO"], lse, ws, scale=1 / np.sqrt(128))
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert rel_fro(to_np(dq), to_np(dq2)) < 1e-3


def test_nonzero_stream_and_invalid_args_raise():
    x = workloads.make_inputs(1, 1, 128, 64, seed=3)
    g = {k: t.to(DEV) for k, t in x.items()}
    s = torch.cuda.Stream()
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True, stream=s)
    s.synchronize()
    o2, lse2 = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    with pytest.raises(fa2.FA2Error):
        fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=-1.0)
    with pytest.raises(fa2.FA2Error):  # output aliasing an input
        fa2.fa2_fwd(g["q"], g["k"], g["v"], o=g["q"])


def test_host_step_pipeline_matches_device_calls():
    # fa2_step_from_host (C ABI) pipelines host<->device copies with the
    # kernels over groups of heads (equal groups, the default plan, explicit
    # groups; one to four compute streams); its results must be those of
    # plain fa2_fwd / fa2_bwd on the same inputs (bit-identical except dQ,
    # whose fp32 reduction order varies between runs).
    import tiled_exact_attention_fa2_gb300 as fa2
    from parity_util import check_grad, to_np
    w = workloads.WORKLOADS["small"]
    x = workloads.workload_inputs(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, causal=True)
    host = {k: x[k].pin_memory() for k in ("q", "k", "v", "dO")}
    host.update({k: torch.zeros_like(host["q"]).pin_memory() for k in ("o", "dq", "dk", "dv")})
    host["lse"] = torch.zeros((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    plans = [dict(chunks=1, compute_streams=1), dict(chunks=3), dict(),  # default: ramp of groups, 2 streams
             dict(groups=[1, 5, 10, 10, 6], compute_streams=3), dict(chunks=32, compute_streams=4)]
    for plan in plans:
        for name in ("o", "lse", "dq", "dk", "dv"):
            host[name].zero_()
        fa2.fa2_step_from_host(host, True, None, None, **plan)
        torch.cuda.synchronize()
        assert fa2.fa2_device_status(reset=True) == 0
        assert torch.equal(host["o"], o.cpu()) and torch.equal(host["lse"], lse.cpu())
        assert torch.equal(host["dk"], dk.cpu()) and torch.equal(host["dv"], dv.cpu())
        check_grad(to_np(host["dq"]), to_np(dq), "dQ")
    # a caller-owned workspace, reused; a side stream as `stream`
    ws = torch.empty(fa2.fa2_step_from_host_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()
    for _ in range(2):
        host["o"].zero_()
        fa2.fa2_step_from_host(host, True, None, side, workspace=ws)
        side.synchronize()
        assert torch.equal(host["o"], o.cpu()) and torch.equal(host["dv"], dv.cpu())
    # pageable (not page-locked) host memory: slower, same results
    pageable = {k: t.clone() for k, t in host.items()}
    for name in ("o", "lse", "dq", "dk", "dv"):
        pageable[name].zero_()
    assert not pageable["q"].is_pinned()
    fa2.fa2_step_from_host(pageable, True, None, None, chunks=2)
    torch.cuda.synchronize()
    assert torch.equal(pageable["o"], o.cpu()) and torch.equal(pageable["lse"], lse.cpu())
    assert torch.equal(pageable["dk"], dk.cpu()) and torch.equal(pageable["dv"], dv.cpu())
    check_grad(to_np(pageable["dq"]), to_np(dq), "dQ (pageable)")
    with pytest.raises(ValueError):
        fa2.fa2_step_from_host(host, True, None, None, groups=[16, 15])
