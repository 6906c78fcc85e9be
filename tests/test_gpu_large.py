"""The stress and long workloads at full size (GPU only).

stress (B=2, H=16, N=4096, d=128, Q and K x3, causal): every output against
the full fp64 oracle.  long (B=1, H=32, N=16384, d=128, causal and
non-causal): O, LSE and dQ on 64 seeded query rows per head, which the
oracle computes row by row; every output of head (0, 0) (O, LSE, dQ, dK, dV)
element by element against the full oracle of that head, under both masks;
and the gradient identities sum_j dK_j = 0, sum_j dV_j = sum_i dO_i on all
heads.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import GRAD_REL_TOL, check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _gpu(x, scale, causal):
    g = {k: t.to(DEV) for k, t in x.items()}
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    return o, lse, dq, dk, dv


def test_stress_full_oracle():
    w = workloads.WORKLOADS["stress"]
    x = workloads.workload_inputs(w)
    o, lse, dq, dk, dv = _gpu(x, w.scale, True)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], w.scale, True)
    check_o(to_np(o), ref["O"])
    check_lse(to_np(lse), ref["LSE"])
    check_grad(to_np(dq), ref["dQ"], "dQ")
    check_grad(to_np(dk), ref["dK"], "dK")
    check_grad(to_np(dv), ref["dV"], "dV")


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_long_sampled_rows_and_identities(causal):
    w = workloads.WORKLOADS["long"]
    x = workloads.workload_inputs(w)
    o, lse, dq, dk, dv = _gpu(x, w.scale, causal)
    rows = workloads.sample_rows(w.N, 64, w.seed)
    ref = oracle.attn_rows(x["q"], x["k"], x["v"], x["dO"], w.scale, causal, rows)
    check_o(to_np(o[:, :, rows]), ref["O"])
    check_lse(to_np(lse[:, :, rows]), ref["LSE"])
    check_grad(to_np(dq[:, :, rows]), ref["dQ"], "dQ rows")
    # sum over keys of dK vanishes; sum over keys of dV equals sum over queries of dO
    dk_sum = to_np(dk).sum(axis=2)
    dv_sum = to_np(dv).sum(axis=2)
    do_sum = oracle.as_f64(x["dO"]).sum(axis=2)
    dk_scale = np.sqrt((to_np(dk) ** 2).sum(axis=2))
    assert np.all(np.abs(dk_sum) <= GRAD_REL_TOL * dk_scale + 1e-3)
    assert np.linalg.norm(dv_sum - do_sum) <= GRAD_REL_TOL * np.linalg.norm(do_sum)


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_long_one_head_full_gradients(causal):
    # Head (0, 0) of the long workload in full: with causal=False every key
    # tile of every query tile is visited (no causal skip), so this is the
    # only element-wise check of dK and dV on the full-size non-causal path.
    w = workloads.WORKLOADS["long"]
    x = workloads.workload_inputs(w)
    o, lse, dq, dk, dv = _gpu(x, w.scale, causal)
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], w.scale, causal, heads=[(0, 0)])
    check_o(to_np(o[0, 0]), ref["O"][0, 0], "O head0")
    check_lse(to_np(lse[0, 0]), ref["LSE"][0, 0], "LSE head0")
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        check_grad(to_np(got[0, 0]), ref[name][0, 0], f"{name} head0")
