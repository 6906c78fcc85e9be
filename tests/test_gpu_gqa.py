"""Grouped-query / multi-query attention (K/V heads shared by groups of query
heads) on the GPU against the fp64 oracle's attn_bwd_gqa (GPU only).

Same tolerances as the main parity tests: O max-abs <= 1e-2 (one bf16 ulp
where |O| >= 4), LSE max-abs <= 2e-3, gradients relative Frobenius <= 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (B, H, H_kv, N, d, causal)
CASES = [
    (1, 4, 2, 200, 64, True),     # GQA, ragged
    (2, 8, 1, 256, 128, True),    # MQA
    (1, 6, 3, 129, 128, False),   # GQA, non-causal, 1-row tail
    (1, 4, 4, 160, 32, True),     # group of one == plain attention
    (1, 8, 2, 1024, 128, True),   # several query tiles per K/V tile
    (2, 4, 2, 100, 16, False),
]


def _gqa_inputs(B, H, Hkv, N, d, seed):
    x = workloads.make_inputs(B, H, N, d, seed=seed)
    kv = workloads.make_inputs(B, Hkv, N, d, seed=seed + 1, with_grad=False)
    return {"q": x["q"], "dO": x["dO"], "k": kv["k"], "v": kv["v"]}


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}kv{}N{}d{}{}".format(*c[:5], "c" if c[5] else "n"))
def test_gqa_fwd_bwd_against_oracle(case):
    B, H, Hkv, N, d, causal = case
    x = _gqa_inputs(B, H, Hkv, N, d, 400 + N + H)
    scale = 1.0 / np.sqrt(d)
    g = {k: t.to(DEV) for k, t in x.items()}
    o, lse = fa2.fa2_fwd_gqa(g["q"], g["k"], g["v"], scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd_gqa(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    ref = oracle.attn_bwd_gqa(x["q"], x["k"], x["v"], x["dO"], scale, causal)
    check_o(to_np(o), ref["O"])
    check_lse(to_np(lse), ref["LSE"])
    check_grad(to_np(dq), ref["dQ"], "dQ")
    check_grad(to_np(dk), ref["dK"], "dK")
    check_grad(to_np(dv), ref["dV"], "dV")


def test_group_of_one_matches_plain_entry_points_bitwise():
    x = workloads.make_inputs(1, 4, 300, 64, seed=77)
    g = {k: t.to(DEV) for k, t in x.items()}
    o1, l1 = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True)
    o2, l2 = fa2.fa2_fwd_gqa(g["q"], g["k"], g["v"], causal=True)
    dq1, dk1, dv1 = fa2.fa2_bwd(g["q"], g["k"], g["v"], o1, g["dO"], l1, causal=True)
    dq2, dk2, dv2 = fa2.fa2_bwd_gqa(g["q"], g["k"], g["v"], o2, g["dO"], l2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)


def test_bad_group_rejected():
    x = workloads.make_inputs(1, 6, 64, 64, seed=1)
    g = {k: t.to(DEV) for k, t in x.items()}
    kv = g["k"][:, :4].contiguous()
    with pytest.raises(fa2.FA2Error):  # 6 query heads do not split into 4 groups
        fa2.fa2_fwd_gqa(g["q"], kv, kv)
