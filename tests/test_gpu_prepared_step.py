"""prepared_step: the forward + backward pass with arguments marshalled once
gives what fa2_fwd_ws + fa2_bwd_ws give on the same buffers (O, LSE, dK, dV
bit for bit; dQ, whose fp32 reduce-adds land in any order, to rounding), and
matches the fp64 oracle (GPU only)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_grad, check_lse, check_o, rel_fro, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 3, 200, 64, True), (1, 2, 333, 128, False)])
def test_prepared_step_matches_the_plain_calls_and_the_oracle(B, H, N, d, causal):
    x = workloads.make_inputs(B, H, N, d, seed=77 + N)
    g = {k: t.to(DEV) for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    fws = torch.empty(fa2.fa2_fwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=DEV)
    bws = torch.empty(fa2.fa2_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=DEV)
    o1, l1 = fa2.fa2_fwd_ws(g["q"], g["k"], g["v"], fws, scale=scale, causal=causal)
    dq1, dk1, dv1 = fa2.fa2_bwd_ws(g["q"], g["k"], g["v"], o1, g["dO"], l1, bws, scale=scale, causal=causal)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    dq2, dk2, dv2 = (torch.empty_like(o1) for _ in range(3))
    step = fa2.prepared_step(g["q"], g["k"], g["v"], o2, l2, g["dO"], dq2, dk2, dv2, fws, bws, scale, causal)
    step()
    step()  # twice on the same buffers: the second call overwrites the first
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert rel_fro(to_np(dq2), to_np(dq1)) < 1e-3
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], scale, causal)
    check_o(to_np(o2), ref["O"], "O prepared")
    check_lse(to_np(l2), ref["LSE"], "LSE prepared")
    for name, got in (("dQ", dq2), ("dK", dk2), ("dV", dv2)):
        check_grad(to_np(got), ref[name], f"{name} prepared")


def test_prepared_step_rejects_mismatched_shapes():
    q = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 2, 65, 64, dtype=torch.bfloat16, device=DEV)
    lse = torch.zeros(1, 2, 64, dtype=torch.float32, device=DEV)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        fa2.prepared_step(q, k, q, q, lse, q, q, q, q, ws, ws)
