"""The backward kernel runs its CTAs in groups of K/V heads whose re-read
rows (Q, dO, the fp32 dQ accumulator) fit in a share of the L2, heavy key
tiles first inside a group; the last group also takes the heads left over.
With 33 heads at N = 4096, d = 128 that is more than one group with a
remainder: every head's O, LSE, dQ, dK and dV is checked against the fp64
oracle, so a head dropped, repeated or mapped to the wrong tiles fails
(GPU only)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_grad, check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "noncausal"])
def test_every_head_of_a_multi_group_problem(causal):
    B, H, N, d = 1, 33, 4096, 128
    x = workloads.make_inputs(B, H, N, d, seed=4133)
    g = {k: t.to(DEV) for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    for h in range(H):
        sl = slice(h, h + 1)
        ref = oracle.attn_bwd(x["q"][:, sl], x["k"][:, sl], x["v"][:, sl], x["dO"][:, sl], scale, causal)
        check_o(to_np(o[:, sl]), ref["O"], f"O head {h}")
        check_lse(to_np(lse[:, sl]), ref["LSE"], f"LSE head {h}")
        for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
            check_grad(to_np(got[:, sl]), ref[name], f"{name} head {h}")
