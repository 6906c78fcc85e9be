"""Forward and backward on inputs whose row maxima move late in the key
sequence, against the fp64 oracle (GPU only).

The forward kernel subtracts a reference maximum that may trail a row's
running maximum (it is raised only when a tile's maximum exceeds it by more
than a slack, and O is rescaled then); these inputs make the running maximum
grow tile after tile ('ramp'), or jump late and far ('spike'), so that both
the no-rescale path, with weights above 1, and the rescale path carry most of
the result.  Tolerances as the main parity tests.
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

# (profile, strength, N, d, causal)
CASES = [
    ("ramp", 0.5, 1024, 128, True),
    ("ramp", 4.0, 1024, 128, True),
    ("ramp", 4.0, 700, 64, False),
    ("spike", 2.0, 1024, 128, True),
    ("spike", 6.0, 520, 128, False),
    ("spike", 6.0, 333, 32, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "{}{}_N{}d{}{}".format(c[0], c[1], c[2], c[3], "c" if c[4] else "n"))
def test_late_maxima_against_oracle(case):
    profile, strength, N, d, causal = case
    B, H = 1, 2
    x = workloads.make_profile_inputs(B, H, N, d, profile, strength, seed=900 + N + d)
    g = {n: t.to(DEV) for n, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=causal)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    ref = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], scale, causal)
    check_o(to_np(o), ref["O"])
    check_lse(to_np(lse), ref["LSE"])
    check_grad(to_np(dq), ref["dQ"], "dQ")
    check_grad(to_np(dk), ref["dK"], "dK")
    check_grad(to_np(dv), ref["dV"], "dV")
