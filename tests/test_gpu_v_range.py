"""The forward pass multiplies the weights with an fp16 copy of V.  A K/V head
holding a finite value beyond the fp16 range (|v| > 65504) is copied scaled
by a power of two, which the epilogue multiplies back.  These cases give a
head the same Q, K and dO as head 0 and V = 2^e x (head 0's V), which must
give O = 2^e x (head 0's O) (scaling by a power of two is exact in every
format involved; the two copies differ only below fp16's normal range, so O
is allowed one bf16 ulp), the same LSE bit for bit, and gradients scaled
the same way; head 0 itself is checked against the fp64 oracle (GPU only).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import bf16_ulp, check_grad, check_lse, check_o, rel_fro, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _scaled_copies(x, exps, head_dim=1):
    """Head i + 1 = head 0 with V multiplied by 2^exps[i] (the other tensors copied)."""
    out = {}
    for name, t in x.items():
        t = t.float()
        base = t.select(head_dim, 0)
        heads = [base]
        for e in exps:
            heads.append(base * (2.0 ** e) if name == "v" else base)
        out[name] = torch.stack(heads, dim=head_dim).to(torch.bfloat16).contiguous()
    return out


def _check_scaled(o, lse, e, h, what):
    got = to_np(o.select(1, h)) / 2.0 ** e
    want = to_np(o.select(1, 0))
    err = np.abs(got - want)
    assert np.all(err <= bf16_ulp(want) + 1e-30), f"{what}: O of the 2^{e} head off by up to {err.max():.3e}"
    assert torch.equal(lse.select(1, h), lse.select(1, 0)), f"{what}: LSE differs"


@pytest.mark.parametrize("exps,N,d", [((20,), 300, 64), ((14,), 300, 64), ((20,), 1100, 128)],
                         ids=["2^20", "2^14", "2^20_large_head"])
def test_heads_beyond_fp16_range_forward_and_backward(exps, N, d):
    # 2^20: values up to about 4e6; 2^14: up to about 65536 (the range's
    # edge).  Heads of at most 64K elements are copied to fp16 and rescaled by
    # one kernel, larger ones (1100 x 128) by the grid-wide copy and the
    # per-head rescale.
    B = 1
    x = _scaled_copies(workloads.make_inputs(B, 1, N, d, seed=31), exps)
    assert float(x["v"][0, 1].float().abs().max()) > 65504.0
    g = {k: t.to(DEV) for k, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], scale=scale, causal=True)
    dq, dk, dv = fa2.fa2_bwd(g["q"], g["k"], g["v"], o, g["dO"], lse, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    ref = oracle.attn_bwd(x["q"][:, :1], x["k"][:, :1], x["v"][:, :1], x["dO"][:, :1], scale, True)
    check_o(to_np(o[:, :1]), ref["O"], "O head0")
    check_lse(to_np(lse[:, :1]), ref["LSE"], "LSE head0")
    for name, got in (("dQ", dq), ("dK", dk), ("dV", dv)):
        check_grad(to_np(got[:, :1]), ref[name], f"{name} head0")
    _check_scaled(o, lse, exps[0], 1, "fwd")
    # dV = P^T dO does not depend on V; dQ and dK scale with V (dP = dO V^T).
    assert rel_fro(to_np(dv[:, 1]), to_np(dv[:, 0])) < 1e-2
    for name, got in (("dQ", dq), ("dK", dk)):
        r = rel_fro(to_np(got[:, 1]) / 2.0 ** exps[0], to_np(got[:, 0]))
        assert r < 1e-2, f"{name} of the 2^{exps[0]} head: {r:.3e}"


def test_largest_bf16_value_in_fp16_range_needs_no_scaling():
    # 65280 is the largest bf16 value not above the fp16 maximum (65504):
    # the copy holds it exactly, without scaling (the next bf16 value, 65536,
    # is beyond the range).
    B, H, N, d = 1, 1, 128, 32
    x = workloads.make_inputs(B, H, N, d, seed=32, with_grad=False)
    v = x["v"].float()
    v[0, 0, 5, 3] = 65280.0
    x["v"] = v.to(torch.bfloat16).contiguous()
    assert float(x["v"].float().abs().max()) == 65280.0
    g = {k: t.to(DEV) for k, t in x.items()}
    o, lse = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=False)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], 1 / np.sqrt(d), False)
    check_o(to_np(o), ref_o, "O at fp16 max")
    check_lse(to_np(lse), ref_l, "LSE at fp16 max")


def test_varlen_head_beyond_fp16_range():
    # Packed batch with 2 K/V heads of 1 query head each: K/V head 1 = K/V
    # head 0 with V x 2^20, query head 1 = query head 0.
    lens = [200, 77, 130]
    d = 128
    x = workloads.make_varlen_inputs(lens, lens, 1, 1, d, seed=33)
    cu = {n: x.pop(n) for n in ("cu_q", "cu_k")}
    x = _scaled_copies(x, (20,))
    g = {n: t.to(DEV) for n, t in x.items()}
    cuq, cuk = cu["cu_q"].to(DEV), cu["cu_k"].to(DEV)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], cuq, cuk, max(lens), max(lens), scale=scale, causal=True)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    ref = oracle.attn_varlen(x["q"][:, :1], x["k"][:, :1], x["v"][:, :1], None, cu["cu_q"], cu["cu_k"], scale, True)
    check_o(to_np(o[:, :1]), ref["O"], "O varlen head0")
    check_lse(to_np(lse[:1]), ref["LSE"], "LSE varlen head0")
    got = to_np(o[:, 1]) / 2.0 ** 20
    want = to_np(o[:, 0])
    assert np.all(np.abs(got - want) <= bf16_ulp(want) + 1e-30)
    assert torch.equal(lse[1], lse[0])
