"""Variable-length (packed) batches, forward and backward, against the fp64
oracle's attn_varlen (GPU only).  Tolerances as the main parity tests: O
max-abs 1e-2 (or one bf16 ulp where that is larger), LSE max-abs 2e-3,
dQ / dK / dV relative Frobenius 2e-2.
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

# (lens_q, lens_k, H, H_kv, d, causal)
CASES = {
    # ragged lengths around the 128-row tile, one single-token sequence, one empty sequence
    "ragged_d128_causal": ([300, 1, 128, 129, 517, 0], [300, 1, 128, 129, 517, 0], 4, 4, 128, True),
    "ragged_d64_noncausal": ([300, 1, 128, 129, 517, 0], [300, 1, 128, 129, 517, 0], 4, 4, 64, False),
    # fewer queries than keys (key-value-cache alignment), GQA 4
    "cache_gqa_d128": ([200, 64, 1, 300], [450, 64, 257, 300], 8, 2, 128, True),
    # more queries than keys under causal masking: leading queries see no key
    "queries_without_keys_d64": ([300, 5, 7], [100, 0, 7], 2, 1, 64, True),
    "small_heads_d32": ([33, 250, 96], [33, 250, 96], 3, 1, 32, True),
    "small_heads_d16": ([70, 1, 190], [90, 40, 190], 2, 2, 16, False),
    # a sequence with keys but no queries (its dK, dV must be zero)
    "keys_without_queries_d64": ([0, 140, 3], [200, 140, 3], 2, 2, 64, True),
}


def _run(case, seed):
    lq, lk, H, Hkv, d, causal = CASES[case]
    x = workloads.make_varlen_inputs(lq, lk, H, Hkv, d, seed)
    g = {n: t.to(DEV) for n, t in x.items()}
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], g["cu_q"], g["cu_k"], max(lq), max(lk), scale=scale,
                                causal=causal)
    dq, dk, dv = fa2.fa2_bwd_varlen(g["q"], g["k"], g["v"], o, g["dO"], lse, g["cu_q"], g["cu_k"], max(lq),
                                    max(lk), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    return x, scale, causal, o, lse, dq, dk, dv


def _check_lse_with_empty_rows(got, ref):
    empty = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), empty), "rows without visible keys must have LSE = -inf"
    if (~empty).any():
        check_lse(got[~empty], ref[~empty])


@pytest.mark.parametrize("case", sorted(CASES))
def test_varlen_against_oracle(case):
    x, scale, causal, o, lse, dq, dk, dv = _run(case, 700 + len(case))
    ref = oracle.attn_varlen(x["q"], x["k"], x["v"], x["dO"], x["cu_q"], x["cu_k"], scale, causal)
    check_o(to_np(o), ref["O"])
    _check_lse_with_empty_rows(to_np(lse), ref["LSE"])
    check_grad(to_np(dq), ref["dQ"], "dQ")
    check_grad(to_np(dk), ref["dK"], "dK")
    check_grad(to_np(dv), ref["dV"], "dV")
    # rows that see no key: exactly zero output and zero dQ
    empty = np.isneginf(ref["LSE"]).T  # [total_q, H]
    assert np.all(to_np(o)[empty] == 0) and np.all(to_np(dq)[empty] == 0)


def test_varlen_single_sequence_matches_square_kernels():
    # One sequence of N rows is the [1, H, N, d] problem: the forward results
    # and dK, dV must be bit-identical to fa2_fwd / fa2_bwd (same arithmetic,
    # different addressing); dQ sums in a run-dependent order, so it is
    # compared within the gradient tolerance.
    N, H, d = 333, 4, 128
    x = workloads.make_varlen_inputs([N], [N], H, H, d, seed=720)
    g = {n: t.to(DEV) for n, t in x.items()}
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], g["cu_q"], g["cu_k"], N, N, causal=True)
    dq, dk, dv = fa2.fa2_bwd_varlen(g["q"], g["k"], g["v"], o, g["dO"], lse, g["cu_q"], g["cu_k"], N, N,
                                    causal=True)
    sq = {n: g[n].permute(1, 0, 2).unsqueeze(0).contiguous() for n in ("q", "k", "v", "dO")}
    o2, lse2 = fa2.fa2_fwd(sq["q"], sq["k"], sq["v"], causal=True)
    dq2, dk2, dv2 = fa2.fa2_bwd(sq["q"], sq["k"], sq["v"], o2, sq["dO"], lse2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o2[0].permute(1, 0, 2))
    assert torch.equal(lse, lse2[0])
    assert torch.equal(dk, dk2[0].permute(1, 0, 2)) and torch.equal(dv, dv2[0].permute(1, 0, 2))
    check_grad(to_np(dq), to_np(dq2[0].permute(1, 0, 2)), "dQ")


def test_varlen_sequence_order_does_not_matter():
    # Reversing the order of the sequences in the packed batch permutes the
    # outputs and nothing else (each sequence sees only itself).
    lq = [130, 7, 260]
    x = workloads.make_varlen_inputs(lq, lq, 2, 1, 64, seed=721, with_grad=False)
    g = {n: t.to(DEV) for n, t in x.items()}
    cu = x["cu_q"].tolist()
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], g["cu_q"], g["cu_k"], causal=True)
    order = [2, 1, 0]
    rq = torch.cat([g["q"][cu[b]:cu[b + 1]] for b in order])
    rk = torch.cat([g["k"][cu[b]:cu[b + 1]] for b in order])
    rv = torch.cat([g["v"][cu[b]:cu[b + 1]] for b in order])
    rcu = torch.tensor(np.concatenate([[0], np.cumsum([lq[b] for b in order])]), dtype=torch.int32, device=DEV)
    o2, lse2 = fa2.fa2_fwd_varlen(rq, rk, rv, rcu, rcu, causal=True)
    torch.cuda.synchronize()
    rc = rcu.tolist()
    for i, b in enumerate(order):
        assert torch.equal(o[cu[b]:cu[b + 1]], o2[rc[i]:rc[i + 1]])
        assert torch.equal(lse[:, cu[b]:cu[b + 1]], lse2[:, rc[i]:rc[i + 1]])


def test_varlen_bad_offsets_are_reported_not_faulted():
    # Offsets the host cannot see (device memory): a decreasing pair is caught
    # by the kernels' own check, which skips that sequence and sets the device
    # status word to 3; the valid sequence is still computed.
    H, d = 2, 64
    x = workloads.make_varlen_inputs([64, 64], [64, 64], H, H, d, seed=722)
    g = {n: t.to(DEV) for n, t in x.items()}
    bad = torch.tensor([0, 64, 40], dtype=torch.int32, device=DEV)  # second sequence runs backwards
    fa2.fa2_device_status(reset=True)
    o = torch.zeros_like(g["q"])
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], bad, bad, 64, 64, o=o, causal=True)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 3
    ref = oracle.attn_varlen(x["q"][:64], x["k"][:64], x["v"][:64], None, [0, 64], [0, 64], 1 / 8, True)
    check_o(to_np(o[:64]), ref["O"])
    assert torch.count_nonzero(o[64:]) == 0  # the skipped sequence's rows are left untouched


def test_varlen_empty_batch_and_no_keys():
    H, d = 2, 64
    q = torch.zeros(0, H, d, dtype=torch.bfloat16, device=DEV)
    cu0 = torch.zeros(2, dtype=torch.int32, device=DEV)
    o, lse = fa2.fa2_fwd_varlen(q, q, q, cu0, cu0, 0, 0, causal=True)
    assert o.shape == (0, H, d) and lse.shape == (H, 0)
    # queries but no keys anywhere: O = 0, LSE = -inf, dQ = 0
    x = workloads.make_varlen_inputs([5, 3], [0, 0], H, H, d, seed=723)
    g = {n: t.to(DEV) for n, t in x.items()}
    o, lse = fa2.fa2_fwd_varlen(g["q"], g["k"], g["v"], g["cu_q"], g["cu_k"], 5, 0, causal=False)
    dq, dk, dv = fa2.fa2_bwd_varlen(g["q"], g["k"], g["v"], o, g["dO"], lse, g["cu_q"], g["cu_k"], 5, 0,
                                    causal=False)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    assert torch.count_nonzero(o) == 0 and bool(torch.isneginf(lse).all()) and torch.count_nonzero(dq) == 0
