"""Split-KV forward (flash-decoding) with Nq <= Nk, key-value-cache causal
alignment and packed grouped query heads, against the fp64 oracle's
attn_fwd_general (GPU only).  Tolerances as the main forward parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
import tiled_exact_attention_fa2_gb300 as fa2
from parity_util import check_lse, check_o, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

# (B, H, H_kv, Nq, Nk, d, causal, splits)
CASES = [
    (1, 32, 8, 1, 4096, 128, True, 8),     # decode, GQA 4, eight splits
    (2, 8, 1, 1, 1000, 64, True, 3),       # decode, MQA, ragged key tail
    (1, 16, 16, 1, 2048, 128, False, 16),  # decode, plain heads
    (1, 8, 2, 16, 777, 128, True, 4),      # short chunk of queries (speculative / chunked prefill)
    (1, 4, 4, 200, 600, 64, True, 2),      # Nq > 128 rows, two row tiles
    (1, 4, 2, 64, 64, 32, True, 1),        # one split == plain forward
    (1, 2, 1, 3, 300, 16, False, 5),
    (1, 8, 4, 1, 130, 128, True, 64),      # more splits requested than key tiles
    # long caches: many key tiles per split and several units per CTA, so the
    # decode path's double-buffered S runs ahead of slow K/V loads
    (4, 16, 4, 1, 16384, 128, True, 16),
    (1, 8, 2, 1, 65536, 128, True, 16),
    (2, 8, 8, 3, 20000, 64, True, 8),      # several queries per sequence, ragged cache
    # one split: bf16 O straight from the kernel (TMA stores of 32-row boxes
    # that the few packed rows clip)
    (1, 8, 2, 1, 700, 128, True, 1),       # 4 packed rows per K/V head
    (2, 8, 8, 3, 900, 64, False, 1),       # 3 rows per head
    (1, 16, 4, 40, 1000, 128, True, 1),    # 160 rows: a full and a clipped warp block
]


def _ids(c):
    return "B{}H{}kv{}q{}k{}d{}{}s{}".format(*c[:6], "c" if c[6] else "n", c[7])


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_splitkv_against_oracle(case):
    B, H, Hkv, Nq, Nk, d, causal, splits = case
    q = workloads.make_inputs(B, H, Nq, d, seed=600 + Nk, with_grad=False)["q"]
    kv = workloads.make_inputs(B, Hkv, Nk, d, seed=601 + Nk, with_grad=False)
    scale = 1.0 / np.sqrt(d)
    o, lse = fa2.fa2_fwd_splitkv(q.to(DEV), kv["k"].to(DEV), kv["v"].to(DEV), splits, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    ref_o, ref_l = oracle.attn_fwd_general(q, kv["k"], kv["v"], scale, causal)
    check_o(to_np(o), ref_o)
    check_lse(to_np(lse), ref_l)


def test_single_split_equal_lengths_matches_fa2_fwd():
    # Same problem through the split-KV form (P V in bf16 on V) and fa2_fwd
    # (P V in fp16 on an fp16 copy of V): the same LSE bit for bit (the
    # weights' fp32 sums do not depend on their type), O within the parity
    # bound of each other and of the oracle.
    x = workloads.make_inputs(1, 4, 256, 128, seed=9, with_grad=False)
    g = {k: t.to(DEV) for k, t in x.items()}
    o1, l1 = fa2.fa2_fwd(g["q"], g["k"], g["v"], causal=True)
    o2, l2 = fa2.fa2_fwd_splitkv(g["q"], g["k"], g["v"], 1, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)
    ref_o, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], 1 / np.sqrt(128), True)
    check_o(to_np(o1), ref_o, "O fa2_fwd")
    check_o(to_np(o2), ref_o, "O split-KV")
    check_o(to_np(o2), to_np(o1), "O split-KV vs fa2_fwd")


def test_splitkv_rejects_causal_with_more_queries_than_keys():
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(fa2.FA2Error):
        fa2.fa2_fwd_splitkv(q, kv, kv, 2, causal=True)


def test_default_split_count_follows_the_suggestion():
    # num_splits omitted: the binding asks fa2_fwd_splitkv_suggest_splits for
    # this GPU's SM count; the result equals an explicit call with that count.
    B, H, Hkv, Nq, Nk, d = 2, 16, 4, 1, 8192, 128
    q = workloads.make_inputs(B, H, Nq, d, seed=611, with_grad=False)["q"].to(DEV)
    kv = workloads.make_inputs(B, Hkv, Nk, d, seed=612, with_grad=False)
    k, v = kv["k"].to(DEV), kv["v"].to(DEV)
    sms = torch.cuda.get_device_properties(DEV).multi_processor_count
    n = fa2.load_library().fa2_fwd_splitkv_suggest_splits(sms, B, H, Hkv, Nq, Nk)
    assert n >= 1
    o1, l1 = fa2.fa2_fwd_splitkv(q, k, v, causal=True)
    o2, l2 = fa2.fa2_fwd_splitkv(q, k, v, n, causal=True)
    torch.cuda.synchronize()
    assert fa2.fa2_device_status(reset=True) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ref_o, ref_l = oracle.attn_fwd_general(q.cpu(), kv["k"], kv["v"], 1.0 / np.sqrt(d), True)
    check_o(to_np(o1), ref_o)
    check_lse(to_np(l1), ref_l)
