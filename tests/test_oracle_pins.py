"""Pins for the fp64 oracle, independent of the oracle itself (CPU only).

The pages print no worked numerical example of attention, so the oracle is
pinned by what the mathematics fixes: a hand-derived closed form
(tests/golden/hand_cases.json), the N = 1 case, uniform keys (mean of V),
row/gradient invariants, central finite differences of L = sum(O * dO), an
independent brute-force scalar loop, and torch's fp64 CPU attention with
autograd.  ``test_planted_mistakes_are_caught`` plants plausible mistakes in
a copy of the oracle and checks that at least one pin fails for each.
"""
import inspect
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


# ---------------------------------------------------------------------------
# Pins written against an implementation with attn_bwd_head's signature, so
# they can be run on the oracle and on mutated copies of it.
# ---------------------------------------------------------------------------

def _rand(n, d, seed, scale=1.0):
    r = np.random.Generator(np.random.PCG64(seed))
    return [scale * r.standard_normal((n, d)) for _ in range(4)]


def pin_hand_case(impl):
    g = json.load(open(GOLDEN))
    x = {k: np.array(v, dtype=np.float64) for k, v in g["inputs"].items() if k != "scale"}
    for mode in ("noncausal", "causal"):
        r = impl(x["q"], x["k"], x["v"], x["dO"], g["inputs"]["scale"], mode == "causal")
        for key, want in g[mode].items():
            np.testing.assert_allclose(r[key], np.array(want), rtol=0, atol=1e-12,
                                       err_msg=f"{mode} {key}")


def pin_single_key(impl):
    # N = 1: the only key has weight 1, so O = V_0, LSE = s q.k, dV = dO, dQ = dK = 0.
    for causal in (False, True):
        for d in (1, 3, 16):
            q, k, v, dO = _rand(1, d, 11 + d)
            s = 0.37
            r = impl(q, k, v, dO, s, causal)
            np.testing.assert_allclose(r["O"], v, atol=1e-14)
            np.testing.assert_allclose(r["LSE"], [s * float(q[0] @ k[0])], atol=1e-14)
            np.testing.assert_allclose(r["dV"], dO, atol=1e-14)
            np.testing.assert_allclose(r["dQ"], 0, atol=1e-14)
            np.testing.assert_allclose(r["dK"], 0, atol=1e-14)


def pin_uniform_keys(impl):
    # All K rows equal: every visible key gets the same weight, so O_i is the
    # mean of the visible V rows, LSE_i = s q_i.k + ln(#visible) and dQ = 0.
    N, d, s = 9, 5, 0.4
    q, _, v, dO = _rand(N, d, 21)
    krow = np.random.Generator(np.random.PCG64(22)).standard_normal(d)
    k = np.tile(krow, (N, 1))
    for causal in (False, True):
        r = impl(q, k, v, dO, s, causal)
        for i in range(N):
            vis = i + 1 if causal else N
            np.testing.assert_allclose(r["O"][i], v[:vis].mean(axis=0), atol=1e-12)
            np.testing.assert_allclose(r["LSE"][i], s * q[i] @ krow + math.log(vis), atol=1e-12)
        np.testing.assert_allclose(r["dQ"], 0, atol=1e-12)


def pin_zero_query(impl):
    # Q = 0 makes every score 0: uniform weights regardless of K.
    N, d, s = 7, 3, 0.9
    _, k, v, dO = _rand(N, d, 31)
    q = np.zeros((N, d))
    for causal in (False, True):
        r = impl(q, k, v, dO, s, causal)
        for i in range(N):
            vis = i + 1 if causal else N
            np.testing.assert_allclose(r["O"][i], v[:vis].mean(axis=0), atol=1e-12)
            np.testing.assert_allclose(r["LSE"][i], math.log(vis), atol=1e-12)


def pin_gradient_invariants(impl):
    # Rows of P sum to 1 => rows of dS sum to 0 => sum_j dK_j = 0 and
    # sum_j dV_j = sum_i dO_i.
    N, d, s = 13, 6, 0.5
    q, k, v, dO = _rand(N, d, 41)
    for causal in (False, True):
        r = impl(q, k, v, dO, s, causal)
        np.testing.assert_allclose(r["dK"].sum(axis=0), 0, atol=1e-12)
        np.testing.assert_allclose(r["dV"].sum(axis=0), dO.sum(axis=0), atol=1e-12)


def pin_shift_invariance(impl):
    # K -> K + 1 c^T leaves O unchanged and shifts LSE_i by s q_i.c;
    # V -> V + 1 c^T shifts O by c.
    N, d, s = 10, 4, 0.6
    q, k, v, dO = _rand(N, d, 51)
    c = np.random.Generator(np.random.PCG64(52)).standard_normal(d)
    for causal in (False, True):
        r0 = impl(q, k, v, dO, s, causal)
        r1 = impl(q, k + c, v, dO, s, causal)
        np.testing.assert_allclose(r1["O"], r0["O"], atol=1e-12)
        np.testing.assert_allclose(r1["LSE"], r0["LSE"] + s * (q @ c), atol=1e-12)
        r2 = impl(q, k, v + c, dO, s, causal)
        np.testing.assert_allclose(r2["O"], r0["O"] + c, atol=1e-12)


def pin_key_permutation(impl):
    # Non-causal attention is invariant to a joint permutation of K and V rows,
    # and dK, dV permute with them.
    N, d, s = 11, 4, 0.7
    q, k, v, dO = _rand(N, d, 61)
    perm = np.random.Generator(np.random.PCG64(62)).permutation(N)
    r0 = impl(q, k, v, dO, s, False)
    r1 = impl(q, k[perm], v[perm], dO, s, False)
    np.testing.assert_allclose(r1["O"], r0["O"], atol=1e-12)
    np.testing.assert_allclose(r1["dQ"], r0["dQ"], atol=1e-12)
    np.testing.assert_allclose(r1["dK"], r0["dK"][perm], atol=1e-12)
    np.testing.assert_allclose(r1["dV"], r0["dV"][perm], atol=1e-12)


def pin_finite_differences(impl):
    # Central differences of L = sum(O * dO) against the analytic gradients.
    h = 1e-6
    for causal in (False, True):
        for (N, d, seed) in ((5, 3, 71), (8, 4, 72), (2, 1, 73)):
            q, k, v, dO = _rand(N, d, seed)
            s = 0.8
            r = impl(q, k, v, dO, s, causal)

            def loss(qq, kk, vv):
                return float((impl(qq, kk, vv, dO, s, causal)["O"] * dO).sum())

            for name, grad in (("q", r["dQ"]), ("k", r["dK"]), ("v", r["dV"])):
                fd = np.zeros_like(grad)
                for idx in np.ndindex(*grad.shape):
                    args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                    args[name][idx] += h
                    lp = loss(args["q"], args["k"], args["v"])
                    args[name][idx] -= 2 * h
                    lm = loss(args["q"], args["k"], args["v"])
                    fd[idx] = (lp - lm) / (2 * h)
                err = np.abs(fd - grad).max() / max(1.0, np.abs(grad).max())
                assert err < 1e-7, (name, causal, N, d, err)


def _brute_force(q, k, v, dO, s, causal):
    """Scalar-loop attention written independently of the oracle (pure Python).

    len(q) queries, len(k) keys; with causal masking query i sees key j iff
    j <= i + len(k) - len(q).  A query that sees nothing gets O = 0, LSE = -inf.
    """
    N, Nk, d = len(q), len(k), len(q[0])
    off = Nk - N
    O = [[0.0] * d for _ in range(N)]
    LSE = [-math.inf] * N
    P = [[0.0] * Nk for _ in range(N)]
    for i in range(N):
        vis = [j for j in range(Nk) if (not causal or j <= i + off)]
        if not vis:
            continue
        logits = {j: s * sum(q[i][c] * k[j][c] for c in range(d)) for j in vis}
        top = max(logits.values())
        tot = sum(math.exp(x - top) for x in logits.values())
        LSE[i] = top + math.log(tot)
        for j in vis:
            P[i][j] = math.exp(logits[j] - LSE[i])
        for c in range(d):
            O[i][c] = sum(P[i][j] * v[j][c] for j in vis)
    dQ = [[0.0] * d for _ in range(N)]
    dK = [[0.0] * d for _ in range(Nk)]
    dV = [[0.0] * d for _ in range(Nk)]
    for i in range(N):
        # dL/dlogit_ij = p_ij * dO_i . (v_j - O_i)
        for j in range(Nk):
            if P[i][j] == 0.0:
                continue
            g = P[i][j] * sum(dO[i][c] * (v[j][c] - O[i][c]) for c in range(d))
            for c in range(d):
                dQ[i][c] += s * g * k[j][c]
                dK[j][c] += s * g * q[i][c]
                dV[j][c] += P[i][j] * dO[i][c]
    return {"O": np.array(O), "LSE": np.array(LSE), "dQ": np.array(dQ),
            "dK": np.array(dK), "dV": np.array(dV)}


def pin_brute_force(impl):
    N, d, s = 12, 5, 0.45
    q, k, v, dO = _rand(N, d, 81, scale=1.5)
    for causal in (False, True):
        want = _brute_force(q.tolist(), k.tolist(), v.tolist(), dO.tolist(), s, causal)
        got = impl(q, k, v, dO, s, causal)
        for key in want:
            np.testing.assert_allclose(got[key], want[key], rtol=1e-11, atol=1e-12, err_msg=key)


def pin_torch_sdpa(impl):
    # Library special case: torch fp64 CPU attention + autograd.
    N, d, s = 17, 8, 0.3
    q, k, v, dO = _rand(N, d, 91)
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
        o = torch.nn.functional.scaled_dot_product_attention(
            tq[None, None], tk[None, None], tv[None, None], is_causal=causal, scale=s)[0, 0]
        (o * torch.tensor(dO)).sum().backward()
        logits = s * (torch.tensor(q) @ torch.tensor(k).T)
        if causal:
            logits = logits.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        lse = torch.logsumexp(logits, dim=1)
        r = impl(q, k, v, dO, s, causal)
        np.testing.assert_allclose(r["O"], o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(r["LSE"], lse.numpy(), atol=1e-12)
        np.testing.assert_allclose(r["dQ"], tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(r["dK"], tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(r["dV"], tv.grad.numpy(), atol=1e-12)


PINS = [pin_hand_case, pin_single_key, pin_uniform_keys, pin_zero_query,
        pin_gradient_invariants, pin_shift_invariance, pin_key_permutation,
        pin_finite_differences, pin_brute_force, pin_torch_sdpa]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_head_pins(pin):
    pin(oracle.attn_bwd_head)


# ---------------------------------------------------------------------------
# Batched entry points agree with the per-head function and with each other.
# ---------------------------------------------------------------------------

def test_batched_matches_per_head_and_rows():
    w = workloads.WORKLOADS["tiny"]
    x = workloads.workload_inputs(w)
    for causal in (True, False):
        full = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], w.scale, causal)
        O, L = oracle.attn_fwd(x["q"], x["k"], x["v"], w.scale, causal)
        np.testing.assert_array_equal(O, full["O"])
        np.testing.assert_array_equal(L, full["LSE"])
        rows = workloads.sample_rows(w.N, 9, 5)
        rr = oracle.attn_rows(x["q"], x["k"], x["v"], x["dO"], w.scale, causal, rows)
        for key in ("O", "LSE", "D", "dQ"):
            np.testing.assert_allclose(rr[key], full[key][:, :, rows], rtol=1e-12, atol=1e-12)


def test_tiny_workload_against_brute_force_and_probability_rows():
    # The tiny workload end to end (bf16 inputs widened to fp64) against the
    # scalar loop, plus: every probability row sums to one.
    w = workloads.WORKLOADS["tiny"]
    x = workloads.workload_inputs(w)
    q, k, v, dO = (oracle.as_f64(x[n])[0, 0][:24, :8] for n in ("q", "k", "v", "dO"))
    s = oracle.fp32_scale(w.scale)
    for causal in (True, False):
        want = _brute_force(q.tolist(), k.tolist(), v.tolist(), dO.tolist(), s, causal)
        got = oracle.attn_bwd_head(q, k, v, dO, s, causal)
        for key in want:
            np.testing.assert_allclose(got[key], want[key], rtol=1e-11, atol=1e-12)
        _, _, P = oracle.attn_fwd_head(q, k, v, s, causal)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
        if causal:
            assert np.all(np.triu(P, 1) == 0)


def test_lse_matches_library_logsumexp_large_logits():
    # Large logits (the stress workload's x3 scaling and beyond): the stable
    # LSE equals scipy's logsumexp and never overflows.
    from scipy.special import logsumexp
    r = np.random.Generator(np.random.PCG64(3))
    S = 40.0 * r.standard_normal((16, 33))
    np.testing.assert_allclose(oa.row_logsumexp(S), logsumexp(S, axis=1), rtol=0, atol=1e-12)
    S[3, :] = -np.inf
    assert oa.row_logsumexp(S)[3] == -np.inf


def test_fp32_scale_is_what_the_gpu_receives():
    assert oracle.fp32_scale(1 / math.sqrt(128)) == float(np.float32(1 / math.sqrt(128)))
    assert oracle.fp32_scale(0.1) != 0.1


# ---------------------------------------------------------------------------
# Planted mistakes: each mutant of the oracle must fail at least one pin.
# ---------------------------------------------------------------------------

MUTANTS = {
    "dropped_D_term": ("dS = P * (dP - D[:, None])", "dS = P * dP"),
    "flipped_dS_sign": ("dS = P * (dP - D[:, None])", "dS = P * (D[:, None] - dP)"),
    "transposed_dK": ("dK = scale * (dS.T @ q)", "dK = scale * (dS @ q)"),
    "dQ_missing_scale": ("dQ = scale * (dS @ k)", "dQ = dS @ k"),
    "dV_not_transposed": ("dV = P.T @ dO", "dV = P @ dO"),
    "D_from_dO_only": ("D = (dO * O).sum(axis=1)", "D = dO.sum(axis=1)"),
    "dP_wrong_operand": ("dP = dO @ v.T", "dP = dO @ k.T"),
}

FWD_MUTANTS = {
    "mask_hides_diagonal": ("np.where(j > i, -np.inf, S)", "np.where(j >= i, -np.inf, S)"),
    "mask_off_by_one_late": ("np.where(j > i, -np.inf, S)", "np.where(j > i + 1, -np.inf, S)"),
    "scale_applied_twice": ("return scale * (q @ k.T)", "return scale * scale * (q @ k.T)"),
    "lse_in_base_2": ("m_safe + np.log(s)", "m_safe + np.log2(s)"),
    "lse_without_max": ("m_safe + np.log(s)", "np.log(s)"),
}


def _mutant_module(src_fn_names, old, new):
    """Copy oracle.attention into a fresh module with one textual mistake planted."""
    src = inspect.getsource(oa)
    assert src.count(old) == 1, f"mutation target not unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS) + sorted(FWD_MUTANTS))
def test_planted_mistakes_are_caught(name):
    old, new = MUTANTS.get(name) or FWD_MUTANTS[name]
    mod = _mutant_module(None, old, new)
    failed = []
    for pin in PINS:
        try:
            pin(mod.attn_bwd_head)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught planted mistake {name}"


# ---------------------------------------------------------------------------
# Grouped-query attention (K/V heads shared by groups of query heads).
# ---------------------------------------------------------------------------

def test_gqa_with_one_query_head_per_group_is_plain_attention():
    x = workloads.make_inputs(2, 3, 17, 8, seed=301)
    for causal in (True, False):
        a = oracle.attn_bwd_gqa(x["q"], x["k"], x["v"], x["dO"], 0.35, causal)
        b = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dO"], 0.35, causal)
        for key in a:
            np.testing.assert_allclose(a[key], b[key], rtol=0, atol=1e-13)


def test_gqa_equals_attention_on_repeated_kv_with_summed_gradients():
    # Independent construction: repeat each K/V head G times (a library
    # routine, np.repeat), run plain attention on the repeated tensors with
    # torch's fp64 autograd, and sum the K/V gradients back over each group.
    B, H, Hkv, N, d = 1, 6, 2, 13, 4
    r = np.random.Generator(np.random.PCG64(302))
    q, dO = r.standard_normal((B, H, N, d)), r.standard_normal((B, H, N, d))
    k, v = r.standard_normal((B, Hkv, N, d)), r.standard_normal((B, Hkv, N, d))
    G = H // Hkv
    for causal in (True, False):
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        kr = tk.repeat_interleave(G, dim=1)
        vr = tv.repeat_interleave(G, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(tq, kr, vr, is_causal=causal, scale=0.5)
        (o * torch.tensor(dO)).sum().backward()
        got = oracle.attn_bwd_gqa(q, k, v, dO, 0.5, causal)
        np.testing.assert_allclose(got["O"], o.detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(got["dQ"], tq.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(got["dK"], tk.grad.numpy(), atol=1e-12)
        np.testing.assert_allclose(got["dV"], tv.grad.numpy(), atol=1e-12)


def test_gqa_finite_differences_through_shared_kv():
    # dL/dK and dL/dV of a shared head collect every query head of its group.
    B, H, Hkv, N, d, s, h = 1, 4, 1, 5, 3, 0.7, 1e-6
    r = np.random.Generator(np.random.PCG64(303))
    q, dO = r.standard_normal((B, H, N, d)), r.standard_normal((B, H, N, d))
    k, v = r.standard_normal((B, Hkv, N, d)), r.standard_normal((B, Hkv, N, d))
    for causal in (True, False):
        g = oracle.attn_bwd_gqa(q, k, v, dO, s, causal)

        def loss(kk, vv):
            return float((oracle.attn_bwd_gqa(q, kk, vv, dO, s, causal)["O"] * dO).sum())

        for name, grad in (("k", g["dK"]), ("v", g["dV"])):
            fd = np.zeros_like(grad)
            for idx in np.ndindex(*grad.shape):
                args = {"k": k.copy(), "v": v.copy()}
                args[name][idx] += h
                lp = loss(args["k"], args["v"])
                args[name][idx] -= 2 * h
                lm = loss(args["k"], args["v"])
                fd[idx] = (lp - lm) / (2 * h)
            assert np.abs(fd - grad).max() < 1e-7 * max(1.0, np.abs(grad).max()), name


# ---------------------------------------------------------------------------
# Separate query / key lengths (key-value-cache alignment) and grouped heads.
# ---------------------------------------------------------------------------

def test_general_forward_equal_lengths_is_plain_attention():
    x = workloads.make_inputs(1, 2, 40, 8, seed=501, with_grad=False)
    for causal in (True, False):
        a = oracle.attn_fwd_general(x["q"], x["k"], x["v"], 0.3, causal)
        b = oracle.attn_fwd(x["q"], x["k"], x["v"], 0.3, causal)
        np.testing.assert_allclose(a[0], b[0], atol=1e-13)
        np.testing.assert_allclose(a[1], b[1], atol=1e-13)


def test_general_forward_is_suffix_of_square_causal_problem():
    # With Nq < Nk the queries are the last Nq positions: embedding them at the
    # end of a full-length query block and running square causal attention
    # must give the same rows.
    r = np.random.Generator(np.random.PCG64(502))
    Nk, Nq, d = 23, 5, 6
    k, v = r.standard_normal((1, 1, Nk, d)), r.standard_normal((1, 1, Nk, d))
    full_q = r.standard_normal((1, 1, Nk, d))
    q = full_q[:, :, Nk - Nq:]
    o, lse = oracle.attn_fwd_general(q, k, v, 0.6, True)
    o_full, lse_full = oracle.attn_fwd(full_q, k, v, 0.6, True)
    np.testing.assert_allclose(o, o_full[:, :, Nk - Nq:], atol=1e-12)
    np.testing.assert_allclose(lse, lse_full[:, :, Nk - Nq:], atol=1e-12)


def test_general_forward_against_torch_with_explicit_mask_and_groups():
    r = np.random.Generator(np.random.PCG64(503))
    B, H, Hkv, Nq, Nk, d = 2, 6, 3, 4, 19, 8
    q = r.standard_normal((B, H, Nq, d))
    k, v = r.standard_normal((B, Hkv, Nk, d)), r.standard_normal((B, Hkv, Nk, d))
    kr = torch.tensor(k).repeat_interleave(H // Hkv, dim=1)
    vr = torch.tensor(v).repeat_interleave(H // Hkv, dim=1)
    for causal in (True, False):
        mask = None
        if causal:
            mask = torch.tensor(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq))
        # 0.375 is exact in fp32, so the oracle's fp32 scale equals torch's
        o = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q), kr, vr, attn_mask=mask, scale=0.375)
        got, _ = oracle.attn_fwd_general(q, k, v, 0.375, causal)
        np.testing.assert_allclose(got, o.numpy(), atol=1e-12)


def test_single_query_decode_sees_every_key():
    # Nq = 1 with causal masking: the one query is the last position and sees
    # all Nk keys, so causal and non-causal agree.
    x = workloads.make_inputs(1, 2, 1, 16, seed=504, with_grad=False)
    kv = workloads.make_inputs(1, 2, 33, 16, seed=505, with_grad=False)
    a = oracle.attn_fwd_general(x["q"], kv["k"], kv["v"], 0.25, True)
    b = oracle.attn_fwd_general(x["q"], kv["k"], kv["v"], 0.25, False)
    np.testing.assert_allclose(a[0], b[0], atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], atol=1e-14)


# ---------------------------------------------------------------------------
# Variable-length batches (packed [total, H, d], cu_seqlens offsets).
# ---------------------------------------------------------------------------

# (lens_q, lens_k) mixes: ragged, equal, Lq < Lk (cache alignment), Lq > Lk
# (leading queries see nothing under causal masking) and empty sequences.
VARLEN_CASES = {
    "mixed": ([5, 1, 9, 3], [5, 7, 9, 2]),
    "with_empty": ([0, 4, 3], [3, 0, 6]),
}


def _varlen_inputs(case, H, Hkv, d, seed):
    lq, lk = VARLEN_CASES[case]
    return workloads.make_varlen_inputs(lq, lk, H, Hkv, d, seed)


def pin_varlen_brute_force(fn):
    # Each sequence and head against the pure-Python scalar loop, with K/V
    # head h // G and K/V gradients summed over the group by hand.
    for case in VARLEN_CASES:
        for causal in (True, False):
            x = _varlen_inputs(case, 4, 2, 3, 611)
            q, k, v, dO = (oa.as_f64(x[n]) for n in ("q", "k", "v", "dO"))
            cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
            got = fn(x["q"], x["k"], x["v"], x["dO"], cq, ck, 0.625, causal)
            dK = np.zeros_like(k)
            dV = np.zeros_like(v)
            for b in range(len(cq) - 1):
                for h in range(4):
                    hk = h // 2
                    sq, sk = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
                    if cq[b + 1] == cq[b]:
                        continue
                    if ck[b + 1] == ck[b]:
                        np.testing.assert_allclose(got["O"][sq, h], 0, atol=0)
                        assert np.all(got["LSE"][h, sq] == -np.inf)
                        continue
                    w = _brute_force(q[sq, h].tolist(), k[sk, hk].tolist(), v[sk, hk].tolist(),
                                     dO[sq, h].tolist(), 0.625, causal)
                    np.testing.assert_allclose(got["O"][sq, h], w["O"], atol=1e-12)
                    np.testing.assert_allclose(got["LSE"][h, sq], w["LSE"], atol=1e-12)
                    np.testing.assert_allclose(got["dQ"][sq, h], w["dQ"], atol=1e-12)
                    dK[sk, hk] += w["dK"]
                    dV[sk, hk] += w["dV"]
            np.testing.assert_allclose(got["dK"], dK, atol=1e-12)
            np.testing.assert_allclose(got["dV"], dV, atol=1e-12)


def pin_varlen_torch_autograd(fn):
    # Library special case: per sequence, torch fp64 attention with an explicit
    # bottom-right causal mask on the repeated K/V heads, plus autograd.
    lq, lk = [6, 2, 7], [9, 2, 7]  # every query sees at least one key
    x = workloads.make_varlen_inputs(lq, lk, 6, 3, 5, seed=612)
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    for causal in (True, False):
        got = fn(x["q"], x["k"], x["v"], x["dO"], cq, ck, 0.375, causal)
        for b in range(3):
            tq = x["q"][cq[b]:cq[b + 1]].double().permute(1, 0, 2).clone().requires_grad_(True)
            tk = x["k"][ck[b]:ck[b + 1]].double().permute(1, 0, 2).clone().requires_grad_(True)
            tv = x["v"][ck[b]:ck[b + 1]].double().permute(1, 0, 2).clone().requires_grad_(True)
            g = x["dO"][cq[b]:cq[b + 1]].double().permute(1, 0, 2)
            Lq, Lk = lq[b], lk[b]
            mask = None
            if causal:
                mask = torch.tensor(np.arange(Lk)[None, :] <= np.arange(Lq)[:, None] + (Lk - Lq))
            o = torch.nn.functional.scaled_dot_product_attention(
                tq, tk.repeat_interleave(2, dim=0), tv.repeat_interleave(2, dim=0), attn_mask=mask, scale=0.375)
            (o * g).sum().backward()
            sl, kl = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
            np.testing.assert_allclose(got["O"][sl], o.detach().permute(1, 0, 2).numpy(), atol=1e-12)
            np.testing.assert_allclose(got["dQ"][sl], tq.grad.permute(1, 0, 2).numpy(), atol=1e-12)
            np.testing.assert_allclose(got["dK"][kl], tk.grad.permute(1, 0, 2).numpy(), atol=1e-12)
            np.testing.assert_allclose(got["dV"][kl], tv.grad.permute(1, 0, 2).numpy(), atol=1e-12)


def pin_varlen_rows_without_keys(fn):
    # Lq = 5 queries, Lk = 2 keys, causal: queries 0..2 see nothing (O = 0,
    # LSE = -inf, dQ = 0); query 3 sees key 0 only (O = V_0, LSE = s q.k_0).
    x = workloads.make_varlen_inputs([5], [2], 1, 1, 4, seed=613)
    got = fn(x["q"], x["k"], x["v"], x["dO"], [0, 5], [0, 2], 0.5, True)
    q, k, v = (oa.as_f64(x[n]) for n in ("q", "k", "v"))
    np.testing.assert_allclose(got["O"][:3], 0, atol=0)
    assert np.all(got["LSE"][0, :3] == -np.inf)
    np.testing.assert_allclose(got["dQ"][:3], 0, atol=0)
    np.testing.assert_allclose(got["O"][3, 0], v[0, 0], atol=1e-14)
    np.testing.assert_allclose(got["LSE"][0, 3], 0.5 * float(q[3, 0] @ k[0, 0]), atol=1e-14)


def pin_varlen_sequences_are_independent(fn):
    # Changing one sequence's inputs leaves every other sequence's outputs
    # and gradients bit-identical.
    x = _varlen_inputs("mixed", 2, 1, 4, 614)
    cq, ck = x["cu_q"].tolist(), x["cu_k"].tolist()
    a = fn(x["q"], x["k"], x["v"], x["dO"], cq, ck, 0.5, True)
    y = {n: x[n].clone() for n in ("q", "k", "v", "dO")}
    y["q"][cq[1]:cq[2]] *= -2
    y["k"][ck[1]:ck[2]] += 1
    y["v"][ck[1]:ck[2]] *= 3
    b = fn(y["q"], y["k"], y["v"], y["dO"], cq, ck, 0.5, True)
    for key, rows in (("O", cq), ("dQ", cq), ("dK", ck), ("dV", ck)):
        for s0 in (0, 2, 3):
            np.testing.assert_array_equal(a[key][rows[s0]:rows[s0 + 1]], b[key][rows[s0]:rows[s0 + 1]])
    assert not np.array_equal(a["O"][cq[1]:cq[2]], b["O"][cq[1]:cq[2]])


def pin_varlen_finite_differences(fn):
    # Central differences of L = sum(O * dO) with respect to every entry of
    # Q, K, V of a tiny packed batch (GQA, Lq != Lk, causal).
    lq, lk = [3, 2], [4, 2]
    r = np.random.Generator(np.random.PCG64(615))
    q = r.standard_normal((5, 2, 2))
    k = r.standard_normal((6, 1, 2))
    v = r.standard_normal((6, 1, 2))
    dO = r.standard_normal((5, 2, 2))
    cq, ck, s, h = [0, 3, 5], [0, 4, 6], 0.8, 1e-6
    g = fn(q, k, v, dO, cq, ck, s, True)

    def loss(qq, kk, vv):
        return float((fn(qq, kk, vv, None, cq, ck, s, True)["O"] * dO).sum())

    for name, grad in (("q", g["dQ"]), ("k", g["dK"]), ("v", g["dV"])):
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
            args[name][idx] += h
            lp = loss(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * h
            lm = loss(args["q"], args["k"], args["v"])
            fd[idx] = (lp - lm) / (2 * h)
        assert np.abs(fd - grad).max() < 1e-7 * max(1.0, np.abs(grad).max()), name


VARLEN_PINS = [pin_varlen_brute_force, pin_varlen_torch_autograd, pin_varlen_rows_without_keys,
               pin_varlen_sequences_are_independent, pin_varlen_finite_differences]


@pytest.mark.parametrize("pin", VARLEN_PINS, ids=lambda p: p.__name__)
def test_varlen_oracle_pins(pin):
    pin(oracle.attn_varlen)


def test_varlen_equal_lengths_is_batched_attention():
    # All sequences of one length N: the packed batch is the [B, H, N, d]
    # problem with the sequence and head axes swapped.
    x = workloads.make_varlen_inputs([24, 24], [24, 24], 4, 2, 8, seed=616)
    q, k, v, dO = (x[n].reshape(2, 24, -1, 8).permute(0, 2, 1, 3) for n in ("q", "k", "v", "dO"))
    for causal in (True, False):
        got = oracle.attn_varlen(x["q"], x["k"], x["v"], x["dO"], x["cu_q"], x["cu_k"], 0.3, causal)
        want = oracle.attn_bwd_gqa(q, k, v, dO, 0.3, causal)
        np.testing.assert_allclose(got["O"], want["O"].transpose(0, 2, 1, 3).reshape(48, 4, 8), atol=1e-13)
        np.testing.assert_allclose(got["LSE"], want["LSE"].transpose(1, 0, 2).reshape(4, 48), atol=1e-13)
        np.testing.assert_allclose(got["dK"], want["dK"].transpose(0, 2, 1, 3).reshape(48, 2, 8), atol=1e-13)


VARLEN_MUTANTS = {
    "top_left_alignment": ("S = np.where(j > i + (Lk - Lq), -np.inf, S)\n            lse = row_logsumexp(S)\n            P",
                           "S = np.where(j > i, -np.inf, S)\n            lse = row_logsumexp(S)\n            P"),
    "offset_sign": ("S = np.where(j > i + (Lk - Lq), -np.inf, S)\n            lse = row_logsumexp(S)\n            P",
                    "S = np.where(j > i - (Lk - Lq), -np.inf, S)\n            lse = row_logsumexp(S)\n            P"),
    "head_group_modulo": ("            hk = h // G\n            S = scores(q[q0:q1, h]",
                          "            hk = h % Hkv\n            S = scores(q[q0:q1, h]"),
    "dK_overwritten": ('out["dK"][k0:k1, hk] += s', 'out["dK"][k0:k1, hk] = s'),
    "dQ_wrong_keys": ('out["dQ"][q0:q1, h] = s * (dS @ k[k0:k1, hk])', 'out["dQ"][q0:q1, h] = s * (dS @ k[q0:q0 + Lk, hk])'),
}


@pytest.mark.parametrize("name", sorted(VARLEN_MUTANTS))
def test_varlen_planted_mistakes_are_caught(name):
    old, new = VARLEN_MUTANTS[name]
    mod = _mutant_module(None, old, new)
    failed = []
    for pin in VARLEN_PINS:
        try:
            pin(mod.attn_varlen)
        except (AssertionError, ValueError, FloatingPointError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught planted mistake {name}"
