"""fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, header, table or helper with the CUDA path.

What it computes.  The article "Revolutionizing Web-Based AI: How a Plain
JavaScript Prototype Paved the Way for High-Performance WebGPU Flash
Attention 2" (section "Translating to WGSL and Optimizing Passes") describes a
blocked forward pass that keeps an online-softmax state and never stores the
N x N attention matrix, and a backward pass that recomputes the attention
weights from Q, K and the saved log-sum-exp.  Both are exact reorganisations
of plain softmax attention, so the oracle is that plain definition written out
in fp64, one (batch, head) at a time, with the N x N score matrix
materialised:

    S   = scale * Q K^T                 (S[i, j] = -inf where j > i if causal)
    LSE = m + ln sum_j exp(S[:, j] - m),  m = max_j S[:, j]   (natural log)
    P   = exp(S - LSE)                  (each row sums to 1)
    O   = P V
    D   = rowsum(dO * O)
    dV  = P^T dO
    dP  = dO V^T
    dS  = P * (dP - D)
    dQ  = scale * dS K
    dK  = scale * dS^T Q

Readings where the pages are silent (each is stated again where it is used):
  * causal means key j is visible to query i iff j <= i (N_q = N_k);
  * LSE is the natural-log log-sum-exp of the *scaled*, masked scores;
  * a row with no visible key (impossible for N_q = N_k causal) has O = 0,
    LSE = -inf and zero gradients;
  * inputs are the bf16 values the GPU receives, widened exactly to fp64, and
    the scale is the fp32 value the GPU receives, widened to fp64;
  * separate query / key lengths (attn_fwd_general, attn_varlen) align the
    queries with the end of the keys (key-value-cache alignment): query i
    sees key j iff j <= i + Nk - Nq under causal masking;
  * a variable-length batch (attn_varlen) is packed [total, H, d] with
    cu_seqlens offsets, LSE [H, total_q]; sequences never see each other.

Every function here is pinned by tests/test_oracle_pins.py against closed
forms, invariants, central finite differences, a brute-force scalar loop and
torch's fp64 CPU attention + autograd.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64", "fp32_scale", "scores", "apply_causal_mask", "row_logsumexp",
    "attn_fwd_head", "attn_bwd_head", "attn_fwd", "attn_bwd", "attn_rows",
    "attn_bwd_gqa", "attn_fwd_general", "attn_varlen",
]


def as_f64(x) -> np.ndarray:
    """Widen a torch tensor (any float dtype, incl. bf16) or array to fp64 numpy."""
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(device="cpu", dtype=torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def fp32_scale(scale: float) -> float:
    """The softmax scale exactly as an fp32 argument carries it, widened to fp64."""
    return float(np.float32(scale))


def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for one head: q [Nq, d], k [Nk, d] -> [Nq, Nk]."""
    return scale * (q @ k.T)


def apply_causal_mask(S: np.ndarray) -> np.ndarray:
    """Set S[i, j] = -inf where key j lies after query i (j > i)."""
    nq, nk = S.shape
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return np.where(j > i, -np.inf, S)


def row_logsumexp(S: np.ndarray) -> np.ndarray:
    """ln sum_j exp(S[i, j]) per row, shifted by the row max for stability.

    A row whose entries are all -inf gets -inf.
    """
    m = S.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    s = np.exp(S - m_safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        return np.where(finite, m_safe + np.log(s), -np.inf)


def _probabilities(S: np.ndarray, lse: np.ndarray) -> np.ndarray:
    """P = exp(S - LSE); rows with LSE = -inf (nothing visible) are all zero."""
    finite = np.isfinite(lse)
    P = np.exp(S - np.where(finite, lse, 0.0)[:, None])
    return np.where(finite[:, None], P, 0.0)


def attn_fwd_head(q, k, v, scale: float, causal: bool):
    """Forward pass for one head.  Returns (O [N, d], LSE [N], P [N, N])."""
    S = scores(q, k, scale)
    if causal:
        S = apply_causal_mask(S)
    lse = row_logsumexp(S)
    P = _probabilities(S, lse)
    O = P @ v
    return O, lse, P


def attn_bwd_head(q, k, v, dO, scale: float, causal: bool):
    """Forward + backward for one head, gradients of L = sum(O * dO).

    Returns a dict with O, LSE, D, dQ, dK, dV (fp64).
    """
    O, lse, P = attn_fwd_head(q, k, v, scale, causal)
    D = (dO * O).sum(axis=1)
    dV = P.T @ dO
    dP = dO @ v.T
    dS = P * (dP - D[:, None])
    dQ = scale * (dS @ k)
    dK = scale * (dS.T @ q)
    return {"O": O, "LSE": lse, "D": D, "dQ": dQ, "dK": dK, "dV": dV}


def attn_fwd(q, k, v, scale: float, causal: bool):
    """Forward over [B, H, N, d] inputs.  Returns (O [B,H,N,d], LSE [B,H,N]) in fp64."""
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    s = fp32_scale(scale)
    B, H, N, d = q.shape
    O = np.empty((B, H, N, d))
    L = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h], _ = attn_fwd_head(q[b, h], k[b, h], v[b, h], s, causal)
    return O, L


def attn_bwd(q, k, v, dO, scale: float, causal: bool, heads=None):
    """Forward + backward over [B, H, N, d] inputs, fp64.

    ``heads`` optionally restricts the work to a list of (b, h) pairs; entries
    of the returned arrays for other heads are NaN.  Returns a dict with
    O, LSE, D, dQ, dK, dV.
    """
    q, k, v, dO = as_f64(q), as_f64(k), as_f64(v), as_f64(dO)
    s = fp32_scale(scale)
    B, H, N, d = q.shape
    out = {
        "O": np.full((B, H, N, d), np.nan), "LSE": np.full((B, H, N), np.nan),
        "D": np.full((B, H, N), np.nan), "dQ": np.full((B, H, N, d), np.nan),
        "dK": np.full((B, H, N, d), np.nan), "dV": np.full((B, H, N, d), np.nan),
    }
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        r = attn_bwd_head(q[b, h], k[b, h], v[b, h], dO[b, h], s, causal)
        for key, val in r.items():
            out[key][b, h] = val
    return out


def attn_rows(q, k, v, dO, scale: float, causal: bool, rows):
    """O, LSE, D and dQ at a chosen set of query rows, for every (b, h).

    Each query row's outputs depend only on that row of Q and dO and on all
    of K and V, so this is the same definition as ``attn_bwd`` restricted to
    the rows in ``rows`` (a 1-D integer array).  Returns a dict of arrays
    shaped [B, H, len(rows)(, d)].
    """
    q, k, v, dO = as_f64(q), as_f64(k), as_f64(v), as_f64(dO)
    s = fp32_scale(scale)
    rows = np.asarray(rows, dtype=np.int64)
    B, H, N, d = q.shape
    R = len(rows)
    out = {"O": np.empty((B, H, R, d)), "LSE": np.empty((B, H, R)),
           "D": np.empty((B, H, R)), "dQ": np.empty((B, H, R, d))}
    cols = np.arange(N)[None, :]
    for b in range(B):
        for h in range(H):
            S = scores(q[b, h][rows], k[b, h], s)                  # [R, N]
            if causal:
                S = np.where(cols > rows[:, None], -np.inf, S)
            lse = row_logsumexp(S)
            P = _probabilities(S, lse)
            O = P @ v[b, h]
            Dr = (dO[b, h][rows] * O).sum(axis=1)
            dP = dO[b, h][rows] @ v[b, h].T
            dS = P * (dP - Dr[:, None])
            out["O"][b, h] = O
            out["LSE"][b, h] = lse
            out["D"][b, h] = Dr
            out["dQ"][b, h] = s * (dS @ k[b, h])
    return out


def attn_bwd_gqa(q, k, v, dO, scale: float, causal: bool):
    """Grouped-query attention, forward + backward, fp64.

    Grouped-query attention is named as a next primitive in the article
    (section "Next Frontiers in WebGPU ML"); the pages give no formula, so the
    plain reading is used: q, dO are [B, H, N, d], k, v are [B, H_kv, N, d]
    with H a multiple of H_kv, and query head h attends to key/value head
    h // (H / H_kv).  Each query head is ordinary attention against its
    key/value head; because a key/value head feeds H / H_kv query heads, its
    gradients dK, dV are the sums of the per-query-head gradients over that
    group.  Returns a dict with O, LSE, D, dQ ([B, H, ...]) and dK, dV
    ([B, H_kv, N, d]).
    """
    q, k, v, dO = as_f64(q), as_f64(k), as_f64(v), as_f64(dO)
    s = fp32_scale(scale)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    G = H // Hkv
    out = {"O": np.empty((B, H, N, d)), "LSE": np.empty((B, H, N)), "D": np.empty((B, H, N)),
           "dQ": np.empty((B, H, N, d)), "dK": np.zeros((B, Hkv, N, d)), "dV": np.zeros((B, Hkv, N, d))}
    for b in range(B):
        for h in range(H):
            hk = h // G
            r = attn_bwd_head(q[b, h], k[b, hk], v[b, hk], dO[b, h], s, causal)
            for key in ("O", "LSE", "D", "dQ"):
                out[key][b, h] = r[key]
            out["dK"][b, hk] += r["dK"]
            out["dV"][b, hk] += r["dV"]
    return out


def attn_fwd_general(q, k, v, scale: float, causal: bool):
    """Forward pass with separate query and key lengths and grouped K/V heads.

    q is [B, H, Nq, d]; k, v are [B, H_kv, Nk, d] with H a multiple of H_kv
    (query head h reads key/value head h // (H / H_kv)).  The pages name
    flash-decoding as a next primitive (article, section "Next Frontiers in
    WebGPU ML") but give no formula; the plain reading for Nq != Nk is the
    usual key-value-cache alignment: the Nq queries are the last Nq positions
    of the Nk-long sequence, so with causal masking query i sees key j iff
    j <= i + (Nk - Nq).  Requires Nk >= Nq when causal.  Returns
    (O [B, H, Nq, d], LSE [B, H, Nq]) in fp64.
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    s = fp32_scale(scale)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    if causal and Nk < Nq:
        raise ValueError("causal attention needs Nk >= Nq")
    G = H // Hkv
    O = np.empty((B, H, Nq, d))
    L = np.empty((B, H, Nq))
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    for b in range(B):
        for h in range(H):
            S = scores(q[b, h], k[b, h // G], s)
            if causal:
                S = np.where(j > i + (Nk - Nq), -np.inf, S)
            lse = row_logsumexp(S)
            O[b, h] = _probabilities(S, lse) @ v[b, h // G]
            L[b, h] = lse
    return O, L


def attn_varlen(q, k, v, dO, cu_seqlens_q, cu_seqlens_k, scale: float, causal: bool):
    """Variable-length batch: forward (and backward when dO is given), fp64.

    The pages do not treat batches of sequences of different lengths; this is
    the usual packed form of the same attention (read here the plainest way):
    q, dO are [total_q, H, d], k, v are [total_k, H_kv, d]; sequence b owns
    query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1] - 1 and key rows
    cu_seqlens_k[b] .. cu_seqlens_k[b+1] - 1, and attends only within itself.
    Query head h reads key/value head h // (H / H_kv).  With causal masking
    the Lq queries of a sequence are its last Lq positions (key-value-cache
    alignment, as in attn_fwd_general): query i sees key j iff
    j <= i + (Lk - Lq).  A query that sees no key (Lk = 0, or Lk < Lq under
    causal masking) gets O = 0, LSE = -inf and zero gradients.
    Returns a dict with O [total_q, H, d] and LSE [H, total_q]; with dO also
    dQ [total_q, H, d], dK and dV [total_k, H_kv, d].
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    dO = None if dO is None else as_f64(dO)
    cq = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    ck = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0:
        raise ValueError("cu_seqlens must start at 0 and have the same length")
    if any(b < a for a, b in zip(cq, cq[1:])) or any(b < a for a, b in zip(ck, ck[1:])):
        raise ValueError("cu_seqlens must be non-decreasing")
    s = fp32_scale(scale)
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if cq[-1] != total_q or ck[-1] != total_k:
        raise ValueError("cu_seqlens must end at the packed lengths")
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    G = H // Hkv
    out = {"O": np.zeros((total_q, H, d)), "LSE": np.full((H, total_q), -np.inf)}
    if dO is not None:
        out["dQ"] = np.zeros((total_q, H, d))
        out["dK"] = np.zeros((total_k, Hkv, d))
        out["dV"] = np.zeros((total_k, Hkv, d))
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        Lq, Lk = q1 - q0, k1 - k0
        if Lq == 0 or Lk == 0:
            continue  # no query, or nothing to see: outputs stay 0 / -inf
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        for h in range(H):
            hk = h // G
            S = scores(q[q0:q1, h], k[k0:k1, hk], s)
            if causal:
                S = np.where(j > i + (Lk - Lq), -np.inf, S)
            lse = row_logsumexp(S)
            P = _probabilities(S, lse)
            O = P @ v[k0:k1, hk]
            out["O"][q0:q1, h] = O
            out["LSE"][h, q0:q1] = lse
            if dO is None:
                continue
            g = dO[q0:q1, h]
            D = (g * O).sum(axis=1)
            dS = P * (g @ v[k0:k1, hk].T - D[:, None])
            out["dQ"][q0:q1, h] = s * (dS @ k[k0:k1, hk])
            out["dK"][k0:k1, hk] += s * (dS.T @ q[q0:q1, h])
            out["dV"][k0:k1, hk] += P.T @ g
    return out
