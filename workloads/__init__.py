"""Seeded synthetic inputs for the attention hot path.

This module only draws random numbers and rounds them to bf16; it holds none
of the attention arithmetic.  Both the CPU oracle (``oracle/``) and the CUDA
path (``tiled_exact_attention_fa2_gb300``) consume what it returns, so the two
sides see bit-identical inputs.

Recipe (the pages fix no input distribution, so this is the plainest one that
matches the stated workloads): Q, K, V and dO are drawn i.i.d. N(0, 1) in fp32
from a PCG64 generator seeded per workload, in the order Q, K, V, dO; Q and K
are then multiplied by ``qk_mult`` (3 for the large-logit stress workload),
and every tensor is rounded to bf16 once (round-to-nearest-even).  Layout is
row-major contiguous [B, H, N, d].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple = (True,)
    qk_mult: float = 1.0
    seed: int = 0
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self, causal: bool) -> float:
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if causal else f

    def bwd_flops(self, causal: bool) -> float:
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if causal else f


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 16, (True, False), 1.0, 1000,
                     "oracle finishes in well under a second"),
    "small": Workload("small", 8, 4, 256, 32, (True,), 1.0, 1001,
                      "small GPT layer"),
    "medium": Workload("medium", 4, 16, 1024, 64, (True, False), 1.0, 1002,
                       "medium GPT layer"),
    "stress": Workload("stress", 2, 16, 4096, 128, (True,), 3.0, 1003,
                       "large-logit stress: Q, K x3"),
    "long": Workload("long", 1, 32, 16384, 128, (True, False), 1.0, 1004,
                     "long sequence; oracle on 64 sampled query rows per head"),
}


def make_inputs(B: int, H: int, N: int, d: int, seed: int, qk_mult: float = 1.0,
                with_grad: bool = True):
    """Return dict q, k, v (and dO) as CPU bf16 tensors of shape [B, H, N, d]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shape = (B, H, N, d)
    names = ("q", "k", "v", "dO") if with_grad else ("q", "k", "v")
    out = {}
    for name in names:
        x = rng.standard_normal(size=shape, dtype=np.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x *= np.float32(qk_mult)
        out[name] = torch.from_numpy(x).to(torch.bfloat16).contiguous()
    return out


def make_profile_inputs(B: int, H: int, N: int, d: int, profile: str, strength: float, seed: int):
    """make_inputs with K reshaped so that the largest scores of a query row
    come late in the key sequence (CPU bf16 tensors, with dO).

    'ramp'  scales key row j by 1 + strength * j / N, so score magnitudes, and
            with them each row's running maximum, grow along the keys;
    'spike' replaces key row i - 3 by strength * (query row i) for every
            eighth query row i >= 8, which gives row i one very large score
            just before its own position (a causal row sees it).
    """
    x = make_inputs(B, H, N, d, seed)
    k = x["k"].float()
    if profile == "ramp":
        ramp = 1.0 + strength * torch.arange(N, dtype=torch.float32) / N
        k = k * ramp[None, None, :, None]
    elif profile == "spike":
        q = x["q"].float()
        for i in range(8, N, 8):
            k[:, :, i - 3] = strength * q[:, :, i]
    else:
        raise ValueError(profile)
    x["k"] = k.to(torch.bfloat16).contiguous()
    return x


def workload_inputs(w: Workload, with_grad: bool = True):
    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_grad)


def sample_rows(N: int, count: int, seed: int) -> np.ndarray:
    """Seeded sorted sample of distinct row indices in [0, N) (always includes 0 and N-1)."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    count = min(count, N)
    if count >= N:
        return np.arange(N)
    rows = set(rng.choice(N, size=count - 2, replace=False).tolist()) | {0, N - 1}
    extra = iter(rng.permutation(N).tolist())
    while len(rows) < count:
        rows.add(next(extra))
    return np.array(sorted(rows), dtype=np.int64)


def make_varlen_inputs(lens_q, lens_k, H: int, H_kv: int, d: int, seed: int, qk_mult: float = 1.0,
                       with_grad: bool = True):
    """Packed variable-length batch: q, dO [total_q, H, d], k, v [total_k, H_kv, d].

    Same recipe as make_inputs (i.i.d. N(0, 1) fp32 in the order Q, K, V, dO,
    Q and K times qk_mult, bf16 once); sequence b owns query rows
    cu_q[b] .. cu_q[b+1] - 1 and key rows cu_k[b] .. cu_k[b+1] - 1.  Returns
    a dict with those tensors (CPU) and cu_q, cu_k as int32 tensors of B + 1
    entries.
    """
    lens_q, lens_k = [int(x) for x in lens_q], [int(x) for x in lens_k]
    if len(lens_q) != len(lens_k) or min(lens_q + lens_k) < 0:
        raise ValueError("need one non-negative query and key length per sequence")
    rng = np.random.Generator(np.random.PCG64(seed))
    tq, tk = sum(lens_q), sum(lens_k)
    shapes = {"q": (tq, H, d), "k": (tk, H_kv, d), "v": (tk, H_kv, d), "dO": (tq, H, d)}
    names = ("q", "k", "v", "dO") if with_grad else ("q", "k", "v")
    out = {}
    for name in names:
        x = rng.standard_normal(size=shapes[name], dtype=np.float32)
        if name in ("q", "k") and qk_mult != 1.0:
            x *= np.float32(qk_mult)
        out[name] = torch.from_numpy(x).to(torch.bfloat16).contiguous()
    out["cu_q"] = torch.tensor(np.concatenate([[0], np.cumsum(lens_q)]), dtype=torch.int32)
    out["cu_k"] = torch.tensor(np.concatenate([[0], np.cumsum(lens_k)]), dtype=torch.int32)
    return out


def varlen_lengths(B: int, max_len: int, seed: int) -> list:
    """Seeded length mix for a variable-length batch: uniform in [1, max_len],
    with the first sequence at max_len (so the longest is always present)."""
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    lens = rng.integers(1, max_len + 1, size=B).tolist()
    lens[0] = max_len
    return [int(x) for x in lens]
