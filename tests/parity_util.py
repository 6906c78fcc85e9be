"""Comparison helpers shared by the GPU parity tests (no attention arithmetic here).

Every check records the error it measured against its bound; the pytest
session prints the worst margin of every test at the end (tests/conftest.py),
so a run's output shows how close each comparison came to its tolerance.
"""
import os

import numpy as np
import torch

O_ABS_TOL = 1e-2      # O max-abs error
LSE_ABS_TOL = 2e-3    # LSE max-abs error
GRAD_REL_TOL = 2e-2   # dQ / dK / dV relative Frobenius error
# Where |O_ref| >= 4 the bf16 spacing is 2^-5 and rounding O to bf16 alone can
# move it by 2^-6 > 1e-2; there the bound is one bf16 ulp of the reference.
O_ULP_FROM = 4.0

# (test id, quantity, error, bound) of every check in this process.
RECORDS = []


def _record(what, err, bound):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    RECORDS.append((test, what, float(err), float(bound)))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def o_bound(ref: np.ndarray) -> np.ndarray:
    """Element-wise O bound: 1e-2 where |O_ref| < 4, one bf16 ulp of O_ref above."""
    return np.where(np.abs(ref) < O_ULP_FROM, O_ABS_TOL, bf16_ulp(ref))


def check_o(got: np.ndarray, ref: np.ndarray, what: str = "O"):
    """|err| <= 1e-2 wherever |O_ref| < 4; <= one bf16 ulp of O_ref where |O_ref| >= 4."""
    err = np.abs(got - ref)
    bound = o_bound(ref)
    ratio = err / bound
    worst = int(np.argmax(ratio)) if ratio.size else 0
    if ratio.size:
        _record(what, err.flat[worst], bound.flat[worst])
    assert np.all(err <= bound), (
        f"{what}: max-abs {err.max():.3e}; worst excess at flat index {worst}: "
        f"got {got.flat[worst]} ref {ref.flat[worst]} bound {bound.flat[worst]:.3e}")
    return float(err.max()) if err.size else 0.0


def check_lse(got: np.ndarray, ref: np.ndarray, what: str = "LSE"):
    err = float(np.abs(got - ref).max()) if np.size(ref) else 0.0
    _record(what, err, LSE_ABS_TOL)
    assert err <= LSE_ABS_TOL, f"{what} max-abs {err:.3e}"
    return err


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def check_grad(got: np.ndarray, ref: np.ndarray, name: str):
    rel = rel_fro(got, ref)
    _record(name, rel, GRAD_REL_TOL)
    assert rel <= GRAD_REL_TOL, f"{name}: relative Frobenius error {rel:.3e}"
    return rel


def margin_report(records=None):
    """Lines for the session summary: per test its worst error / bound, then
    the worst of each quantity over the whole session."""
    records = RECORDS if records is None else records
    if not records:
        return []
    per_test = {}
    for test, what, err, bound in records:
        key = (test, what)
        if key not in per_test or err / bound > per_test[key][0] / per_test[key][1]:
            per_test[key] = (err, bound)
    lines = []
    for (test, what), (err, bound) in sorted(per_test.items()):
        lines.append(f"{test} {what}: {err:.3e} (bound {bound:.1e}, {err / bound:.2f} of it)")
    worst = {}
    for test, what, err, bound in records:
        kind = what.split(" ")[0]
        if kind not in worst or err / bound > worst[kind][1] / worst[kind][2]:
            worst[kind] = (test, err, bound)
    for kind, (test, err, bound) in sorted(worst.items()):
        lines.append(f"WORST {kind}: {err:.3e} = {err / bound:.2f} of bound {bound:.1e} in {test}")
    return lines
