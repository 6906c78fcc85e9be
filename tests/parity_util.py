"""Comparison helpers shared by the GPU parity tests (no attention arithmetic here)."""
import numpy as np
import torch

O_ABS_TOL = 1e-2      # O max-abs error
LSE_ABS_TOL = 2e-3    # LSE max-abs error
GRAD_REL_TOL = 2e-2   # dQ / dK / dV relative Frobenius error


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def check_o(got: np.ndarray, ref: np.ndarray, what: str = "O"):
    """O bound: |err| <= 1e-2, or <= one bf16 ulp of the reference where that
    ulp alone exceeds 1e-2 (|O| >= 4: output rounding to bf16 can then exceed
    the absolute bound by itself)."""
    err = np.abs(got - ref)
    bound = np.maximum(O_ABS_TOL, bf16_ulp(ref))
    worst = np.argmax(err - bound)
    assert np.all(err <= bound), (
        f"{what}: max-abs {err.max():.3e}; worst excess at flat index {worst}: "
        f"got {got.flat[worst]} ref {ref.flat[worst]} bound {bound.flat[worst]:.3e}")
    return float(err.max())


def check_lse(got: np.ndarray, ref: np.ndarray):
    err = np.abs(got - ref).max()
    assert err <= LSE_ABS_TOL, f"LSE max-abs {err:.3e}"
    return float(err)


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))


def check_grad(got: np.ndarray, ref: np.ndarray, name: str):
    rel = rel_fro(got, ref)
    assert rel <= GRAD_REL_TOL, f"{name}: relative Frobenius error {rel:.3e}"
    return rel
