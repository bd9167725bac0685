"""Shared helpers of the GPU parity tests: seeded inputs, oracle evaluation on chosen rows, and
the tolerance (max-abs error 1e-2 for f16, 2e-2 for bf16 on N(0,1) data)."""
from __future__ import annotations

import numpy as np
import torch

import fa_inputs
import oracle

TOL = {"f16": 1e-2, "bf16": 2e-2}


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact upcast of a (CPU or GPU) f16/bf16 tensor to f64."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def sample_rows(B: int, Hq: int, Sq: int, per_head: int = 12, seed: int = 0) -> np.ndarray:
    """Flat row indices (b*Hq + h)*Sq + i: tile edges, the last rows and a few random rows of
    every (b, h)."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, 255, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1]
    fixed = sorted({i for i in fixed if 0 <= i < Sq})
    rows = []
    for bh in range(B * Hq):
        extra = rng.integers(0, Sq, size=max(0, per_head - len(fixed)))
        for i in sorted(set(fixed) | set(int(x) for x in extra)):
            rows.append(bh * Sq + i)
    return np.array(rows, dtype=np.int64)


def q4_planes_gpu(q4) -> tuple[np.ndarray, np.ndarray]:
    return (q4.nibbles().cpu().numpy(), q4.scales().cpu().view(torch.int16).numpy().view(np.uint16))


def oracle_q4_planes(x: torch.Tensor):
    return oracle.quantize_q4_0(x.detach().cpu().to(torch.float32).numpy())


def max_abs_err(got: np.ndarray, want: np.ndarray) -> float:
    return float(np.max(np.abs(got - want))) if got.size else 0.0


def check_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = ""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = max_abs_err(got, want)
    assert err <= TOL[dtype], f"{what}: max-abs error {err:.3e} > {TOL[dtype]}"
    return err
