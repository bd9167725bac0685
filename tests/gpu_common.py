"""Shared helpers of the GPU parity tests: seeded inputs, oracle evaluation on chosen rows, and
the tolerance.

Two bounds must both hold for every compared slice:
  * the absolute one the method's acceptance bar states: max-abs error 1e-2 (f16) and 2e-2
    (bf16) on N(0,1) data ("Build FlashAttention (CK backend) on gfx90a", Verification uses
    max_diff < 0.01);
  * a relative one that still bites at long context, where an output element of N(0,1) data
    has an RMS of only ~1/sqrt(visible keys) (0.0064 at 65 536 keys): for every element,
        |got - want| <= u * (|want| + c * RMS(want's row)),
    u the unit roundoff of the dtype (2^-11 f16, 2^-8 bf16).  The kernels round O once when
    storing it (at most u * |O| for that element) and round P (or P times a V scale) once to
    the dtype before the PV contraction; a q4_0 side is also rounded once when dequantized.
    The P rounding perturbs an output element by sum_j delta_j w_j v_j (|delta_j| <= u): a
    near-Gaussian error of standard deviation ~u/sqrt(3) * sqrt(sum_j w_j^2 v_j^2), which is
    about u/sqrt(3) times the RMS of the row's output whether the softmax is diffuse or peaked;
    over a few million outputs its maximum stays near 5.6 sigma, ~3.2 u * RMS(row).  c = 6 for
    dense K/V, 9 when a side is q4_0 (one more rounding of comparable size).  A kernel that
    dropped a single 128-key block out of 16 384 would be off by ~25 % of the row's RMS on some
    element of that row."""
from __future__ import annotations

import numpy as np
import torch

import fa_inputs
import oracle

TOL = {"f16": 1e-2, "bf16": 2e-2}
UNIT_ROUNDOFF = {"f16": 2.0 ** -11, "bf16": 2.0 ** -8}
REL_FACTOR = {False: 6.0, True: 9.0}  # dense K/V, some side q4_0


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


def rel_bound(want: np.ndarray, dtype: str, q4: bool = False) -> np.ndarray:
    """The per-element relative bound u * (|want| + c * RMS(row)) (see the module docstring);
    rows are the last axis."""
    want = np.asarray(want, dtype=np.float64)
    rms = np.sqrt(np.mean(np.square(want), axis=-1, keepdims=True))
    return UNIT_ROUNDOFF[dtype] * (np.abs(want) + REL_FACTOR[bool(q4)] * rms)


def check_close(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "",
                q4: bool = False):
    """Both bounds of the module docstring; q4: some K/V side is q4_0.  Returns the max-abs
    error."""
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = max_abs_err(got, want)
    assert err <= TOL[dtype], f"{what}: max-abs error {err:.3e} > {TOL[dtype]}"
    if got.size:
        ratio = np.abs(got - want) / rel_bound(want, dtype, q4)
        i = int(np.argmax(ratio))
        assert ratio.flat[i] <= 1.0, (
            f"{what}: error {abs(got.flat[i] - want.flat[i]):.3e} at element {i} (oracle "
            f"{want.flat[i]:.4e}) exceeds u (|want| + {REL_FACTOR[bool(q4)]:g} RMS(row)) by "
            f"{ratio.flat[i]:.2f}x")
    return err
