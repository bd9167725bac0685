"""The FLOP count used for every TFLOP/s figure, pinned to the figures printed on
"perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" (Measurements and
Summary): ms/call and TFLOP/s of the chunked-prefill call (B=1, GQA 32/8, D=128, Sq=2048) at
2K/8K/16K keys.  FLOPs = 4 * D * Hq * B * (visible query-key pairs), bottom-right causal mask,
diagonal included, masked pairs not counted."""
import pytest

import fa_inputs

# (keys, ms/call, TFLOP/s) as printed, before and after the change and for the gated 16K run
PRINTED = [
    (2048, 19.0, 1.81), (8192, 124.5, 1.93), (16384, 429.2, 1.20),
    (2048, 24.4, 1.41), (8192, 161.7, 1.49), (16384, 540.1, 0.95),
    (16384, 392.6, 1.31),
]


@pytest.mark.parametrize("sk,ms,tflops", PRINTED)
def test_flop_convention_reproduces_printed_rates(sk, ms, tflops):
    w = fa_inputs.Workload("x", 1, 32, 8, 2048, sk, 128, "f16", "dense")
    rate = w.flops() / (ms * 1e-3) / 1e12
    assert round(rate, 2) == pytest.approx(tflops, abs=0.006)


def test_closed_form_visible_pairs():
    w = fa_inputs.Workload("x", 1, 32, 8, 2048, 16384, 128, "f16", "dense")
    sq, sk = 2048, 16384
    assert w.visible_pairs() == sq * (sk - sq) + sq * (sq + 1) // 2
    assert abs(w.flops() - 515.41e9) < 0.005e9
