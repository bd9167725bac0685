"""The synthetic input recipe, on the CPU: workload names against their shapes, seeding and draw
order, and the score ramp -- its values, and the frame movement it exists to cause (the deferred
rescale of "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)",
Summary: a row's frame moves only when a block's max exceeds it by more than 10)."""
import math
import re

import numpy as np
import pytest
import torch

import fa_inputs

PREFILL = re.compile(r"prefill(_q4_0)?_gqa(\d+)x(\d+)_d(\d+)_sq(\d+)_sk(\d+)_(f16|bf16)(_ramp)?$")
SELF = re.compile(r"selfattn_b(\d+)_s(\d+)_h(\d+)_d(\d+)_(f16|bf16)$")
DECODE = re.compile(r"decode_q4_0_b(\d+)_gqa(\d+)x(\d+)_d(\d+)_sk(\d+)_(f16|bf16)$")


def test_names_describe_the_shapes():
    for name, w in fa_inputs.WORKLOADS.items():
        assert w.name == name and w.causal
        if m := PREFILL.match(name):
            q4, hq, hkv, d, sq, sk, dt, ramp = m.groups()
            assert (w.B, w.Hq, w.Hkv, w.D, w.Sq, w.Sk, w.dtype) == (1, int(hq), int(hkv), int(d),
                                                                     int(sq), int(sk), dt)
            assert w.kv_format == ("q4_0" if q4 else "dense") and w.ramp == bool(ramp)
        elif m := SELF.match(name):
            b, s, h, d, dt = m.groups()
            assert (w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.dtype) == (int(b), int(h), int(h),
                                                                     int(s), int(s), int(d), dt)
        elif m := DECODE.match(name):
            b, hq, hkv, d, sk, dt = m.groups()
            assert (w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.dtype, w.kv_format) == (
                int(b), int(hq), int(hkv), 1, int(sk), int(d), dt, "q4_0")
        else:
            raise AssertionError(f"unrecognised workload name {name}")
        # the query chunk sits at the end of the keys (decode: at position Sk - 1)
        assert w.q_pos_offset == w.Sk - w.Sq


def test_draws_are_seeded_and_in_q_k_v_order():
    q, k, v = fa_inputs.make_tensors(2, 4, 2, 5, 9, 64, "bf16", seed=77)
    g = torch.Generator().manual_seed(77)
    want = [torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
            for shape in ((2, 4, 5, 64), (2, 2, 9, 64), (2, 2, 9, 64))]
    for got, ref in zip((q, k, v), want):
        assert got.dtype == torch.bfloat16 and torch.equal(got, ref)
    again = fa_inputs.make_tensors(2, 4, 2, 5, 9, 64, "bf16", seed=77)
    assert all(torch.equal(a, b) for a, b in zip((q, k, v), again))
    other = fa_inputs.make_tensors(2, 4, 2, 5, 9, 64, "bf16", seed=78)
    assert not torch.equal(q, other[0])


def test_ramp_values():
    D, Sk = 128, 1000
    scale = 1.0 / math.sqrt(D)
    q, k, v = fa_inputs.make_tensors(1, 2, 1, 4, Sk, D, "f16", seed=3, ramp=True)
    plain = fa_inputs.make_tensors(1, 2, 1, 4, Sk, D, "f16", seed=3)
    assert (q[..., 0] == 8.0).all()
    for j in (0, 127, 128, 255, 256, 640, 999):
        want = np.float16(2.0 * (j // 128) / (8.0 * scale))
        assert k[0, 0, j, 0].item() == float(want), j
    # nothing else changes: the other columns and V are the plain draw
    assert torch.equal(q[..., 1:], plain[0][..., 1:]) and torch.equal(k[..., 1:], plain[1][..., 1:])
    assert torch.equal(v, plain[2])


def frame_moves(s_nat, margin=10.0, block=128):
    """Moves of a row's frame over its visible scores (natural-log units of the scaled score):
    the first block sets the frame, later blocks move it only when their max exceeds it by more
    than the margin."""
    f, moves = -math.inf, 0
    for b0 in range(0, s_nat.size, block):
        m = float(s_nat[b0:b0 + block].max())
        if m > f + margin:
            f, moves = m, moves + 1
    return moves


@pytest.mark.parametrize("name", ["prefill_gqa32x8_d128_sq2048_sk8192_f16_ramp",
                                  "prefill_gqa32x8_d128_sq2048_sk16384_f16_ramp"])
def test_ramp_moves_the_frame_about_every_five_blocks(name):
    """Scores of sampled rows in f64 from the dtype-rounded inputs: each 128-key block adds about
    2 to the scaled score, so the frame moves about every fifth block -- the count the GPU tests
    hold the kernel's rescale counter to (1 + (blocks - 1) / 5, within 30 %)."""
    w = fa_inputs.WORKLOADS[name]
    q, k, _ = fa_inputs.make_qkv(w)
    q64 = q.double().numpy()
    k64 = k.double().numpy()
    ratios = []
    for h in (0, 13, 31):
        g = h // (w.Hq // w.Hkv)
        for i in (0, 700, w.Sq - 1):
            pos = w.q_pos_offset + i
            s = w.scale * (k64[0, g, :pos + 1] @ q64[0, h, i])
            nblocks = pos // 128 + 1
            ratios.append(frame_moves(s) / (1 + (nblocks - 1) / 5.0))
    assert 0.7 < float(np.mean(ratios)) < 1.3, ratios
    assert min(ratios) > 0.5
