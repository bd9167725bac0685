"""Pins for the CPU oracle: facts fixed by the pages and by mathematics, not by the oracle.

Each test below would fail on a plausible mistake in ``oracle/fa_oracle.c``: a wrong mask index
or a dropped diagonal (prefix-mean closed form, brute force), a wrong GQA head map (brute force,
library SDPA), a missing max-subtraction or normalisation (row sums, constant V, huge scores),
swapped nibbles or a wrong scale sign (hand-worked block, grid round-trip), a wrong rounding mode
(binary16 conversion against numpy).
"""
import decimal
import fractions
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------------------
# binary16 conversion (library special case: numpy's own binary16 rounding)
# ----------------------------------------------------------------------------------------------

def test_f32_to_f16_matches_numpy(oracle_mod):
    rng = np.random.default_rng(7)
    parts = [
        rng.standard_normal(4000).astype(np.float32),
        (rng.standard_normal(3000) * 1e-5).astype(np.float32),       # f16 subnormal range
        (rng.standard_normal(2000) * 3e4).astype(np.float32),        # near overflow
        np.float32(2.0) ** rng.integers(-30, 17, 500).astype(np.float32),
    ]
    # exact ties between two binary16 neighbours (odd and even mantissas)
    base = np.arange(1024, 2048, dtype=np.float64)
    ties = ((base + 0.5) * 2.0 ** -10).astype(np.float32)
    sub_ties = ((np.arange(0, 64) + 0.5) * 2.0 ** -24).astype(np.float32)
    special = np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, np.inf, -np.inf,
                        2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -24],
                       dtype=np.float32)
    x = np.concatenate(parts + [ties, -ties, sub_ties, special])
    got = oracle_mod.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_f16_decode_all_patterns(oracle_mod):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(vals)
    got = oracle_mod.f16_bits_to_f64(bits[finite])
    np.testing.assert_array_equal(got, vals[finite])


# ----------------------------------------------------------------------------------------------
# q4_0 quantizer
# ----------------------------------------------------------------------------------------------

def _read_golden_block():
    fields = {}
    with open(os.path.join(GOLDEN, "q4_0_hand_block.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            fields[key] = vals
    return fields


def test_q4_0_hand_block(oracle_mod):
    g = _read_golden_block()
    x = np.array([float(v) for v in g["x"]], dtype=np.float32)
    nib, scale = oracle_mod.quantize_q4_0(x[None, :])
    assert int(scale[0, 0]) == int(g["scale_bits"][0], 16)
    np.testing.assert_array_equal(nib[0], np.array([int(b, 16) for b in g["bytes"]], np.uint8))
    codes = np.concatenate([nib[0] & 0xF, nib[0] >> 4])
    np.testing.assert_array_equal(codes, np.array([int(c) for c in g["codes"]]))
    vals = oracle_mod.dequantize_q4_0(nib, scale)[0]
    np.testing.assert_array_equal(vals, np.array([float(v) for v in g["values"]]))


def test_q4_0_zero_block(oracle_mod):
    nib, scale = oracle_mod.quantize_q4_0(np.zeros((3, 32), np.float32))
    # m = +0 and d = m / -8 = -0 under IEEE division, so the stored scale is -0 (0x8000)
    assert (scale == 0x8000).all()
    assert (nib == 0x88).all()
    assert (oracle_mod.dequantize_q4_0(nib, scale) == 0).all()


def test_q4_0_tie_break_and_sign(oracle_mod):
    x = np.zeros(32, np.float32)
    x[3] = 2.0
    x[5] = -2.0
    x[9] = 1.0
    nib, scale = oracle_mod.quantize_q4_0(x[None])
    # first element of largest magnitude is +2.0 -> d = 2 / -8 = -0.25 (fp16 0xB400)
    assert int(scale[0, 0]) == 0xB400
    vals = oracle_mod.dequantize_q4_0(nib, scale)[0]
    assert vals[3] == 2.0             # the max element round-trips exactly (code 0)
    assert (nib[0, 3] & 0xF) == 0
    assert vals[5] == -1.75           # opposite sign clamps at code 15: 7 * -0.25
    assert vals[9] == 1.0             # 1.0 / -0.25 = -4 -> code 4 -> (4 - 8) * -0.25
    flipped = -x
    nib2, scale2 = oracle_mod.quantize_q4_0(flipped[None])
    assert int(scale2[0, 0]) == 0x3400   # d = -2 / -8 = +0.25


def test_q4_0_grid_round_trip(oracle_mod):
    """Values already on a q4_0 grid (d a power of two, an element at code 0 carrying the largest
    magnitude) must come back bit for bit: codes, scale and values."""
    rng = np.random.default_rng(11)
    nblk = 400
    codes = rng.integers(1, 16, size=(nblk, 32))
    first = rng.integers(0, 32, size=nblk)
    codes[np.arange(nblk), first] = 0
    # put any other code-0 elements after 'first' would still be fine; make sure none precede it
    for b in range(nblk):
        codes[b, :first[b]][codes[b, :first[b]] == 0] = 1
    exps = rng.integers(-8, 6, size=nblk)
    sign = rng.choice([-1.0, 1.0], size=nblk)
    d = sign * 2.0 ** exps
    x = ((codes - 8) * d[:, None]).astype(np.float32)
    nib, scale = oracle_mod.quantize_q4_0(x)
    got_codes = np.concatenate([nib & 0xF, nib >> 4], axis=1)
    np.testing.assert_array_equal(got_codes, codes)
    np.testing.assert_array_equal(scale.view(np.float16).astype(np.float64)[:, 0], d)
    np.testing.assert_array_equal(oracle_mod.dequantize_q4_0(nib, scale), x.astype(np.float64))


def test_q4_0_error_bounds(oracle_mod):
    """Rounding bound: |x - x'| <= |d16|/2 + 8|d - d16| where x/d <= 7.5 (plus f32 slack); the
    clamped elements (x/d > 7.5, opposite sign to m) stay within |d16| + 8|d - d16|; the element
    of largest magnitude is exact.  (A bound of half a step for every element cannot hold for
    this signed-scale format: x = -m lands at code 15, one full step away.)"""
    rng = np.random.default_rng(5)
    x16 = rng.standard_normal((2000, 32)).astype(np.float16)
    x = x16.astype(np.float32)
    nib, scale = oracle_mod.quantize_q4_0(x)
    xq = oracle_mod.dequantize_q4_0(nib, scale)
    xd = x.astype(np.float64)
    idx = np.argmax(np.abs(xd), axis=1)
    m = xd[np.arange(len(xd)), idx]
    d = m / -8.0
    d16 = scale.view(np.float16).astype(np.float64)[:, 0]
    err = np.abs(xd - xq)
    ratio = xd / d[:, None]
    slack = 1e-6 * np.abs(xd) + 1e-12
    lim_round = np.abs(d16)[:, None] / 2 + 8 * np.abs(d - d16)[:, None] + slack
    lim_clamp = np.abs(d16)[:, None] + 8 * np.abs(d - d16)[:, None] + slack
    unclamped = ratio <= 7.5
    assert (err[unclamped] <= np.broadcast_to(lim_round, err.shape)[unclamped]).all()
    assert (err[~unclamped] <= np.broadcast_to(lim_clamp, err.shape)[~unclamped]).all()
    assert (~unclamped).any()   # the clamp case does occur on N(0,1) blocks
    np.testing.assert_array_equal(xq[np.arange(len(xd)), idx], m)


# ----------------------------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------------------------

def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.mark.parametrize("causal", [True, False])
def test_softmax_rows_sum_to_one(oracle_mod, causal):
    q = _rand((1, 4, 24, 16), 1)
    k = _rand((1, 2, 40, 16), 2)
    v = _rand((1, 2, 40, 16), 3)
    _, p = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=16, scale=0.3,
                                return_probs=True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    if causal:
        # row i sees keys 0..16+i only
        for r in range(p.shape[0]):
            i = r % 24
            assert (p[r, 16 + i + 1:] == 0).all()
            assert (p[r, :16 + i + 1] > 0).all()


def test_constant_v(oracle_mod):
    q = _rand((2, 4, 9, 8), 4)
    k = _rand((2, 2, 13, 8), 5)
    c = _rand((8,), 6)
    v = np.broadcast_to(c, (2, 2, 13, 8)).copy()
    o = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=4, scale=0.7)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-12)


def test_single_key_returns_v(oracle_mod):
    q = _rand((3, 8, 1, 64), 7)
    k = _rand((3, 2, 1, 64), 8)
    v = _rand((3, 2, 1, 64), 9)
    o = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=0, scale=0.125)
    for h in range(8):
        np.testing.assert_array_equal(o[:, h, 0], v[:, h // 4, 0])


def test_key_value_permutation_invariance(oracle_mod):
    q = _rand((1, 2, 7, 16), 10)
    k = _rand((1, 1, 33, 16), 11)
    v = _rand((1, 1, 33, 16), 12)
    perm = np.random.default_rng(13).permutation(33)
    o1 = oracle_mod.attention(q, k, v, causal=False, scale=0.25)
    o2 = oracle_mod.attention(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.25)
    np.testing.assert_allclose(o1, o2, atol=1e-12)


def test_zero_query_is_causal_prefix_mean(oracle_mod):
    """Q = 0 makes every visible score equal, so causal row i (position off+i) is the mean of
    V[0..off+i]: pins the bottom-right alignment and that the diagonal key is visible."""
    B, Hq, Hkv, Sq, Sk, D = 2, 6, 3, 5, 11, 4
    off = Sk - Sq
    q = np.zeros((B, Hq, Sq, D))
    k = _rand((B, Hkv, Sk, D), 14)
    v = _rand((B, Hkv, Sk, D), 15)
    o = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=off, scale=1.0)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(Sq):
                want = v[b, g, :off + i + 1].mean(axis=0)
                np.testing.assert_allclose(o[b, h, i], want, atol=1e-13)


def test_dominant_key(oracle_mod):
    """One key whose scaled score exceeds all others by ~60 takes all the weight."""
    D = 8
    q = np.zeros((1, 1, 1, D))
    q[..., 0] = 1.0
    k = _rand((1, 1, 20, D), 16, 0.01)
    k[0, 0, 7, 0] = 60.0
    v = _rand((1, 1, 20, D), 17)
    o = oracle_mod.attention(q, k, v, causal=False, scale=1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 7], atol=1e-20 + 1e-24, rtol=1e-24)


def _brute_force(q, k, v, causal, off, scale):
    """An independent evaluator: exact rational dot products, 50-digit decimal exponentials, no
    max subtraction, every (i, j) pair enumerated."""
    ctx = decimal.Context(prec=50)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    out = np.zeros(q.shape)
    for b in range(B):
        for h in range(Hq):
            g = h * Hkv // Hq
            for i in range(Sq):
                w = []
                for j in range(Sk):
                    if causal and j > off + i:
                        w.append(decimal.Decimal(0))
                        continue
                    dot = sum(fractions.Fraction(float(q[b, h, i, d])) *
                              fractions.Fraction(float(k[b, g, j, d])) for d in range(D))
                    s = dot * fractions.Fraction(scale)
                    sd = ctx.divide(decimal.Decimal(s.numerator), decimal.Decimal(s.denominator))
                    w.append(ctx.exp(sd))
                tot = sum(w, decimal.Decimal(0))
                for d in range(D):
                    acc = sum((wj * decimal.Decimal(float(v[b, g, j, d])) for j, wj in
                               enumerate(w)), decimal.Decimal(0))
                    out[b, h, i, d] = float(ctx.divide(acc, tot))
    return out


@pytest.mark.parametrize("causal,Sq,Sk,off", [(True, 5, 8, 3), (True, 4, 4, 0), (False, 3, 7, 0),
                                              (True, 1, 6, 5), (True, 6, 8, 1)])
def test_brute_force_tiny(oracle_mod, causal, Sq, Sk, off):
    B, Hq, Hkv, D = 2, 4, 2, 3
    q = _rand((B, Hq, Sq, D), 20 + Sq, 1.5)
    k = _rand((B, Hkv, Sk, D), 30 + Sk, 1.5)
    v = _rand((B, Hkv, Sk, D), 40 + off)
    want = _brute_force(q, k, v, causal, off, 0.8)
    got = oracle_mod.attention(q, k, v, causal=causal, q_pos_offset=off, scale=0.8)
    np.testing.assert_allclose(got, want, atol=1e-13, rtol=0)


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(2, 8, 8, 512, 64), (1, 8, 2, 192, 128)])
def test_matches_torch_sdpa_f64(oracle_mod, B, Hq, Hkv, S, D):
    """Library special case: torch's CPU scaled_dot_product_attention in float64, with the key
    heads repeated per group and an explicit boolean mask (torch's is_causal is top-left aligned;
    here Sq = Sk so both alignments agree, and the mask is explicit anyway)."""
    g = torch.Generator().manual_seed(99)
    q = torch.randn(B, Hq, S, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, S, D, generator=g, dtype=torch.float64)
    scale = 1.0 / math.sqrt(D)
    kr = k.repeat_interleave(Hq // Hkv, dim=1)
    vr = v.repeat_interleave(Hq // Hkv, dim=1)
    mask = torch.ones(S, S, dtype=torch.bool).tril()
    ref = torch.nn.functional.scaled_dot_product_attention(q, kr, vr, attn_mask=mask,
                                                           scale=scale)
    got = oracle_mod.attention(q.numpy(), k.numpy(), v.numpy(), causal=True, q_pos_offset=0,
                               scale=scale)
    np.testing.assert_allclose(got, ref.numpy(), atol=1e-12, rtol=0)


def test_bottom_right_chunk_matches_explicit_mask_sdpa(oracle_mod):
    """A query chunk at positions Sk-Sq..Sk-1: torch SDPA with the explicit bottom-right mask."""
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 1, 48, 160, 32
    g = torch.Generator().manual_seed(3)
    q = torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float64)
    off = Sk - Sq
    mask = torch.arange(Sk)[None, :] <= (off + torch.arange(Sq))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.expand(B, Hq, Sk, D), v.expand(B, Hq, Sk, D), attn_mask=mask, scale=0.2)
    got = oracle_mod.attention(q.numpy(), k.numpy(), v.numpy(), causal=True, q_pos_offset=off,
                               scale=0.2)
    np.testing.assert_allclose(got, ref.numpy(), atol=1e-12, rtol=0)


def test_q4_0_attention_equals_dense_on_dequantized(oracle_mod):
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Sq, Sk, D = 1, 4, 2, 6, 40, 64
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Sk, D)).astype(np.float32)
    kp = oracle_mod.quantize_q4_0(k)
    vp = oracle_mod.quantize_q4_0(v)
    o1 = oracle_mod.attention_q4_0(q, kp, vp, causal=True, q_pos_offset=Sk - Sq, scale=0.125)
    o2 = oracle_mod.attention(q, oracle_mod.dequantize_q4_0(*kp), oracle_mod.dequantize_q4_0(*vp),
                              causal=True, q_pos_offset=Sk - Sq, scale=0.125)
    np.testing.assert_array_equal(o1, o2)


def test_row_subset_matches_full(oracle_mod):
    q = _rand((2, 4, 10, 8), 50)
    k = _rand((2, 2, 12, 8), 51)
    v = _rand((2, 2, 12, 8), 52)
    full = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=2, scale=0.5)
    rows = np.array([0, 7, 19, 33, 79])
    sub = oracle_mod.attention(q, k, v, causal=True, q_pos_offset=2, scale=0.5, rows=rows)
    np.testing.assert_array_equal(sub, full.reshape(-1, 8)[rows])
