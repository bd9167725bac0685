"""The prefill's cut schedule on the host (no device): the segment table the kernel builds, read
back through fa_prefill_schedule, against the schedule restated here from its definition.

Definition restated: a work unit is a pair of consecutive 128-row query tiles of one (batch,
query head); tile t's key blocks are the 128-key blocks holding any key that one of its rows may
see (causal: key j visible to query row i iff j <= q_pos_offset + i); a unit takes as many steps
as its longer tile.  Units are ordered from the last pair of query tiles to the first, then by
batch, then by head, and their steps concatenated; CTA c of n runs global steps
[floor(c W / n), floor((c + 1) W / n)).  A CTA's segments are the maximal runs of one unit in its
range.  A unit cut between CTAs keeps each piece in slot 0 of its CTA when the CTA's range
starts inside or at the unit, else slot 1: every CTA needs at most one piece per slot.
"""
import numpy as np
import pytest

import quantized_kv_cache_sm_gb300 as fa


@pytest.fixture(autouse=True)
def _library(built):
    return built


BM = BN = 128


def visible_blocks(q0, Sq, Sk, off, causal):
    """Key blocks of the query tile at rows [q0, q0 + 128): blocks holding a visible key."""
    if q0 >= Sq:
        return 0
    last = min(q0 + BM, Sq) - 1
    max_key = min(Sk - 1, off + last) if causal else Sk - 1
    return max_key // BN + 1


def visible_blocks_by_mask(q0, Sq, Sk, off, causal):
    """The same count from the explicit mask (small shapes only)."""
    rows = np.arange(q0, min(q0 + BM, Sq))
    if rows.size == 0:
        return 0
    keys = np.arange(Sk)
    mask = keys[None, :] <= (off + rows)[:, None] if causal else np.ones((rows.size, Sk), bool)
    seen = mask.any(axis=0)
    return len({int(j) // BN for j in np.nonzero(seen)[0]})


def units_of(B, Hq, Sq, Sk, off, causal):
    n_tiles = -(-Sq // BM)
    n_pairs = -(-n_tiles // 2)
    units = []
    for pair in reversed(range(n_pairs)):
        q0A = 2 * BM * pair
        nbA = visible_blocks(q0A, Sq, Sk, off, causal)
        nbB = visible_blocks(q0A + BM, Sq, Sk, off, causal)
        for b in range(B):
            for h in range(Hq):
                units.append((b, h, q0A, nbA, nbB, max(nbA, nbB)))
    return units


def expected_segments(units, n):
    starts = np.cumsum([0] + [u[5] for u in units])
    W = int(starts[-1])
    rows = []
    for c in range(n):
        t, t_end = c * W // n, (c + 1) * W // n
        while t < t_end:
            k = int(np.searchsorted(starts, t, side="right")) - 1
            u, us = units[k], int(starts[k])
            j0 = t - us
            j1 = min(u[5], j0 + (t_end - t))
            rows.append((c, *u, j0, j1, us))
            t += j1 - j0
    return W, rows


def check_schedule(B, Hq, Hkv, Sq, Sk, D, off, causal, n, force=False):
    plan, rows = fa.fa_prefill_schedule(B, Hq, Hkv, Sq, Sk, D, off, causal, n, force_cut=force)
    units = units_of(B, Hq, Sq, Sk, off, causal)
    W, want = expected_segments(units, n)
    assert plan["W"] == W and plan["units"] == len(units)
    if not plan["cut"] and not force:
        assert plan["ctas"] == 0 and plan["workspace_bytes"] == 0 and rows.shape[0] == 0
        return plan, rows
    assert plan["ctas"] == n
    if plan["cut"]:
        flags = -(-(n * 2 * 4) // 256) * 256
        assert plan["workspace_bytes"] == flags + n * 2 * 2 * (D + 4) * BM * 4
    got = [tuple(int(x) for x in r[:10]) for r in rows]
    assert got == want
    # every step of every unit exactly once, the pieces of a unit in CTA order
    cover = {}
    for r in rows:
        cover.setdefault(int(r[9]), []).append((int(r[0]), int(r[7]), int(r[8])))
    for us, pieces in cover.items():
        assert [p[0] for p in pieces] == sorted(p[0] for p in pieces)
        assert pieces[0][1] == 0
        assert all(a[2] == b[1] for a, b in zip(pieces, pieces[1:]))
    # slots: -1 for a unit inside one CTA, else at most one piece per (CTA, slot)
    used = set()
    for r in rows:
        c, us, slot = int(r[0]), int(r[9]), int(r[10])
        whole_in_cta = len(cover[us]) == 1
        assert (slot == -1) == whole_in_cta
        if slot >= 0:
            assert (c, slot) not in used
            used.add((c, slot))
            assert slot == (0 if c * W // n >= us else 1)
    # the ranges are equal to one step
    per_cta = np.bincount(rows[:, 0], weights=rows[:, 8] - rows[:, 7], minlength=n)
    assert per_cta.sum() == W and per_cta.max() - per_cta.min() <= 1
    return plan, rows


def test_visible_blocks_match_the_mask():
    for Sq, Sk, off, causal in [(300, 300, 0, True), (200, 700, 500, True), (129, 1000, 871, True),
                                (257, 513, 0, False), (5, 900, 895, True), (128, 128, 0, True)]:
        for q0 in range(0, Sq + BM, BM):
            assert (visible_blocks(q0, Sq, Sk, off, causal)
                    == visible_blocks_by_mask(q0, Sq, Sk, off, causal)), (Sq, Sk, off, q0)


@pytest.mark.parametrize("Sk", [2048, 8192, 16384])
def test_chunked_prefill_plans(Sk):
    """The GQA 32/8 chunk of 2048 queries on 152 SMs: cut at 16K keys, whole units at 2K and 8K
    (the launches measured fastest there)."""
    plan, rows = check_schedule(1, 32, 8, 2048, Sk, 128, Sk - 2048, True, 152)
    assert plan["units"] == 256
    assert plan["cut"] == (Sk == 16384)
    if plan["cut"]:
        assert np.bincount(rows[:, 0]).max() <= 16


@pytest.mark.parametrize("shape", [
    (2, 16, 4, 1152, 20000, 128, 20000 - 1152, True),  # odd tile count, ragged Sq and Sk
    (1, 64, 8, 640, 8192, 128, 0, False),               # non-causal, no tile B in the last pair
    (4, 32, 8, 1000, 30000, 128, 29000, True),
    (3, 40, 8, 777, 777, 128, 0, True),                 # self-attention, ragged
])
@pytest.mark.parametrize("n", [1, 7, 100, 148, 152, 160])
def test_forced_cuts_cover_every_step(shape, n):
    """Cuts laid out for any CTA count: either every step is covered exactly once with at most
    one piece per slot, or the range does not fit the kernel's segment table and the query says
    so (the plan never cuts there)."""
    try:
        check_schedule(*shape, n, force=True)
    except fa.FaError as e:
        assert e.status == fa.FA_ERR_UNSUPPORTED
        plan, _ = fa.fa_prefill_schedule(*shape, n)
        assert not plan["cut"]


def test_planned_cuts_always_fit_the_segment_table():
    rng = np.random.default_rng(5)
    seen_cut = 0
    for _ in range(150):
        B = int(rng.integers(1, 5))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 8]))
        Sq = int(rng.integers(2, 4097))
        causal = bool(rng.integers(0, 2))
        Sk = Sq + int(rng.integers(0, 40000)) if causal else int(rng.integers(1, 40000))
        off = Sk - Sq if causal else 0
        n = int(rng.choice([132, 148, 152, 160]))
        plan, rows = check_schedule(B, Hq, Hkv, Sq, Sk, 128, off, causal, n)
        if plan["cut"]:
            seen_cut += 1
            assert plan["units"] > n
            assert np.bincount(rows[:, 0], minlength=n).max() <= 16
    assert seen_cut >= 10


def test_whole_units_when_no_cut_pays():
    # no more units than SMs, and D = 64, keep one unit per CTA
    assert not fa.fa_prefill_schedule(1, 8, 8, 2048, 16384, 128, 14336, True, 152)[0]["cut"]
    assert not fa.fa_prefill_schedule(1, 32, 8, 2048, 16384, 64, 14336, True, 152)[0]["cut"]


@pytest.mark.parametrize("args", [
    (1, 32, 8, 1, 16384, 128, 16383, True, 152),   # decode shape
    (1, 32, 8, 2048, 16384, 128, 14336, True, 0),  # no SMs
    (1, 32, 7, 2048, 16384, 128, 14336, True, 152),  # Hq % Hkv
    (1, 32, 8, 2048, 16384, 96, 14336, True, 152),   # D
    (1, 32, 8, 2048, 1024, 128, 0, True, 152),       # causal chunk past the keys
])
def test_invalid_arguments(args):
    with pytest.raises(fa.FaError) as e:
        fa.fa_prefill_schedule(*args)
    assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_cut_never_has_more_ctas_than_steps():
    """A cut over more CTAs than key-block steps would leave CTAs with empty ranges between a
    unit's pieces, whose merge waits for every CTA in between: the schedule then uses one CTA
    per step (the fused append forces the cut on small chunks)."""
    B, Hq, Hkv, Sq, Sk, D, off = 2, 8, 4, 300, 429, 128, 129
    W, _ = expected_segments(units_of(B, Hq, Sq, Sk, off, True), 1)
    assert W < 152
    plan, rows = fa.fa_prefill_schedule(B, Hq, Hkv, Sq, Sk, D, off, True, 152, force_cut=True)
    assert plan["ctas"] == W
    assert sorted(set(int(c) for c in rows[:, 0])) == list(range(W))
    check_schedule(B, Hq, Hkv, Sq, Sk, D, off, True, W, force=True)
