"""The decode kernels' work split on the host (no device), read back through fa_decode_schedule
and checked against the plan restated from its definition.

Uniform batch (fa_fwd, Sq = 1): every (sequence, kv head) is cut into the same number of splits;
the splits fill one wave of resident CTAs (3 per SM with q4_0 K and V, else 2), up to one split
per tile, and share the key tiles out as evenly as whole tiles allow, the longer splits first.  Paged batch (fa_decode_paged): the CTAs of a kv head, one wave's
worth (at least one per sequence), are shared out over the sequences: sequence b gets
1 + floor((CTAs - B) * tiles_b / total tiles) consecutive CTAs, and its key tiles are shared out
over that many splits as evenly as whole tiles allow (the longer splits first; a sequence with
fewer tiles than splits leaves its last splits empty).  Either way, every key of every sequence must
belong to exactly one split.
"""
import numpy as np
import pytest

import quantized_kv_cache_sm_gb300 as fa


@pytest.fixture(autouse=True)
def _library(built):
    return built


def tile_keys(kf, vf):
    return 128 if "q4_0" in (kf, vf) else 64


def ctas_per_sm(kf, vf):
    return 3 if (kf, vf) == ("q4_0", "q4_0") else 2


def check_cover(rows, length):
    """Rows of one sequence: in split order, contiguous, covering [0, length) once."""
    ns = rows.shape[0]
    assert (rows[:, 1] == np.arange(ns)).all() and (rows[:, 2] == ns).all()
    live = rows[rows[:, 4] > rows[:, 3]]
    assert live.shape[0] >= 1 and live[0, 3] == 0 and live[-1, 4] == length
    assert (live[1:, 3] == live[:-1, 4]).all()
    # splits past the end of a short sequence are empty, never partial or overlapping
    assert (rows[live.shape[0]:, 3] >= length).all()


@pytest.mark.parametrize("fmt", [("q4_0", "q4_0"), ("dense", "dense"), ("dense", "q4_0")])
@pytest.mark.parametrize("B,Hkv,Sk,n", [(4, 8, 65536, 152), (1, 8, 1, 152), (2, 4, 1000, 7),
                                        (8, 8, 131072, 148), (1, 1, 300, 1), (3, 2, 64, 152)])
def test_uniform_split(fmt, B, Hkv, Sk, n):
    rows = fa.fa_decode_schedule(B, Hkv, n, Sk=Sk, k_format=fmt[0], v_format=fmt[1])
    tile = tile_keys(*fmt)
    ns = int(rows[0, 2])
    assert rows.shape == (B * ns, 5)
    for b in range(B):
        r = rows[rows[:, 0] == b]
        check_cover(r, Sk)
        assert (r[:, 4] > r[:, 3]).all()  # no empty split in a uniform batch
        # whole tiles (the last split may end at Sk), lengths in tiles never growing, within one
        tiles = -(-(r[:, 4] - r[:, 3]) // tile)
        assert (r[:-1, 4] % tile == 0).all()
        assert (np.diff(tiles) <= 0).all() and tiles.max() - tiles.min() <= 1
    assert ns == 1 or B * Hkv * ns <= n * ctas_per_sm(*fmt)  # one wave
    want = expected_uniform(B, Hkv, Sk, n, fmt)
    assert [tuple(int(x) for x in row[3:5]) for row in rows[rows[:, 0] == 0]] == want


def even_split(length, ns, tile):
    """(first key, end key) of ns splits sharing the ceil(length / tile) tiles out as evenly as
    whole tiles allow, the first (tiles mod ns) splits taking one more."""
    tiles = -(-length // tile)
    out, t = [], 0
    for s in range(ns):
        nt = tiles // ns + (1 if s < tiles % ns else 0)
        out.append((min(length, t * tile), min(length, (t + nt) * tile)))
        t += nt
    return out


def expected_uniform(B, Hkv, Sk, n, fmt):
    """As many splits as one wave holds (at least 1, at most one per tile and 1024); the key tiles
    are shared out as evenly as whole tiles allow, the first (tiles mod splits) splits taking one
    more.  Returns the (first key, end key) of each split."""
    tile = tile_keys(*fmt)
    ns = min(max(1, n * ctas_per_sm(*fmt) // (B * Hkv)), -(-Sk // tile), 1024)
    return even_split(Sk, ns, tile)


def expected_paged(lens, cap, Hkv, n, fmt):
    tile = tile_keys(*fmt)
    B = len(lens)
    nt = max(B, n * ctas_per_sm(*fmt) // Hkv)
    L = [max(1, min(int(x), cap)) for x in lens]
    t = [-(-x // tile) for x in L]
    total = sum(t)
    ns = [1 + (nt - B) * tb // total for tb in t]
    return nt, L, ns, tile


@pytest.mark.parametrize("fmt", [("q4_0", "q4_0"), ("dense", "q4_0"), ("dense", "dense")])
def test_paged_split_random_mixes(fmt):
    rng = np.random.default_rng(11)
    for trial in range(200):
        B = int(rng.integers(1, 17))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        page = 128 * int(rng.integers(1, 5))
        pps = int(rng.integers(1, 600))
        cap = page * pps
        lens = rng.integers(1, cap + 1, size=B)
        if trial % 7 == 0:
            lens[0] = 1
        n = int(rng.choice([1, 7, 100, 148, 152]))
        rows = fa.fa_decode_schedule(B, Hkv, n, seq_lens=lens, page_size=page, pages_per_seq=pps,
                                     k_format=fmt[0], v_format=fmt[1])
        nt, L, ns, tile = expected_paged(lens, cap, Hkv, n, fmt)
        assert rows.shape == (nt, 5)
        c = 0
        for b in range(B):
            r = rows[c:c + ns[b]]
            assert (r[:, 0] == b).all(), (trial, b)
            check_cover(r, L[b])
            assert [tuple(int(x) for x in row[3:5]) for row in r] == even_split(L[b], ns[b], tile)
            c += ns[b]
        assert c <= nt and (rows[c:, 0] == -1).all()


def test_paged_lengths_out_of_range_are_clamped():
    """A length of 0 (or one past the table's capacity) is planned as 1 key (or the capacity),
    as the kernel plans it while reporting the bad length."""
    rows = fa.fa_decode_schedule(3, 8, 152, seq_lens=[0, 5000, 10 ** 6], page_size=256,
                                 pages_per_seq=16)
    cap = 256 * 16
    for b, want in enumerate([1, cap, cap]):
        check_cover(rows[rows[:, 0] == b], want)


def test_paged_varlen_batch_of_the_benchmark():
    """The 65 536 / 32 768 / 16 384 / 8 192-key batch on 152 SMs: 57 CTAs per kv head, 53 beyond
    one per sequence, shared 1 + floor(53 * tiles / 960) = 29 / 15 / 8 / 4 (one left idle)."""
    rows = fa.fa_decode_schedule(4, 8, 152, seq_lens=[65536, 32768, 16384, 8192], page_size=256,
                                 pages_per_seq=256)
    assert rows.shape[0] == 152 * 3 // 8
    assert [int((rows[:, 0] == b).sum()) for b in range(4)] == [29, 15, 8, 4]
    assert int((rows[:, 0] == -1).sum()) == 1


@pytest.mark.parametrize("kw", [
    dict(Sk=0),                                                       # empty uniform batch
    dict(seq_lens=[5], page_size=100, pages_per_seq=4),               # page not a whole tile
    dict(seq_lens=[5], page_size=128, pages_per_seq=0),
    dict(Sk=16, k_format="q8"),
])
def test_invalid_arguments(kw):
    with pytest.raises((fa.FaError, KeyError)):
        fa.fa_decode_schedule(1, 8, 152, **kw)
