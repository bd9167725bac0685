"""Variable-length batched decode over paged K/V pools (fa_decode_paged) against the f64 oracle,
through the C ABI.  Each sequence's pages sit at shuffled places of a shared pool, its last page
is partly filled (the rest holds unrelated values), and unused pages hold garbage; the oracle
sees each sequence's own keys gathered in order (q4_0 sides: the oracle's own quantization of
the pool, dequantized exactly).  Tolerance: max-abs 1e-2 (f16) / 2e-2 (bf16)."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes

pytestmark = pytest.mark.gpu


def build_pool(fa, lens, Hkv, D, page, dtype, kf, vf, seed, extra_pages=3):
    """Pools holding each sequence's K/V in shuffled pages; returns device pools, the block
    table, and per-sequence f64 K/V for the oracle."""
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    pps = max((n + page - 1) // page for n in lens)
    need = sum((n + page - 1) // page for n in lens)
    NP = need + extra_pages
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16
    kpool = torch.randn(NP, Hkv, page, D, generator=g).to(tdt)
    vpool = torch.randn(NP, Hkv, page, D, generator=g).to(tdt)
    perm = torch.randperm(NP, generator=g).tolist()
    table = torch.full((B, pps), -7, dtype=torch.int32)  # unused entries are never read
    nxt = 0
    for b, n in enumerate(lens):
        for p in range((n + page - 1) // page):
            table[b, p] = perm[nxt]
            nxt += 1
    # what the oracle sees of each pool: its values, or the oracle's q4_0 round trip
    def view(pool, fmt):
        if fmt == "q4_0":
            nib, sc = oracle_q4_planes(pool)
            return fa.fa_quantize_q4_0(pool.cuda()), oracle.dequantize_q4_0(nib, sc)
        return pool.cuda(), np64(pool)
    kd, k64 = view(kpool, kf)
    vd, v64 = view(vpool, vf)
    seqs = []
    for b, n in enumerate(lens):
        pages = [int(table[b, p]) for p in range((n + page - 1) // page)]
        ks = np.concatenate([k64[p] for p in pages], axis=1)[:, :n]  # [Hkv, n, D]
        vs = np.concatenate([v64[p] for p in pages], axis=1)[:, :n]
        seqs.append((ks, vs))
    return kd, vd, table.cuda(), seqs


CASES = [
    # lens, Hq, Hkv, D, page, dtype, k_fmt, v_fmt
    ([5000, 257, 1, 3001], 32, 8, 128, 128, "f16", "q4_0", "q4_0"),
    ([129, 2048, 700], 8, 2, 128, 256, "bf16", "q4_0", "q4_0"),
    ([1000, 64, 1500], 16, 2, 64, 128, "f16", "q4_0", "q4_0"),
    ([300, 1, 999, 4096], 8, 8, 128, 64, "f16", "dense", "dense"),
    ([777, 2000], 12, 4, 128, 128, "bf16", "dense", "q4_0"),
    ([100, 3000, 513], 8, 1, 64, 128, "f16", "q4_0", "dense"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c[1:])) + f"-B{len(c[0])}")
def test_paged_varlen_decode_matches_oracle(fa, case):
    lens, Hq, Hkv, D, page, dtype, kf, vf = case
    B = len(lens)
    kd, vd, table, seqs = build_pool(fa, lens, Hkv, D, page, dtype, kf, vf, seed=sum(lens))
    q = fa_inputs.make_tensors(B, Hq, Hkv, 1, 1, D, dtype, seed=41)[0]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = fa.fa_decode_paged(q.cuda(), kd, vd, table, sl)
    assert fa.fa_get_status() == fa.FA_OK
    got = np64(o)
    for b in range(B):
        ks, vs = seqs[b]
        want = oracle.attention(np64(q[b:b + 1]), ks[None], vs[None], causal=False,
                                scale=D ** -0.5)
        check_close(got[b:b + 1], want, dtype, f"sequence {b} ({lens[b]} keys)",
                    q4="q4_0" in (kf, vf))


def test_paged_decode_repeated_calls_and_stale_workspace(fa):
    lens, Hq, Hkv, D, page = [4000, 700, 2500, 33], 32, 8, 128, 128
    kd, vd, table, _ = build_pool(fa, lens, Hkv, D, page, "f16", "q4_0", "q4_0", seed=5)
    q = fa_inputs.make_tensors(4, Hq, Hkv, 1, 1, D, "f16", seed=43, device="cuda")[0]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = torch.full((fa.load().fa_decode_paged_workspace_bytes(4, Hq, Hkv, D, page,
                                                               table.shape[1]),),
                    255, dtype=torch.uint8, device="cuda")
    first = fa.fa_decode_paged(q, kd, vd, table, sl, workspace=ws)
    for _ in range(5):
        again = fa.fa_decode_paged(q, kd, vd, table, sl, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(first, again)
    assert fa.fa_get_status() == fa.FA_OK


def test_bad_page_number_and_length_are_reported_not_read(fa):
    """A page number past the pool or a zero length is caught by the kernel's own checks: the
    call completes (out-of-pool tiles read as zeros, their scale rows are not loaded) and
    fa_get_status reports FA_ERR_INVALID_ARG."""
    lens, Hq, Hkv, D, page = [300, 200], 8, 2, 128, 128
    kd, vd, table, _ = build_pool(fa, lens, Hkv, D, page, "f16", "q4_0", "q4_0", seed=7)
    q = fa_inputs.make_tensors(2, Hq, Hkv, 1, 1, D, "f16", seed=47, device="cuda")[0]
    bad = table.clone()
    bad[0, 1] = 1 << 20
    fa.fa_decode_paged(q, kd, vd, bad, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert fa.fa_get_status() == fa.FA_ERR_INVALID_ARG
    fa.fa_decode_paged(q, kd, vd, table, torch.tensor([0, 200], dtype=torch.int32, device="cuda"))
    assert fa.fa_get_status() == fa.FA_ERR_INVALID_ARG
    fa.fa_decode_paged(q, kd, vd, table, torch.tensor(lens, dtype=torch.int32, device="cuda"))
    assert fa.fa_get_status() == fa.FA_OK


@pytest.mark.parametrize("lens", [[65536] * 4, [65536, 32768, 16384, 8192]],
                         ids=["65536x4", "varlen_65536_32768_16384_8192"])
def test_paged_decode_at_the_benchmarked_sizes(fa, lens):
    """The benchmark's paged legs: q4_0 K and V pools of 256-token pages in shuffled order, GQA
    32/8, D = 128, every output element against the oracle.  The oracle takes each sequence's
    pages, gathered in order, as q4_0 planes of its own quantizer (nothing is expanded to f64
    beyond one key at a time)."""
    Hq, Hkv, D, page = 32, 8, 128, 256
    B = len(lens)
    npages = [n // page for n in lens]
    NP = sum(npages)
    g = torch.Generator().manual_seed(1006)
    perm = torch.randperm(NP, generator=g)
    table = torch.zeros(B, max(npages), dtype=torch.int32)
    at = 0
    for b, n in enumerate(npages):
        table[b, :n] = perm[at:at + n].to(torch.int32)
        at += n
    kpool = torch.randn(NP, Hkv, page, D, generator=g).to(torch.float16)
    vpool = torch.randn(NP, Hkv, page, D, generator=g).to(torch.float16)
    q = torch.randn(B, Hq, 1, D, generator=g).to(torch.float16)
    kd, vd = fa.fa_quantize_q4_0(kpool.cuda()), fa.fa_quantize_q4_0(vpool.cuda())
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    tab = table.cuda()
    ws = torch.empty(fa.load().fa_decode_paged_workspace_bytes(B, Hq, Hkv, D, page,
                                                              table.shape[1]),
                     dtype=torch.uint8, device="cuda")
    o = fa.fa_decode_paged(q.cuda(), kd, vd, tab, sl, workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    got = np64(o)
    kn, ks = oracle_q4_planes(kpool)
    del kpool
    vn, vs = oracle_q4_planes(vpool)
    del vpool
    for b, n in enumerate(lens):
        pages = table[b, :npages[b]].numpy()

        def seq(plane):  # [pages, Hkv, page, X] -> [1, Hkv, n, X]
            return np.ascontiguousarray(plane[pages].transpose(1, 0, 2, 3)
                                        .reshape(Hkv, -1, plane.shape[-1])[None, :, :n])

        want = oracle.attention_q4_0(np64(q[b:b + 1]), (seq(kn), seq(ks)), (seq(vn), seq(vs)),
                                     causal=True, q_pos_offset=n - 1, scale=D ** -0.5)
        check_close(got[b:b + 1], want, "f16", f"paged sequence {b} ({n} keys)", q4=True)
