"""The chunked prefill that appends its own chunk to q4_0 caches in the same launch
(fa_prefill_append_q4_0), through the C ABI: the cache planes it writes are bit-exact against
the oracle's quantizer, the output matches the oracle's attention over the oracle-quantized
sequence, and it equals, bit for bit, the two-launch flow it replaces (fa_append_q4_0, then
fa_fwd_kv over the cache with the same scratch)."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes, q4_planes_gpu, sample_rows

pytestmark = pytest.mark.gpu


def prepare(fa, B, Hq, Hkv, S_new, pos0, cap, D, dtype, seed):
    """The full sequence's K and V (tokens 0 .. pos0 + S_new - 1), caches holding the first pos0
    tokens (and garbage everywhere else), and the chunk's queries."""
    Sk = pos0 + S_new
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, S_new, Sk, D, dtype, seed=seed)
    kc, vc = fa.q4_0_cache(B, Hkv, cap, D), fa.q4_0_cache(B, Hkv, cap, D)
    kc.buf.fill_(0x77)
    vc.buf.fill_(0x99)
    if pos0 > 0:
        fa.fa_append_q4_0(k[:, :, :pos0].contiguous().cuda(), kc, 0,
                          v[:, :, :pos0].contiguous().cuda(), vc)
    k_new = k[:, :, pos0:].contiguous()
    v_new = v[:, :, pos0:].contiguous()
    return q, k, v, k_new, v_new, kc, vc


def clone_cache(fa, c):
    d = fa.q4_0_cache(c.B, c.H, c.S, c.D)
    d.buf.copy_(c.buf)
    return d


CASES = [
    # B, Hq, Hkv, S_new, pos0, capacity, D, dtype: the 16K chunk (fused), an unaligned position
    # (a cache block holds old and new tokens), a small batch-2 shape, bf16, and D = 64 (which
    # runs as two launches)
    (1, 32, 8, 2048, 14336, 16384, 128, "f16"),
    (1, 8, 2, 700, 3000, 4096, 128, "f16"),
    (2, 8, 4, 300, 129, 1000, 128, "bf16"),
    (1, 4, 1, 256, 0, 512, 128, "f16"),
    (2, 4, 2, 200, 333, 600, 64, "f16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_fused_append_prefill(fa, case):
    B, Hq, Hkv, S_new, pos0, cap, D, dtype = case
    Sk = pos0 + S_new
    q, k, v, k_new, v_new, kc, vc = prepare(fa, B, Hq, Hkv, S_new, pos0, cap, D, dtype, seed=81)
    kc2, vc2 = clone_cache(fa, kc), clone_cache(fa, vc)
    qd, knd, vnd = q.cuda(), k_new.cuda(), v_new.cuda()
    need = fa.fa_prefill_append_workspace_bytes(B, Hq, Hkv, S_new, cap, D, pos0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    ws.fill_(0xEE)
    o = fa.fa_prefill_append_q4_0(qd, knd, vnd, kc, vc, pos0, workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    # the planes: the oracle's quantizer on the whole sequence, garbage kept past it
    for cache, src, fill in ((kc, k, 0x77), (vc, v, 0x99)):
        nib, sc = q4_planes_gpu(cache)
        want_nib, want_sc = oracle_q4_planes(src)
        assert np.array_equal(nib[:, :, :Sk], want_nib)
        assert np.array_equal(sc[:, :, :Sk], want_sc)
        assert (nib[:, :, Sk:] == fill).all()
        assert (sc[:, :, Sk:] == (fill | (fill << 8))).all()
    # the output: the oracle over its own quantization of the sequence
    rows = sample_rows(B, Hq, S_new, per_head=24, seed=S_new) if B * Hq * S_new > 20000 else None
    want = oracle.attention_q4_0(np64(q), oracle_q4_planes(k), oracle_q4_planes(v), causal=True,
                                 q_pos_offset=pos0, scale=D ** -0.5, rows=rows)
    got = np64(o) if rows is None else np64(o).reshape(-1, D)[rows]
    check_close(got, want, dtype, f"fused append + prefill {case}", q4=True)
    # the two-launch flow with the same scratch gives the same bits
    fa.fa_append_q4_0(knd, kc2, pos0, vnd, vc2)
    o2 = fa.fa_fwd_kv(qd, kc2, vc2, Sk=Sk, causal=True, q_pos_offset=pos0, workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    assert torch.equal(kc.buf, kc2.buf) and torch.equal(vc.buf, vc2.buf)
    if need > 0 and D == 128:
        # same cut schedule in both launches where the plan also cuts the two-launch prefill
        plain_need = fa.fa_workspace_bytes(B, Hq, Hkv, S_new, Sk, D, pos0, True)
        if plain_need > 0:
            assert torch.equal(o, o2)
    err = float((o.float() - o2.float()).abs().max())
    assert err <= 4e-3, err


def test_fused_append_replayed_from_a_cuda_graph(fa):
    """A captured fused call replayed with new chunk data: the small flag region is cleared by
    the call itself (a memset node), so every replay waits for its own phase-1 writes."""
    B, Hq, Hkv, S_new, pos0, cap, D = 1, 32, 8, 2048, 6144, 8192, 128
    q, k, v, k_new, v_new, kc, vc = prepare(fa, B, Hq, Hkv, S_new, pos0, cap, D, "f16", seed=83)
    qs, kns, vns = q.cuda(), k_new.cuda(), v_new.cuda()
    os_ = torch.empty_like(qs)
    ws = torch.empty(fa.fa_prefill_append_workspace_bytes(B, Hq, Hkv, S_new, cap, D, pos0),
                     dtype=torch.uint8, device="cuda")
    fa.fa_prefill_append_q4_0(qs, kns, vns, kc, vc, pos0, os_, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_prefill_append_q4_0(qs, kns, vns, kc, vc, pos0, os_, workspace=ws)
    for seed in (1, 2):
        g = torch.Generator(device="cuda").manual_seed(seed)
        kn = torch.randn(k_new.shape, generator=g, device="cuda").half()
        vn = torch.randn(v_new.shape, generator=g, device="cuda").half()
        kns.copy_(kn)
        vns.copy_(vn)
        graph.replay()
        torch.cuda.synchronize()
        kc2, vc2 = clone_cache(fa, kc), clone_cache(fa, vc)
        eager = fa.fa_prefill_append_q4_0(qs, kn, vn, kc2, vc2, pos0, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(kc.buf, kc2.buf) and torch.equal(vc.buf, vc2.buf)
        assert torch.equal(os_, eager), seed
    assert fa.fa_get_status() == fa.FA_OK
