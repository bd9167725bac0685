"""Independent K and V cache formats, caches larger than the filled length, and appending a
chunk to a q4_0 cache (fa_fwd_kv, fa_append_q4_0), against the f64 oracle through the C ABI.

The oracle sees each side as the kernel does: a dense side as its f16/bf16 values, a q4_0 side
as the oracle's own quantization of the same values, dequantized exactly.  Tolerance: max-abs
1e-2 (f16) / 2e-2 (bf16); q4_0 planes written by an append are compared bit for bit."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes, q4_planes_gpu, sample_rows

pytestmark = pytest.mark.gpu


def side(fa, x, fmt):
    """(device operand, f64 values the oracle uses) for one K or V side."""
    if fmt == "q4_0":
        nib, sc = oracle_q4_planes(x)
        return fa.fa_quantize_q4_0(x.cuda()), oracle.dequantize_q4_0(nib, sc)
    return x.cuda(), np64(x)


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, k_fmt, v_fmt
    (1, 4, 2, 200, 450, 128, True, 250, "f16", "dense", "q4_0"),
    (1, 4, 2, 200, 450, 128, True, 250, "f16", "q4_0", "dense"),
    (2, 4, 1, 130, 333, 64, True, 203, "bf16", "dense", "q4_0"),
    (1, 2, 2, 300, 257, 128, False, 0, "bf16", "q4_0", "dense"),
    (1, 8, 2, 1, 3000, 128, True, 2999, "f16", "dense", "q4_0"),    # decode
    (2, 32, 8, 1, 4097, 128, True, 4096, "bf16", "q4_0", "dense"),  # decode
    (1, 6, 2, 1, 777, 64, True, 776, "f16", "dense", "q4_0"),       # decode, group of 3
    (1, 4, 4, 1, 2048, 64, False, 0, "bf16", "q4_0", "dense"),      # decode, non-causal
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_mixed_formats_match_oracle(fa, case):
    B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, kf, vf = case
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, Sk, D, dtype, seed=21)
    kd, k64 = side(fa, k, kf)
    vd, v64 = side(fa, v, vf)
    o = fa.fa_fwd_kv(q.cuda(), kd, vd, causal=causal, q_pos_offset=off, scale=D ** -0.5)
    assert fa.fa_get_status() == fa.FA_OK
    want = oracle.attention(np64(q), k64, v64, causal=causal, q_pos_offset=off, scale=D ** -0.5)
    check_close(np64(o), want, dtype, f"{kf} K / {vf} V {case}", q4="q4_0" in (kf, vf))


@pytest.mark.parametrize("fmt", [("dense", "dense"), ("q4_0", "q4_0"), ("dense", "q4_0")])
@pytest.mark.parametrize("Sq", [1, 192])
def test_cache_larger_than_filled_length(fa, fmt, Sq):
    """Tokens past Sk in a cache of larger capacity are never read: garbage there (huge values)
    must not change the result."""
    B, Hq, Hkv, D, Sk, cap = 1, 8, 2, 128, 1000, 1536
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, cap, D, "f16", seed=23)
    k[:, :, Sk:] = 3.0e4
    v[:, :, Sk:] = -3.0e4
    kd, _ = side(fa, k, fmt[0])
    vd, _ = side(fa, v, fmt[1])
    _, kf64 = side(fa, k[:, :, :Sk].contiguous(), fmt[0])
    _, vf64 = side(fa, v[:, :, :Sk].contiguous(), fmt[1])
    o = fa.fa_fwd_kv(q.cuda(), kd, vd, Sk=Sk, causal=True)
    assert fa.fa_get_status() == fa.FA_OK
    want = oracle.attention(np64(q), kf64, vf64, causal=True, q_pos_offset=Sk - Sq,
                            scale=D ** -0.5)
    check_close(np64(o), want, "f16", f"capacity {cap} > Sk {Sk}, {fmt}", q4="q4_0" in fmt)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_append_writes_the_quantizer_bits_in_place(fa, dtype):
    """Chunks appended at their positions give the planes of quantizing the whole sequence, and
    the tokens outside the appended range keep their bytes."""
    B, H, D, cap = 2, 3, 128, 700
    chunks = [(0, 256), (256, 300), (556, 100)]
    full = fa_inputs.make_tensors(B, H, H, 1, 656, D, dtype, seed=29)[1]
    fullv = fa_inputs.make_tensors(B, H, H, 1, 656, D, dtype, seed=31)[1]
    kc, vc = fa.q4_0_cache(B, H, cap, D), fa.q4_0_cache(B, H, cap, D)
    kc.buf.fill_(0x5A)
    vc.buf.fill_(0xA5)
    for pos0, n in chunks:
        fa.fa_append_q4_0(full[:, :, pos0:pos0 + n].contiguous().cuda(), kc, pos0,
                          fullv[:, :, pos0:pos0 + n].contiguous().cuda(), vc)
    assert fa.fa_get_status() == fa.FA_OK
    for cache, src, fill in ((kc, full, 0x5A), (vc, fullv, 0xA5)):
        nib, sc = q4_planes_gpu(cache)
        want_nib, want_sc = oracle_q4_planes(src)
        assert np.array_equal(nib[:, :, :656], want_nib)
        assert np.array_equal(sc[:, :, :656], want_sc)
        assert (nib[:, :, 656:] == fill).all()
        assert (sc[:, :, 656:] == (fill | (fill << 8))).all()


def test_append_then_chunked_prefill_over_the_cache(fa):
    """The chunked-prefill flow over a q4_0 cache: append chunk 1 and attend to it, append chunk
    2 and attend to both, with the cache allocated for 4096 tokens."""
    B, Hq, Hkv, D, cap = 1, 32, 8, 128, 4096
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 2048, 2048, D, "f16", seed=33)
    kc, vc = fa.q4_0_cache(B, Hkv, cap, D), fa.q4_0_cache(B, Hkv, cap, D)
    for c0 in (0, 1024):
        fa.fa_append_q4_0(k[:, :, c0:c0 + 1024].contiguous().cuda(), kc, c0,
                          v[:, :, c0:c0 + 1024].contiguous().cuda(), vc)
        qc = q[:, :, c0:c0 + 1024].contiguous()
        o = fa.fa_fwd_kv(qc.cuda(), kc, vc, Sk=c0 + 1024, causal=True, q_pos_offset=c0)
        assert fa.fa_get_status() == fa.FA_OK
        kp = oracle_q4_planes(k[:, :, :c0 + 1024].contiguous())
        vp = oracle_q4_planes(v[:, :, :c0 + 1024].contiguous())
        rows = sample_rows(B, Hq, 1024, per_head=8, seed=c0)
        want = oracle.attention_q4_0(np64(qc), kp, vp, causal=True, q_pos_offset=c0,
                                     scale=D ** -0.5, rows=rows)
        check_close(np64(o).reshape(-1, D)[rows], want, "f16", f"chunk at {c0}", q4=True)


def test_fwd_kv_with_equal_formats_equals_fa_fwd_ex(fa):
    q, k, v = fa_inputs.make_tensors(1, 8, 2, 256, 1024, 128, "bf16", seed=37, device="cuda")
    kq, vq = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    a = fa.fa_fwd_ex(q, kq, vq)
    b = fa.fa_fwd_kv(q, kq, vq)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_mixed_decode_at_the_benchmarked_size(fa):
    """f16 K with a q4_0 V, 4 sequences x 65 536 keys, GQA 32/8, D = 128: the benchmark's mixed
    decode leg, every output element against the oracle (one sequence at a time, so the f64
    copies stay a few hundred MB)."""
    w = fa_inputs.WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"]
    q, k, v = fa_inputs.make_qkv(w)
    vd = fa.fa_quantize_q4_0(v.cuda())
    ws = torch.empty(fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, 1, w.Sk, w.D, w.q_pos_offset, True),
                     dtype=torch.uint8, device="cuda")
    o = fa.fa_fwd_kv(q.cuda(), k.cuda(), vd, causal=True, q_pos_offset=w.q_pos_offset,
                     workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    got = np64(o)
    for b in range(w.B):
        vn, vs = oracle_q4_planes(v[b:b + 1].contiguous())
        want = oracle.attention(np64(q[b:b + 1]), np64(k[b:b + 1]), oracle.dequantize_q4_0(vn, vs),
                                causal=True, q_pos_offset=w.q_pos_offset, scale=w.scale)
        check_close(got[b:b + 1], want, w.dtype, f"f16 K + q4_0 V decode, sequence {b}", q4=True)


def test_append_at_the_benchmarked_size(fa):
    """The benchmark's append leg: a 16 384-token chunk of K and V (B 4, 8 heads, D 128) written
    at position 32 768 of q4_0 caches of 65 536 tokens.  The written planes are bit-exact against
    the oracle's quantizer; every byte outside the chunk keeps its fill."""
    B, H, D, cap, pos0, n = 4, 8, 128, 65536, 32768, 16384
    kn = fa_inputs.make_tensors(B, H, H, 1, n, D, "f16", seed=71)[1]
    vn = fa_inputs.make_tensors(B, H, H, 1, n, D, "f16", seed=73)[1]
    kc, vc = fa.q4_0_cache(B, H, cap, D), fa.q4_0_cache(B, H, cap, D)
    kc.buf.fill_(0x3C)
    vc.buf.fill_(0xC3)
    fa.fa_append_q4_0(kn.cuda(), kc, pos0, vn.cuda(), vc)
    assert fa.fa_get_status() == fa.FA_OK
    for cache, src, fill in ((kc, kn, 0x3C), (vc, vn, 0xC3)):
        nib, sc = q4_planes_gpu(cache)
        want_nib, want_sc = oracle_q4_planes(src)
        assert np.array_equal(nib[:, :, pos0:pos0 + n], want_nib)
        assert np.array_equal(sc[:, :, pos0:pos0 + n], want_sc)
        for lo, hi in ((0, pos0), (pos0 + n, cap)):
            assert (nib[:, :, lo:hi] == fill).all()
            assert (sc[:, :, lo:hi] == (fill | (fill << 8))).all()
