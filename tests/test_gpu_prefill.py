"""Prefill kernel (Sq >= 2) against the f64 oracle, through the C ABI.

Small and ragged shapes are compared on every output element.  The full-size chunked-prefill
workloads are compared here on sampled rows (tile edges, last rows, random rows of every head)
with the per-row frame-move counts, through the one-unit-per-CTA launch (no scratch passed);
tests/test_gpu_prefill_full.py compares every row of them, through both the one-unit-per-CTA
launch and the cut-schedule launch the benchmark times.  Tolerance: the absolute and relative
bounds of gpu_common."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes, sample_rows

pytestmark = pytest.mark.gpu


def run_case(fa, B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, kv, seed, rows=None, ramp=False,
             counts=False):
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, Sk, D, dtype, seed=seed, ramp=ramp)
    scale = D ** -0.5
    qd = q.cuda()
    rc = torch.full((B, Hq, Sq), -1, dtype=torch.int32, device="cuda") if counts else None
    if kv == "q4_0":
        kq = fa.fa_quantize_q4_0(k.cuda())
        vq = fa.fa_quantize_q4_0(v.cuda())
        o = fa.fa_fwd_ex(qd, kq, vq, causal=causal, q_pos_offset=off, scale=scale,
                         rescale_count=rc)
        kp, vp = oracle_q4_planes(k), oracle_q4_planes(v)
        want = oracle.attention_q4_0(np64(q), kp, vp, causal=causal, q_pos_offset=off,
                                     scale=scale, rows=rows)
    else:
        o = fa.fa_fwd_ex(qd, k.cuda(), v.cuda(), causal=causal, q_pos_offset=off, scale=scale,
                         rescale_count=rc)
        want = oracle.attention(np64(q), np64(k), np64(v), causal=causal, q_pos_offset=off,
                                scale=scale, rows=rows)
    assert fa.fa_get_status() == fa.FA_OK
    got = np64(o)
    if rows is not None:
        got = got.reshape(-1, D)[rows]
    err = check_close(got, want, dtype, f"B{B} H{Hq}/{Hkv} Sq{Sq} Sk{Sk} D{D} {dtype} {kv}",
                      q4=kv == "q4_0")
    return err, (rc.cpu().numpy() if counts else None)


SMALL = [
    # B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, kv
    (1, 4, 2, 200, 200, 128, True, 0, "f16", "dense"),
    (2, 4, 4, 130, 333, 64, True, 203, "f16", "dense"),
    (1, 8, 2, 64, 1000, 128, True, 936, "bf16", "dense"),
    (1, 2, 2, 300, 257, 128, False, 0, "f16", "dense"),
    (1, 3, 1, 128, 128, 64, True, 0, "bf16", "dense"),
    (1, 2, 1, 2, 5, 128, True, 3, "f16", "dense"),
    (1, 4, 2, 100, 500, 128, True, 123, "f16", "dense"),
    (1, 2, 1, 257, 640, 64, False, 0, "bf16", "dense"),
    (1, 4, 2, 200, 450, 128, True, 250, "f16", "q4_0"),
    (1, 2, 1, 130, 130, 64, True, 0, "bf16", "q4_0"),
    (2, 4, 1, 77, 301, 128, False, 0, "f16", "q4_0"),
    (1, 2, 2, 3, 1027, 128, True, 1024, "bf16", "q4_0"),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "-".join(map(str, c)))
def test_prefill_small_full_compare(fa, case):
    run_case(fa, *case, seed=7)


@pytest.mark.parametrize("kv", ["dense", "q4_0"])
@pytest.mark.parametrize("mapping", ["one_tile_per_cta", "tile_pairs"])
def test_unit_mapping_on_either_side_of_the_threshold(fa, mapping, kv):
    """One unit per CTA gives each 128-row query tile a CTA of its own when twice the pair units
    fit on the SMs at once (2 x units <= SMs), else a pair of tiles per CTA.  A shape on each
    side of that threshold for this device's SM count, every element against the oracle; three
    ragged query tiles, so the last pair has no tile B either way."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pairs = 2  # per head: tiles (0, 1) and (2, -)
    Hq = max(1, sms // (2 * pairs)) if mapping == "one_tile_per_cta" else sms // (2 * pairs) + 1
    assert (2 * Hq * pairs <= sms) == (mapping == "one_tile_per_cta")
    run_case(fa, 1, Hq, 1, 3 * 128 - 37, 600, 128, True, 600 - (3 * 128 - 37), "f16", kv, seed=5)


@pytest.mark.parametrize("D,dtype", [(128, "f16"), (64, "bf16")])
def test_score_ramp_on_lone_query_tiles(fa, D, dtype):
    """Frame moves in the one-tile-per-CTA launch, where a dense tile's key blocks alternate
    between the two S buffers and each O rescale must wait for the previous block's PV.  The
    2.0-per-block score ramp moves every row's frame about every fifth block; every element is
    checked against the oracle and every row must have moved its frame more than once."""
    B, Hq, Hkv, Sq, Sk = 1, 8, 2, 256, 4096
    assert 2 * B * Hq <= torch.cuda.get_device_properties(0).multi_processor_count
    _, counts = run_case(fa, B, Hq, Hkv, Sq, Sk, D, True, Sk - Sq, dtype, "dense", seed=3,
                         ramp=True, counts=True)
    per_row = counts.reshape(-1, Sq)
    assert (per_row >= 2).all(), "the deferred rescale branch never ran on some row"
    nblocks = (Sk - Sq + np.arange(Sq)) // 128 + 1
    ratio = per_row / (1 + (nblocks - 1) / 5.0)[None, :]
    assert 0.7 < ratio.mean() < 1.3, ratio.mean()


def test_selfattn_b2_s512_h8_d64_full(fa):
    w = fa_inputs.WORKLOADS["selfattn_b2_s512_h8_d64_f16"]
    err, _ = run_case(fa, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True, 0, w.dtype, "dense", w.seed)
    assert err < 5e-3


@pytest.mark.parametrize("kv", ["dense", "q4_0"])
def test_one_tile_launch_replayed_from_a_cuda_graph(fa, kv):
    """The B2 S512 D64 self-attention (one query tile per CTA; dense K/V alternates S buffers)
    captured once in a CUDA graph: replays with new query rows copied in must give the eager
    result bit for bit."""
    w = fa_inputs.WORKLOADS["selfattn_b2_s512_h8_d64_f16"]
    q, k, v = fa_inputs.make_tensors(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.dtype, seed=17,
                                     device="cuda")
    if kv == "q4_0":
        k, v = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    qs, os_ = q.clone(), torch.empty_like(q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fa.fa_fwd_ex(qs, k, v, os_, causal=True, q_pos_offset=0, stream=side)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        fa.fa_fwd_ex(qs, k, v, os_, causal=True, q_pos_offset=0, stream=side)
    for seed in (1, 2, 3):
        qn = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(seed),
                         device="cuda").to(q.dtype)
        qs.copy_(qn)
        graph.replay()
        torch.cuda.synchronize()
        want = fa.fa_fwd_ex(qn, k, v, causal=True, q_pos_offset=0)
        torch.cuda.synchronize()
        assert torch.equal(os_, want), (kv, seed)
    assert fa.fa_get_status() == fa.FA_OK


def test_chunked_prefill_2k_full(fa):
    w = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk2048_f16"]
    run_case(fa, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True, w.q_pos_offset, w.dtype, "dense",
             w.seed)


@pytest.mark.parametrize("name", ["prefill_gqa32x8_d128_sq2048_sk8192_f16",
                                  "prefill_gqa32x8_d128_sq2048_sk8192_bf16",
                                  "prefill_gqa32x8_d128_sq2048_sk16384_f16",
                                  "prefill_gqa32x8_d128_sq2048_sk16384_bf16",
                                  "prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16"])
def test_chunked_prefill_long_sampled(fa, name):
    w = fa_inputs.WORKLOADS[name]
    rows = sample_rows(w.B, w.Hq, w.Sq, per_head=14, seed=w.Sk)
    _, counts = run_case(fa, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True, w.q_pos_offset, w.dtype,
                         w.kv_format, w.seed, rows=rows, counts=True)
    # N(0,1) scores never outgrow the first block's frame by 10: no deferred rescale fires
    assert counts.min() >= 1 and counts.max() <= 2


@pytest.mark.parametrize("name", ["prefill_gqa32x8_d128_sq2048_sk8192_f16_ramp",
                                  "prefill_gqa32x8_d128_sq2048_sk16384_f16_ramp"])
def test_score_ramp_drives_deferred_rescale(fa, name):
    """A per-key bias rising 2.0 per 128-key block: a row's block max outgrows its frame by the
    10-point margin about every fifth block, so the deferred O/l rescale runs ~Sk/640 times per
    row, and the output still matches the oracle."""
    w = fa_inputs.WORKLOADS[name]
    rows = sample_rows(w.B, w.Hq, w.Sq, per_head=10, seed=1)
    _, counts = run_case(fa, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, True, w.q_pos_offset, w.dtype,
                         "dense", w.seed, rows=rows, ramp=True, counts=True)
    nblocks = (w.q_pos_offset + np.arange(w.Sq)) // 128 + 1      # key blocks each row sees
    per_row = counts.reshape(-1, w.Sq)
    assert (per_row >= 2).all(), "the deferred rescale branch never ran on some row"
    expect = 1 + (nblocks - 1) / 5.0
    ratio = per_row / expect[None, :]
    assert 0.7 < ratio.mean() < 1.3, ratio.mean()
    assert ratio.min() > 0.5 and ratio.max() < 1.6


def test_fa_fwd_allocating_equals_ex(fa):
    q, k, v = fa_inputs.make_tensors(1, 4, 2, 256, 512, 128, "f16", seed=3, device="cuda")
    o1 = fa.fa_fwd(q, k, v)
    o2 = fa.fa_fwd_ex(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_status_after_many_calls(fa):
    q, k, v = fa_inputs.make_tensors(1, 8, 2, 512, 4096, 128, "bf16", seed=5, device="cuda")
    for _ in range(20):
        fa.fa_fwd(q, k, v)
    assert fa.fa_get_status() == fa.FA_OK


@pytest.mark.parametrize("shape", [(1, 2, 1, 257, 640, 64, False, 0, "bf16"),
                                   (1, 4, 2, 300, 300, 128, True, 0, "f16"),
                                   (2, 4, 4, 130, 260, 64, True, 130, "f16")],
                         ids=lambda c: "-".join(map(str, c)))
def test_prefill_repeated_calls_stay_exact(fa, shape):
    """Short key ranges (2-5 blocks) leave the least slack between the last PV MMA and the
    epilogue's read of O; repeated launches must all match the oracle (a synchronisation race
    would show up as an occasional wrong row)."""
    B, Hq, Hkv, Sq, Sk, D, causal, off, dtype = shape
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, Sk, D, dtype, seed=17)
    want = oracle.attention(np64(q), np64(k), np64(v), causal=causal, q_pos_offset=off,
                            scale=D ** -0.5)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    outs = [fa.fa_fwd(qd, kd, vd, causal=causal, q_pos_offset=off, scale=D ** -0.5)
            for _ in range(40)]
    assert fa.fa_get_status() == fa.FA_OK
    for o in outs:
        check_close(np64(o), want, dtype, "repeated prefill")


E10 = float(np.exp(10.0))


@pytest.mark.parametrize("launch", ["whole_units", "cut_schedule"])
@pytest.mark.parametrize("name", ["prefill_gqa32x8_d128_sq2048_sk16384_f16_ramp",
                                  "prefill_gqa32x8_d128_sq2048_sk16384_f16"])
def test_p_never_exceeds_e10(fa, name, launch):
    """The deferred rescale keeps a row's frame until a block's maximum score outgrows it by the
    10-point margin, so no P the softmax writes exceeds e^10 ("perf(rocm): defer SDPA
    accumulator rescale, stage Q once per block (#2306)", What changed).  fa_fwd_kv_stats
    reports for every row a bound that is at least its largest P (see fa.h): it must stay at or
    below e^10 (up to the rounding of the f32 exponent argument, < 2e-4 relative at these score
    magnitudes).  On the score ramp every row carries its frame through blocks whose maximum
    climbs ~2 per block, so the bound comes close to e^10 (above e^7 on every row); on N(0,1)
    data the first block sets the frame and P stays far below it."""
    w = fa_inputs.WORKLOADS[name]
    q, k, v = fa_inputs.make_qkv(w, device="cuda", generate_on_device=True)
    ws = None
    if launch == "cut_schedule":
        n = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, True)
        assert n > 0
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    pm = torch.full((w.B, w.Hq, w.Sq), -1.0, dtype=torch.float32, device="cuda")
    rc = torch.full((w.B, w.Hq, w.Sq), -1, dtype=torch.int32, device="cuda")
    o = fa.fa_fwd_kv(q, k, v, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws,
                     rescale_count=rc, p_max=pm)
    plain = fa.fa_fwd_kv(q, k, v, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    assert torch.equal(o, plain), "reporting the statistic changed the result"
    p = pm.cpu().numpy()
    assert np.isfinite(p).all() and p.min() >= 1.0 - 1e-6, p.min()
    assert p.max() <= E10 * (1 + 2e-4), p.max()
    if w.ramp:
        assert p.min() > np.exp(7.0), p.min()
        assert (rc.cpu().numpy() >= 2).all()
    else:
        assert p.max() < np.exp(8.0), p.max()
