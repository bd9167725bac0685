"""The prefill's equal-cuts schedule (more work units than SMs: the units' key-block steps cut
evenly over one CTA per SM, units cut between CTAs merged by their last piece) against the f64
oracle on sampled rows, against the one-unit-per-CTA launch, with a stale workspace, and replayed
from a CUDA graph.  The schedule runs when the caller passes fa_workspace_bytes() of scratch;
without scratch the same call runs one unit per CTA."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, sample_rows

pytestmark = pytest.mark.gpu

CUT = ["prefill_gqa32x8_d128_sq2048_sk16384_f16", "prefill_gqa32x8_d128_sq2048_sk16384_bf16"]


def workspace_for(fa, w, fill=None):
    n = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, True)
    units = w.B * w.Hq * ((w.Sq + 255) // 256)  # pairs of 128-row query tiles
    if torch.cuda.get_device_properties(0).multi_processor_count < units:
        assert n > 0, f"no cut schedule planned for {units} work units on this device"
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    if fill is not None:
        ws.fill_(fill)
    return ws


@pytest.mark.parametrize("name", CUT)
def test_cut_schedule_against_oracle_and_whole_units(fa, name):
    w = fa_inputs.WORKLOADS[name]
    q, k, v = fa_inputs.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = workspace_for(fa, w)
    rc_cut = torch.full((w.B, w.Hq, w.Sq), -1, dtype=torch.int32, device="cuda")
    rc_whole = torch.full_like(rc_cut, -1)
    o_cut = fa.fa_fwd_ex(qd, kd, vd, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws,
                         rescale_count=rc_cut)
    o_whole = fa.fa_fwd_ex(qd, kd, vd, causal=True, q_pos_offset=w.q_pos_offset,
                           rescale_count=rc_whole)
    assert fa.fa_get_status() == fa.FA_OK
    rows = sample_rows(w.B, w.Hq, w.Sq, per_head=14, seed=7)
    want = oracle.attention(np64(q), np64(k), np64(v), causal=True, q_pos_offset=w.q_pos_offset,
                            scale=w.scale, rows=rows)
    check_close(np64(o_cut).reshape(-1, w.D)[rows], want, w.dtype, f"{name} cut schedule")
    # every element of the two launches: the same sums in a different order, rounded once
    diff = (o_cut.float() - o_whole.float()).abs().max().item()
    assert diff <= (4e-3 if w.dtype == "f16" else 3e-2), diff
    # frame moves: a row cut between CTAs counts its first frame once, as the whole launch does
    cut = rc_cut.cpu().numpy()
    whole = rc_whole.cpu().numpy()
    assert cut.min() >= 1 and whole.min() >= 1
    assert np.abs(cut - whole).max() <= 2


def test_cut_schedule_score_ramp(fa):
    """Rows whose frame moves every fifth block, cut between CTAs: the merge weighs each piece's
    frame, and the output still matches the oracle."""
    w = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk16384_f16_ramp"]
    q, k, v = fa_inputs.make_qkv(w)
    ws = workspace_for(fa, w)
    rc = torch.full((w.B, w.Hq, w.Sq), -1, dtype=torch.int32, device="cuda")
    o = fa.fa_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True, q_pos_offset=w.q_pos_offset,
                     workspace=ws, rescale_count=rc)
    assert fa.fa_get_status() == fa.FA_OK
    rows = sample_rows(w.B, w.Hq, w.Sq, per_head=10, seed=2)
    want = oracle.attention(np64(q), np64(k), np64(v), causal=True, q_pos_offset=w.q_pos_offset,
                            scale=w.scale, rows=rows)
    check_close(np64(o).reshape(-1, w.D)[rows], want, w.dtype, "ramp, cut schedule")
    nblocks = (w.q_pos_offset + np.arange(w.Sq)) // 128 + 1
    ratio = rc.cpu().numpy().reshape(-1, w.Sq) / (1 + (nblocks - 1) / 5.0)[None, :]
    assert 0.7 < ratio.mean() < 1.3, ratio.mean()


def test_cut_schedule_stale_workspace_and_graph_replay(fa):
    """The piece flags carry a tag drawn for every call and the merging CTA clears them, so a
    workspace left by anything else, and a graph replayed with one tag, give the eager result bit
    for bit (the cut and the merge order are fixed, so the result is deterministic)."""
    w = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk16384_f16"]
    q, k, v = fa_inputs.make_qkv(w, device="cuda", generate_on_device=True)
    fresh = workspace_for(fa, w, fill=0)
    want = fa.fa_fwd_ex(q, k, v, causal=True, q_pos_offset=w.q_pos_offset, workspace=fresh)
    g = torch.Generator(device="cuda").manual_seed(9)
    stale = [workspace_for(fa, w, fill=255), workspace_for(fa, w)]
    stale[1].copy_(torch.randint(0, 256, stale[1].shape, dtype=torch.uint8, device="cuda",
                                 generator=g))
    for ws in stale:
        for _ in range(2):
            got = fa.fa_fwd_ex(q, k, v, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
            torch.cuda.synchronize()
            assert torch.equal(got, want)
    qs = q.clone()
    os_ = torch.empty_like(q)
    ws = stale[0]
    fa.fa_fwd_ex(qs, k, v, os_, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_fwd_ex(qs, k, v, os_, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
    for seed in (1, 2, 3):
        qn = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(seed),
                         device="cuda").to(q.dtype)
        qs.copy_(qn)
        graph.replay()
        torch.cuda.synchronize()
        eager = fa.fa_fwd_ex(qn, k, v, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(os_, eager), seed
    assert fa.fa_get_status() == fa.FA_OK


@pytest.mark.parametrize("shape", [
    # B, Hq, Hkv, Sq, Sk, causal, dtype: 160 units (odd tile count: the last pair of every head
    # has no tile B), ragged Sq and Sk, two batches
    (2, 16, 4, 1152, 20000, True, "f16"),
    # non-causal, 192 units of 64 steps, last pair of every head without tile B
    (1, 64, 8, 640, 8192, False, "bf16"),
], ids=lambda c: "-".join(map(str, c)))
def test_cut_schedule_other_shapes(fa, shape):
    B, Hq, Hkv, Sq, Sk, causal, dtype = shape
    off = Sk - Sq if causal else 0
    n = fa.fa_workspace_bytes(B, Hq, Hkv, Sq, Sk, 128, off, causal)
    units = B * Hq * ((Sq + 255) // 256)
    if torch.cuda.get_device_properties(0).multi_processor_count < units:
        assert n > 0, "no cut schedule planned"
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, Sk, 128, dtype, seed=Sq + Sk)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")
    o_cut = fa.fa_fwd_ex(qd, kd, vd, causal=causal, q_pos_offset=off, workspace=ws)
    o_whole = fa.fa_fwd_ex(qd, kd, vd, causal=causal, q_pos_offset=off)
    assert fa.fa_get_status() == fa.FA_OK
    rows = sample_rows(B, Hq, Sq, per_head=8, seed=3)
    want = oracle.attention(np64(q), np64(k), np64(v), causal=causal, q_pos_offset=off,
                            scale=128 ** -0.5, rows=rows)
    check_close(np64(o_cut).reshape(-1, 128)[rows], want, dtype, f"{shape} cut schedule")
    diff = (o_cut.float() - o_whole.float()).abs().max().item()
    assert diff <= (4e-3 if dtype == "f16" else 3e-2), diff


@pytest.mark.parametrize("fmt", [("q4_0", "q4_0"), ("dense", "q4_0"), ("q4_0", "dense")],
                         ids=lambda f: f"{f[0]}K-{f[1]}V")
def test_cut_schedule_q4_0_caches(fa, fmt):
    """The cut schedule with q4_0 K and/or V: the dequant warps' tile stream runs on across
    segments; compared with the oracle (its own quantization, dequantized exactly) on sampled
    rows and with the one-unit-per-CTA launch."""
    from gpu_common import oracle_q4_planes
    w = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk16384_f16"]
    q, k, v = fa_inputs.make_qkv(w)

    def side(x, f):
        if f == "q4_0":
            nib, sc = oracle_q4_planes(x)
            return fa.fa_quantize_q4_0(x.cuda()), oracle.dequantize_q4_0(nib, sc)
        return x.cuda(), np64(x)

    kd, k64 = side(k, fmt[0])
    vd, v64 = side(v, fmt[1])
    ws = workspace_for(fa, w)
    qd = q.cuda()
    o_cut = fa.fa_fwd_kv(qd, kd, vd, causal=True, q_pos_offset=w.q_pos_offset, workspace=ws)
    o_whole = fa.fa_fwd_kv(qd, kd, vd, causal=True, q_pos_offset=w.q_pos_offset)
    assert fa.fa_get_status() == fa.FA_OK
    rows = sample_rows(w.B, w.Hq, w.Sq, per_head=8, seed=5)
    want = oracle.attention(np64(q), k64, v64, causal=True, q_pos_offset=w.q_pos_offset,
                            scale=w.scale, rows=rows)
    check_close(np64(o_cut).reshape(-1, w.D)[rows], want, w.dtype, f"{fmt} cut schedule",
                q4=True)
    diff = (o_cut.float() - o_whole.float()).abs().max().item()
    assert diff <= 4e-3, diff
