"""Split-K decode (Sq == 1) against the f64 oracle, through the C ABI: every output element."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes

pytestmark = pytest.mark.gpu


def run_decode(fa, B, Hq, Hkv, Sk, D, causal, off, dtype, kv, seed, use_ws=True):
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 1, Sk, D, dtype, seed=seed)
    scale = D ** -0.5
    qd = q.cuda()
    ws = None
    if use_ws:
        nbytes = fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, off, causal)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    if kv == "q4_0":
        kd, vd = fa.fa_quantize_q4_0(k.cuda()), fa.fa_quantize_q4_0(v.cuda())
    else:
        kd, vd = k.cuda(), v.cuda()
    if use_ws:
        o = fa.fa_fwd_ex(qd, kd, vd, causal=causal, q_pos_offset=off, scale=scale, workspace=ws)
    else:
        o = fa.fa_fwd(qd, kd, vd, causal=causal, q_pos_offset=off, scale=scale)
    assert fa.fa_get_status() == fa.FA_OK
    if kv == "q4_0":
        want = oracle.attention_q4_0(np64(q), oracle_q4_planes(k), oracle_q4_planes(v),
                                     causal=causal, q_pos_offset=off, scale=scale)
    else:
        want = oracle.attention(np64(q), np64(k), np64(v), causal=causal, q_pos_offset=off,
                                scale=scale)
    return check_close(np64(o), want, dtype, f"decode B{B} H{Hq}/{Hkv} Sk{Sk} D{D} {dtype} {kv}",
                       q4=kv == "q4_0")


CASES = [
    # B, Hq, Hkv, Sk, D, causal, off, dtype, kv
    (1, 8, 2, 1, 128, True, 0, "f16", "q4_0"),          # a single key: O = V[0]
    (1, 8, 2, 100, 128, True, 99, "f16", "q4_0"),
    (2, 32, 8, 4097, 128, True, 4096, "f16", "q4_0"),
    (3, 4, 4, 3000, 64, True, 2999, "bf16", "q4_0"),
    (1, 16, 2, 9999, 128, True, 5000, "f16", "q4_0"),  # keys past the position are masked
    (2, 8, 1, 2048, 128, False, 0, "bf16", "q4_0"),
    (1, 6, 2, 777, 64, True, 776, "f16", "q4_0"),       # group of 3
    (1, 8, 2, 100, 128, True, 99, "f16", "dense"),
    (2, 32, 8, 4097, 128, True, 4096, "bf16", "dense"),
    (1, 4, 4, 3000, 64, True, 2999, "f16", "dense"),
    (1, 8, 1, 5000, 128, False, 0, "f16", "dense"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_decode_small(fa, case):
    run_decode(fa, *case, seed=11)


def test_decode_q4_0_b4_sk65536_full(fa):
    w = fa_inputs.WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"]
    run_decode(fa, w.B, w.Hq, w.Hkv, w.Sk, w.D, True, w.q_pos_offset, w.dtype, "q4_0", w.seed)


def test_decode_allocating_entry_point(fa):
    run_decode(fa, 2, 8, 2, 3000, 128, True, 2999, "f16", "q4_0", seed=12, use_ws=False)


def test_decode_ex_rejects_small_workspace(fa):
    q, k, v = fa_inputs.make_tensors(1, 8, 2, 1, 4096, 128, "f16", seed=1, device="cuda")
    need = fa.fa_workspace_bytes(1, 8, 2, 1, 4096, 128, 4095, True)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd_ex(q, k, v, workspace=ws)
    assert e.value.status == fa.FA_ERR_INVALID_ARG


def test_decode_workspace_contents_do_not_matter(fa):
    """The splits of each (batch, kv head) are merged by a CTA that finds all its siblings'
    arrival flags (kept in the workspace) set.  A workspace full of stale bytes (all ones,
    random bytes, or left behind by a call of another shape and cache format) must give the
    same result as a fresh one."""
    shapes = [(2, 32, 8, 4097, 128, True, 4096, "f16", "q4_0"),
              (1, 8, 2, 3001, 64, True, 3000, "bf16", "dense"),
              (3, 12, 3, 999, 128, False, 0, "f16", "q4_0")]
    need = max(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, off, c)
               for (B, Hq, Hkv, Sk, D, c, off, _, _) in shapes)
    g = torch.Generator(device="cuda").manual_seed(5)
    fills = [torch.full((need,), 255, dtype=torch.uint8, device="cuda"),
             torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda", generator=g)]
    for ws in fills:
        for (B, Hq, Hkv, Sk, D, causal, off, dtype, kv) in shapes:
            q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 1, Sk, D, dtype, seed=Sk, device="cuda")
            if kv == "q4_0":
                k, v = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
            fresh = torch.zeros(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, off, causal),
                                dtype=torch.uint8, device="cuda")
            want = fa.fa_fwd_ex(q, k, v, causal=causal, q_pos_offset=off, workspace=fresh)
            for _ in range(3):  # the same stale buffer, call after call
                got = fa.fa_fwd_ex(q, k, v, causal=causal, q_pos_offset=off, workspace=ws)
                torch.cuda.synchronize()
                assert torch.equal(got, want), (B, Hq, Hkv, Sk, D, dtype, kv)
    assert fa.fa_get_status() == fa.FA_OK


def test_decode_replayed_from_a_cuda_graph(fa):
    """A captured decode launch keeps one flag tag for every replay; the merging CTA clears the
    flags, so each replay merges all splits again.  New query rows copied in between
    replays must give the eager result bit for bit."""
    B, Hq, Hkv, Sk, D = 2, 16, 4, 20000, 128
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 1, Sk, D, "f16", seed=31, device="cuda")
    kq, vq = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    ws = torch.empty(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, Sk - 1, True),
                     dtype=torch.uint8, device="cuda")
    qs = torch.empty_like(q)
    os_ = torch.empty_like(q)
    qs.copy_(q)
    fa.fa_fwd_ex(qs, kq, vq, os_, causal=True, q_pos_offset=Sk - 1, workspace=ws)  # warm-up
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.fa_fwd_ex(qs, kq, vq, os_, causal=True, q_pos_offset=Sk - 1, workspace=ws)
    for seed in (1, 2, 3, 4):
        qn = torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(seed),
                         device="cuda").to(q.dtype)
        qs.copy_(qn)
        graph.replay()
        torch.cuda.synchronize()
        want = fa.fa_fwd_ex(qn, kq, vq, causal=True, q_pos_offset=Sk - 1, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(os_, want), seed
    assert fa.fa_get_status() == fa.FA_OK


@pytest.mark.parametrize("recipe", ["ramp", "q_times_8"])
def test_decode_large_magnitude_queries(fa, recipe):
    """The q4_0 decode feeds the K nibbles to the tensor core as offset values (1024 + q and
    1024 + 16 q in f16) and removes the offset by starting each block's sum at -(offset * sum
    of the block's Q elements), a cancellation in f32 that grows with |Q|.  Large query
    magnitudes: the score-ramp recipe at one query per sequence (Q[..., 0] = 8 and a key column
    rising 2.0 per 128 keys in scaled-score units), and N(0,1) queries multiplied by 8 (scores
    8x larger, a sharply peaked softmax).  Every output element against the oracle."""
    B, Hq, Hkv, D = 2, 32, 8, 128
    Sk = 16384 if recipe == "ramp" else 32768
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 1, Sk, D, "f16", seed=61,
                                     ramp=recipe == "ramp")
    if recipe == "q_times_8":
        q = (q.float() * 8.0).to(q.dtype)
    kd, vd = fa.fa_quantize_q4_0(k.cuda()), fa.fa_quantize_q4_0(v.cuda())
    ws = torch.empty(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, Sk - 1, True),
                     dtype=torch.uint8, device="cuda")
    o = fa.fa_fwd_ex(q.cuda(), kd, vd, causal=True, q_pos_offset=Sk - 1, scale=D ** -0.5,
                     workspace=ws)
    assert fa.fa_get_status() == fa.FA_OK
    want = oracle.attention_q4_0(np64(q), oracle_q4_planes(k), oracle_q4_planes(v), causal=True,
                                 q_pos_offset=Sk - 1, scale=D ** -0.5)
    check_close(np64(o), want, "f16", f"decode, large queries ({recipe})", q4=True)
