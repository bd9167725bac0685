"""fa_fwd_decode_noalloc: decode for callers that must not allocate device memory on the call
path (runtimes that reserve all device memory up front and manage it themselves, or hosts that
forbid allocation while serving).  The entry point keeps its split-K scratch in a fixed array the
library holds on each GPU; its results must equal those of the allocating entry point.

Collected last on purpose (file name), and written to pass both alone in a fresh process and
after the rest of the suite (the scratch array then still holds earlier calls' partials)."""
import numpy as np
import pytest
import torch

import fa_inputs

pytestmark = pytest.mark.gpu

TOL = {"f16": 1e-2, "bf16": 2e-2}


def _inputs(fa, B, Hq, Hkv, Sk, D, dtype, kv, seed):
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, 1, Sk, D, dtype, seed=seed, device="cuda")
    if kv == "q4_0":
        k, v = fa.fa_quantize_q4_0(k), fa.fa_quantize_q4_0(v)
    return q, k, v


def _noalloc_via_c_abi(fa, q, k, v, o, Hkv, Sk, off, scale, dtype, kv):
    lib = fa.load()
    B, Hq, _, D = q.shape
    st = lib.fa_fwd_decode_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sk, D, off, 1, scale,
        fa.FA_BF16 if dtype == "bf16" else fa.FA_F16,
        fa.FA_KV_Q4_0 if kv == "q4_0" else fa.FA_KV_DENSE,
        torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.status_name(st)


def test_noalloc_decode_matches_allocating_entry_point_twice_in_a_row(fa):
    w = fa_inputs.WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"]
    cases = [
        # the q4_0 decode workload: 4 sequences, GQA 32/8, D=128, 65536 keys
        (w.B, w.Hq, w.Hkv, w.Sk, w.D, w.dtype, "q4_0", w.seed),
        # a second, different call right after it: dense bf16, ragged key count, D=64
        (2, 8, 2, 3001, 64, "bf16", "dense", 77),
    ]
    for (B, Hq, Hkv, Sk, D, dtype, kv, seed) in cases:
        q, k, v = _inputs(fa, B, Hq, Hkv, Sk, D, dtype, kv, seed)
        off, scale = Sk - 1, D ** -0.5
        ws = torch.empty(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, off, True),
                         dtype=torch.uint8, device="cuda")
        want = fa.fa_fwd_ex(q, k, v, causal=True, q_pos_offset=off, scale=scale, workspace=ws)
        got = torch.full_like(q, float("nan"))
        _noalloc_via_c_abi(fa, q, k, v, got, Hkv, Sk, off, scale, dtype, kv)
        assert fa.fa_get_status() == fa.FA_OK
        g = got.double().cpu().numpy()
        r = want.double().cpu().numpy()
        assert np.isfinite(g).all()
        err = float(np.abs(g - r).max())
        assert err <= TOL[dtype], f"{kv} {dtype}: max-abs difference {err}"


def test_noalloc_rejects_shapes_beyond_the_scratch_limit(fa):
    lib = fa.load()
    P = 1 << 20  # never dereferenced: the size check comes first
    # 64 sequences x 128 query heads of D=128 need more than the fixed area
    st = lib.fa_fwd_decode_noalloc(P, P, P, P, 64, 128, 128, 4096, 128, 4095, 1, 0.088, 0, 0,
                                   None)
    assert st == fa.FA_ERR_UNSUPPORTED
