"""The explicit (non-flash) path, fa_fwd_explicit, against the f64 oracle through the C ABI, and
against the fused path on the same inputs.  Tolerance: max-abs 1e-2 (f16) / 2e-2 (bf16)."""
import numpy as np
import pytest

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes, rel_bound

pytestmark = pytest.mark.gpu


def side(fa, x, fmt):
    if fmt == "q4_0":
        nib, sc = oracle_q4_planes(x)
        return fa.fa_quantize_q4_0(x.cuda()), oracle.dequantize_q4_0(nib, sc)
    return x.cuda(), np64(x)


CASES = [
    # B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, k_fmt, v_fmt
    (1, 4, 2, 200, 450, 128, True, 250, "f16", "dense", "dense"),
    (1, 4, 2, 200, 450, 128, True, 250, "f16", "q4_0", "q4_0"),
    (2, 4, 1, 130, 333, 64, True, 203, "bf16", "dense", "q4_0"),
    (1, 2, 2, 300, 257, 128, False, 0, "bf16", "q4_0", "dense"),
    (2, 8, 2, 1, 3000, 128, True, 2999, "f16", "q4_0", "q4_0"),  # one query per sequence
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_explicit_path_matches_oracle(fa, case):
    B, Hq, Hkv, Sq, Sk, D, causal, off, dtype, kf, vf = case
    q, k, v = fa_inputs.make_tensors(B, Hq, Hkv, Sq, Sk, D, dtype, seed=53)
    kd, k64 = side(fa, k, kf)
    vd, v64 = side(fa, v, vf)
    o = fa.fa_fwd_explicit(q.cuda(), kd, vd, causal=causal, q_pos_offset=off, scale=D ** -0.5)
    assert fa.fa_get_status() == fa.FA_OK
    want = oracle.attention(np64(q), k64, v64, causal=causal, q_pos_offset=off, scale=D ** -0.5)
    q4 = "q4_0" in (kf, vf)
    check_close(np64(o), want, dtype, f"explicit {case}", q4=q4)
    fused = fa.fa_fwd_kv(q.cuda(), kd, vd, causal=causal, q_pos_offset=off, scale=D ** -0.5)
    # two GPU results, each within the bound of the oracle: their difference within twice it
    ratio = np.abs(np64(o) - np64(fused)) / (2 * rel_bound(want, dtype, q4))
    assert ratio.max() <= 1.0, ("explicit vs fused", float(ratio.max()))
