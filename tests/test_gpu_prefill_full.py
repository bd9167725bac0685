"""Every output row of the full-size chunked-prefill workloads against the f64 oracle, through
both prefill launches: one work unit per CTA (no scratch) and the cut schedule (the scratch of
fa_workspace_bytes, the launch bench.py times).  The oracle evaluates each workload once (all
65 536 rows at 16K keys take some seconds on a many-core host) and both launches are checked
against it with the absolute and relative bounds of gpu_common."""
import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import check_close, np64, oracle_q4_planes

pytestmark = pytest.mark.gpu

WORKLOADS = ["prefill_gqa32x8_d128_sq2048_sk8192_f16",
             "prefill_gqa32x8_d128_sq2048_sk8192_bf16",
             "prefill_gqa32x8_d128_sq2048_sk16384_f16",
             "prefill_gqa32x8_d128_sq2048_sk16384_bf16",
             "prefill_gqa32x8_d128_sq2048_sk16384_f16_ramp",
             "prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16"]


def inputs_and_oracle(name):
    w = fa_inputs.WORKLOADS[name]
    q, k, v = fa_inputs.make_qkv(w)
    if w.kv_format == "q4_0":
        # the oracle's own quantization, expanded exactly once (attention over the dequantized
        # planes equals its q4_0 entry, which expands every element at every use: a pinned
        # identity), so that all 65 536 rows take seconds
        k64 = oracle.dequantize_q4_0(*oracle_q4_planes(k))
        v64 = oracle.dequantize_q4_0(*oracle_q4_planes(v))
        want = oracle.attention(np64(q), k64, v64, causal=True, q_pos_offset=w.q_pos_offset,
                                scale=w.scale)
    else:
        want = oracle.attention(np64(q), np64(k), np64(v), causal=True,
                                q_pos_offset=w.q_pos_offset, scale=w.scale)
    return w, q, k, v, want


@pytest.mark.parametrize("name", WORKLOADS)
def test_every_row_against_oracle(fa, name):
    w, q, k, v, want = inputs_and_oracle(name)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if w.kv_format == "q4_0":
        kd, vd = fa.fa_quantize_q4_0(kd), fa.fa_quantize_q4_0(vd)
    q4 = w.kv_format == "q4_0"
    n = fa.fa_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.q_pos_offset, True)
    units = w.B * w.Hq * ((w.Sq + 255) // 256)
    if torch.cuda.get_device_properties(0).multi_processor_count < units and w.Sk >= 16384:
        assert n > 0, "no cut schedule planned for the 16K chunk"
    launches = {"whole units": None}
    if n > 0:  # the plan cuts this shape on this device
        launches["cut schedule"] = torch.empty(n, dtype=torch.uint8, device="cuda")
    for launch, ws in launches.items():
        o = fa.fa_fwd_ex(qd, kd, vd, causal=True, q_pos_offset=w.q_pos_offset, scale=w.scale,
                         workspace=ws)
        assert fa.fa_get_status() == fa.FA_OK
        got = np64(o)
        check_close(got, want, w.dtype, f"{name} {launch}", q4=q4)
