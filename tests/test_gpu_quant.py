"""GPU q4_0 quantizer against the oracle's scalar quantizer: bit-exact nibble and scale planes."""
import os

import numpy as np
import pytest
import torch

import fa_inputs
import oracle
from gpu_common import oracle_q4_planes, q4_planes_gpu

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _assert_bit_exact(fa, x):
    q4 = fa.fa_quantize_q4_0(x.cuda())
    torch.cuda.synchronize()
    assert fa.fa_get_status() == fa.FA_OK
    gn, gs = q4_planes_gpu(q4)
    on, os_ = oracle_q4_planes(x)
    np.testing.assert_array_equal(gn, on)
    np.testing.assert_array_equal(gs, os_)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("shape", [(1, 1, 1, 32), (2, 3, 37, 64), (1, 8, 300, 128), (3, 2, 5, 96)])
def test_quantize_random_bit_exact(fa, dtype, shape):
    g = torch.Generator().manual_seed(sum(shape))
    x = torch.randn(*shape, generator=g).to(dtype)
    _assert_bit_exact(fa, x)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_quantize_special_blocks_bit_exact(fa, dtype):
    rows = []
    rows.append(np.zeros(32))                                     # zero block: scale -0
    rows.append(np.arange(32) * 0.25 - 4.0)                       # hand-worked block
    t = np.zeros(32); t[3], t[5] = 2.0, -2.0; rows.append(t)      # tie on |x|: first wins
    rows.append(np.full(32, 1e-6))                                # scale underflows in fp16
    rows.append(np.linspace(-60000, 60000, 32))                   # near the fp16 range
    rows.append((np.arange(32) % 16 - 8) * 0.5)                   # already on a q4_0 grid
    rows.append(np.random.default_rng(1).standard_normal(32) * 1e3)
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(dtype).reshape(1, 1, len(rows), 32)
    _assert_bit_exact(fa, x)


def test_quantize_hand_block_matches_golden(fa):
    x = (torch.arange(32, dtype=torch.float32) * 0.25 - 4.0).half().reshape(1, 1, 1, 32)
    q4 = fa.fa_quantize_q4_0(x.cuda())
    gn, gs = q4_planes_gpu(q4)
    fields = {}
    for line in open(os.path.join(GOLDEN, "q4_0_hand_block.txt")):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            fields[k] = v
    assert int(gs.ravel()[0]) == int(fields["scale_bits"][0], 16)
    np.testing.assert_array_equal(gn.ravel(), [int(b, 16) for b in fields["bytes"]])


@pytest.mark.parametrize("name", ["prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16",
                                  "decode_q4_0_b4_gqa32x8_d128_sk65536_f16"])
def test_quantize_workload_caches_bit_exact(fa, name):
    w = fa_inputs.WORKLOADS[name]
    _, k, v = fa_inputs.make_qkv(w)
    _assert_bit_exact(fa, k)
    _assert_bit_exact(fa, v)
