"""Device-side failure detection without a fault: a kernel whose barrier never completes gives
up after a short limit, records FA_ERR_TIMEOUT, and the context stays usable."""
import pytest
import torch

import fa_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(fa):
    assert fa.fa_get_status() == fa.FA_OK
    fa.fa_debug_wait_timeout(20_000_000)  # 20 ms
    assert fa.fa_get_status() == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_status() == fa.FA_OK  # the error word is cleared once reported
    q, k, v = fa_inputs.make_tensors(1, 4, 2, 130, 300, 128, "f16", seed=2, device="cuda")
    o = fa.fa_fwd(q, k, v)
    assert fa.fa_get_status() == fa.FA_OK
    assert torch.isfinite(o).all()


def test_invalid_arguments_raise(fa):
    q, k, v = fa_inputs.make_tensors(1, 4, 2, 8, 16, 128, "f16", seed=2, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q, k, v, q_pos_offset=9)  # 9 + 8 > 16
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    q96 = torch.zeros(1, 4, 8, 96, dtype=torch.float16, device="cuda")
    k96 = torch.zeros(1, 2, 16, 96, dtype=torch.float16, device="cuda")
    with pytest.raises(fa.FaError) as e:
        fa.fa_fwd(q96, k96, k96)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
