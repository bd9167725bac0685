"""The Python binding refuses, before any call into the library, tensors the kernels cannot use:
host (CPU) tensors, since the kernels take raw device pointers on the current device, and q4_0
tensors whose buffer is smaller than their shape needs.  Runs without a device."""
import pytest
import torch

import quantized_kv_cache_sm_gb300 as fa


@pytest.fixture(autouse=True)
def _library(built):
    return built


def host_qkv(Sq=4, Sk=8, D=64):
    q = torch.zeros(1, 2, Sq, D, dtype=torch.float16)
    k = torch.zeros(1, 2, Sk, D, dtype=torch.float16)
    return q, k, k.clone()


def test_host_tensors_refused_by_attention_entries():
    q, k, v = host_qkv()
    for call in (lambda: fa.fa_fwd(q, k, v),
                 lambda: fa.fa_fwd_ex(q, k, v),
                 lambda: fa.fa_fwd_kv(q, k, v),
                 lambda: fa.fa_fwd_explicit(q, k, v),
                 lambda: fa.fa_fwd_decode_noalloc(q[:, :, :1].contiguous(), k, v)):
        with pytest.raises(ValueError, match="CUDA tensors"):
            call()


def test_host_tensors_refused_by_cache_entries():
    x = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.fa_quantize_q4_0(x)
    cache = fa.q4_0_cache(1, 2, 16, 64, device="cpu")
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.fa_append_q4_0(x, cache, 0)


def test_host_tensors_refused_by_paged_decode():
    q = torch.zeros(2, 8, 1, 128, dtype=torch.float16)
    pool = torch.zeros(4, 2, 128, 128, dtype=torch.float16)
    table = torch.zeros(2, 2, dtype=torch.int32)
    lens = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.fa_decode_paged(q, pool, pool, table, lens)


def test_short_q4_0_buffer_refused():
    need = fa.fa_q4_0_bytes(1, 2, 16, 64)
    short = fa.Q4Tensor(torch.zeros(need - 1, dtype=torch.uint8), 1, 2, 16, 64)
    q = torch.zeros(1, 4, 4, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="needs"):
        fa.fa_fwd_kv(q, short, short)
    wrong_type = fa.Q4Tensor(torch.zeros(need, dtype=torch.int32), 1, 2, 16, 64)
    with pytest.raises(ValueError, match="uint8"):
        fa.fa_fwd(q, wrong_type, wrong_type)
    x = torch.zeros(1, 2, 16, 64, dtype=torch.float16)
    with pytest.raises(ValueError, match="needs"):
        fa.fa_quantize_q4_0(x, out=short)
    with pytest.raises(ValueError, match="shape of x"):
        fa.fa_quantize_q4_0(x[:, :, :8].contiguous(), out=short)
