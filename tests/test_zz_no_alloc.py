"""fa_fwd_decode_noalloc: decode for callers that must not allocate device memory on the call
path (runtimes that reserve all device memory up front and manage it themselves, or hosts that
forbid allocation while serving).  The entry point keeps its split-K scratch in a fixed array the
library holds on each GPU; its results must equal those of the allocating entry point.

Both calls pick the same split plan, run the same kernel and merge the splits in the same
fixed order, so their outputs must agree bit for bit; a merge that read a stale or misplaced
partial from the shared array would show up as a small difference.  The test also watches the
device's default memory pool (the one the stream-ordered allocator uses) and the device's free
memory around the call, so that a fallback to an allocating path would be seen.

Collected last on purpose (file name), and written to pass both alone in a fresh process and
after the rest of the suite (the scratch array then still holds earlier calls' partials)."""
import ctypes

import numpy as np
import pytest
import torch

import fa_inputs

pytestmark = pytest.mark.gpu

# cudaMemPoolAttr values (driver_types.h)
_ATTR_RESERVED_HIGH = 0x6
_ATTR_USED_HIGH = 0x8


class _DefaultPool:
    """High-water marks of the current device's default memory pool, through the CUDA runtime
    (the pool is a property of the device, whichever runtime instance asks)."""

    def __init__(self):
        self.rt = None
        for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
            try:
                self.rt = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if self.rt is None:
            pytest.skip("CUDA runtime library not found by name")
        self.pool = ctypes.c_void_p()
        dev = torch.cuda.current_device()
        assert self.rt.cudaDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def _get(self, attr):
        v = ctypes.c_uint64()
        assert self.rt.cudaMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset(self):
        """Reset both high-water marks (to the current use)."""
        z = ctypes.c_uint64(0)
        for a in (_ATTR_RESERVED_HIGH, _ATTR_USED_HIGH):
            assert self.rt.cudaMemPoolSetAttribute(self.pool, a, ctypes.byref(z)) == 0

    def high(self):
        return self._get(_ATTR_USED_HIGH), self._get(_ATTR_RESERVED_HIGH)


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
    first = True
    for (B, Hq, Hkv, Sk, D, dtype, kv, seed) in cases:
        q, k, v = _inputs(fa, B, Hq, Hkv, Sk, D, dtype, kv, seed)
        off, scale = Sk - 1, D ** -0.5
        ws = torch.empty(fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, off, True),
                         dtype=torch.uint8, device="cuda")
        want = fa.fa_fwd_ex(q, k, v, causal=True, q_pos_offset=off, scale=scale, workspace=ws)
        got = torch.full_like(q, float("nan"))
        if first:
            # the first call on a device sets up the scratch address; with lazy module loading
            # that is also when the driver loads the module holding the array
            _noalloc_via_c_abi(fa, q, k, v, got, Hkv, Sk, off, scale, dtype, kv)
            first = False
        torch.cuda.synchronize()
        pool = _DefaultPool()
        pool.reset()
        base = pool.high()
        free_before = torch.cuda.mem_get_info()[0]
        _noalloc_via_c_abi(fa, q, k, v, got, Hkv, Sk, off, scale, dtype, kv)
        torch.cuda.synchronize()
        assert pool.high() == base, "the default memory pool was used during the call"
        assert torch.cuda.mem_get_info()[0] == free_before
        assert fa.fa_get_status() == fa.FA_OK
        assert np.isfinite(got.double().cpu().numpy()).all()
        assert torch.equal(got, want), f"{kv} {dtype}: outputs differ"


def test_pool_probe_sees_the_allocating_entry_point(fa):
    """The probe used above is not blind: fa_fwd takes its decode scratch from the default pool
    (cudaMallocAsync), and the pool's high-water mark shows it."""
    q, k, v = _inputs(fa, 2, 8, 2, 3000, 128, "f16", "q4_0", 5)
    torch.cuda.synchronize()
    pool = _DefaultPool()
    pool.reset()
    fa.fa_fwd(q, k, v, causal=True, q_pos_offset=2999)
    torch.cuda.synchronize()
    assert pool.high()[0] > 0


def test_noalloc_rejects_shapes_beyond_the_scratch_limit(fa):
    lib = fa.load()
    P = 1 << 20  # never dereferenced: the size check comes first
    # 64 sequences x 128 query heads of D=128 need more than the fixed area
    st = lib.fa_fwd_decode_noalloc(P, P, P, P, 64, 128, 128, 4096, 128, 4095, 1, 0.088, 0, 0,
                                   None)
    assert st == fa.FA_ERR_UNSUPPORTED
