"""Host-side checks of the C ABI that need no GPU: the library builds and loads, exports every
function include/fa.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import quantized_kv_cache_sm_gb300 as fa
from quantized_kv_cache_sm_gb300 import build as fa_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fa.h")


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(fa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", fa_build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(fa_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    assert fa.fa_status_string(0) == "FA_OK"
    assert fa.fa_status_string(4) == "FA_ERR_TIMEOUT"
    assert fa.fa_version() == 107


def test_q4_0_sizes(lib):
    # [B, H, S, D] = [1, 8, 16384, 128]: 8 MiB of nibbles, scale plane right after (aligned)
    assert fa.fa_q4_0_scale_offset(1, 8, 16384, 128) == 8 * 16384 * 64
    assert fa.fa_q4_0_bytes(1, 8, 16384, 128) == 8 * 16384 * 64 + 8 * 16384 * 4 * 2
    # 4.5 bits per element: the "about 75% smaller" cache of the q4_0 page is 71.9% smaller
    assert fa.fa_q4_0_bytes(4, 8, 65536, 128) == 4 * 8 * 65536 * 72  # K or V: 72 B per row
    # the scale plane starts at a 256-byte boundary
    off = fa.fa_q4_0_scale_offset(1, 1, 3, 32)
    assert off == 256 and fa.fa_q4_0_bytes(1, 1, 3, 32) == 256 + 3 * 2
    assert fa.fa_q4_0_bytes(1, 1, 1, 48) == 0  # D must be a multiple of 32


def test_prefill_workspace_without_a_device(lib):
    # the prefill schedule is planned for the current device's SM count; with no device the plan
    # runs one work unit per CTA, which needs no scratch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert fa.fa_workspace_bytes(1, 32, 8, 2048, 16384, 128, 14336, 1) == 0
    assert fa.fa_workspace_bytes(1, 32, 7, 2, 16, 128, 0, 1) == 0  # invalid: Hq % Hkv


def test_decode_workspace_layout_without_a_device(lib):
    # with no device the decode plan has no SMs to fill and uses one split per (batch, kv head):
    # the scratch is the arrival flags [B, Hkv, 1] u32 padded to 256 bytes, then the partials
    # [B, Hq, 1, D + 4] f32 (m, l, two pads, O)
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    for B, Hq, Hkv, Sk, D in [(4, 32, 8, 65536, 128), (1, 8, 8, 1, 64), (3, 12, 4, 999, 128)]:
        flags = -(-(B * Hkv * 4) // 256) * 256
        want = flags + B * Hq * (D + 4) * 4
        assert fa.fa_workspace_bytes(B, Hq, Hkv, 1, Sk, D, Sk - 1, 1) == want


P = 1 << 20  # a 16-byte aligned fake device address; never dereferenced by these calls


@pytest.mark.parametrize("args,expect", [
    # q, k, v, o, B, Hq, Hkv, Sq, Sk, D, off, causal, scale, dtype, kv
    ((0, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),   # null q
    ((P + 2, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),  # misaligned
    ((P, P, P, P, 0, 8, 8, 4, 4, 64, 0, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),   # B = 0
    ((P, P, P, P, 1, 8, 3, 4, 4, 64, 0, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),   # Hq % Hkv
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, 1, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),   # off+Sq > Sk
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, -1, 1, 0.125, 0, 0), fa.FA_ERR_INVALID_ARG),  # off < 0
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, 0.0, 0, 0), fa.FA_ERR_INVALID_ARG),     # scale 0
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, float("nan"), 0, 0), fa.FA_ERR_INVALID_ARG),
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, 0.125, 2, 0), fa.FA_ERR_INVALID_ARG),   # dtype
    ((P, P, P, P, 1, 8, 8, 4, 4, 64, 0, 1, 0.125, 0, 5), fa.FA_ERR_INVALID_ARG),   # kv format
    ((P, P, P, P, 1, 8, 8, 4, 4, 96, 0, 1, 0.125, 0, 0), fa.FA_ERR_UNSUPPORTED),   # D = 96
    ((P, P, P, P, 1, 16, 1, 1, 4, 64, 3, 1, 0.125, 0, 0), fa.FA_ERR_UNSUPPORTED),  # decode G > 8
])
def test_bad_arguments_rejected_on_host(lib, args, expect):
    assert lib.fa_fwd(*args, None) == expect
    assert lib.fa_fwd_ex(*args, None, 0, None, None) == expect


def test_decode_without_workspace_rejected(lib):
    # Sq == 1 needs scratch; fa_fwd_ex with none is an argument error (checked before launch)
    need = lib.fa_workspace_bytes(1, 8, 2, 1, 4096, 128, 4095, 1)
    if need == 0:
        pytest.skip("no device to size the split")
    st = lib.fa_fwd_ex(P, P, P, P, 1, 8, 2, 1, 4096, 128, 4095, 1, 0.088, 0, 0, None, 0, None,
                       None)
    assert st == fa.FA_ERR_INVALID_ARG


def test_quantize_bad_arguments(lib):
    assert lib.fa_quantize_q4_0(P, P, 1, 1, 1, 48, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_q4_0(0, P, 1, 1, 1, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_q4_0(P, P + 8, 1, 1, 1, 64, 0, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_quantize_q4_0(P, P, 1, 1, 1, 64, 7, None) == fa.FA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        fa.load_from(str(tmp_path / "missing.so"))


@pytest.mark.parametrize("args,expect", [
    # q, k, v, o, B, Hq, Hkv, Sq, Sk, cap, D, off, causal, scale, dtype, kf, vf
    # kv_capacity < Sk
    ((P, P, P, P, 1, 8, 2, 4, 64, 32, 64, 60, 1, 0.125, 0, 0, 1), fa.FA_ERR_INVALID_ARG),
    ((P, P, P, P, 1, 8, 2, 4, 64, 64, 64, 60, 1, 0.125, 0, 0, 7), fa.FA_ERR_INVALID_ARG),  # v fmt
    ((P, P, P, P, 1, 8, 2, 4, 64, 64, 64, 60, 1, 0.125, 0, 3, 1), fa.FA_ERR_INVALID_ARG),  # k fmt
    ((P, P, P, P, 1, 8, 2, 4, 64, 64, 96, 60, 1, 0.125, 0, 1, 0), fa.FA_ERR_UNSUPPORTED),  # D
])
def test_fwd_kv_bad_arguments_rejected_on_host(lib, args, expect):
    assert lib.fa_fwd_kv(*args, None, 0, None, None) == expect


@pytest.mark.parametrize("args", [
    # k_new, v_new, k_cache, v_cache, B, H, S_new, capacity, pos0, D, dtype
    (P, P, P, P, 1, 2, 16, 64, 49, 128, 0),   # pos0 + S_new > capacity
    (P, P, P, P, 1, 2, 16, 64, -1, 128, 0),   # pos0 < 0
    (P, P, P, P, 1, 2, 16, 64, 0, 48, 0),     # D % 32
    (P, 0, P, P, 1, 2, 16, 64, 0, 128, 0),    # v_new without v_cache
    (P, P, P, P, 1, 2, 16, 64, 0, 128, 2),    # dtype
])
def test_append_bad_arguments_rejected_on_host(lib, args):
    assert lib.fa_append_q4_0(*args, None) == fa.FA_ERR_INVALID_ARG


def test_paged_decode_host_checks(lib):
    T = P + 256  # a 4-byte aligned fake table / length pointer
    base = [P, P, P, P, T, T, 2, 8, 2, 128, 16, 128, 8, 0.088, 0, 1, 1, P, 1 << 30, None]
    # every case below is rejected by the host checks, before any tensor map or launch
    bad_page = list(base)
    bad_page[11] = 96  # page_size not a multiple of the 128-key q4_0 tile
    assert lib.fa_decode_paged(*bad_page) in (fa.FA_ERR_UNSUPPORTED,)
    no_table = list(base)
    no_table[4] = None
    assert lib.fa_decode_paged(*no_table) == fa.FA_ERR_INVALID_ARG
    big_group = list(base)
    big_group[7], big_group[8] = 32, 2  # 16 query heads per kv head
    assert lib.fa_decode_paged(*big_group) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_decode_paged_workspace_bytes(2, 8, 3, 128, 128, 8) == 0  # Hq % Hkv


def test_library_needs_no_blas(lib):
    """Every contraction of the library (the fused kernels and the explicit path's two GEMMs)
    is its own tcgen05 code: the shared library neither links nor calls cuBLAS."""
    needed = subprocess.run(["readelf", "-d", fa_build.LIB_PATH], capture_output=True, text=True,
                            check=True).stdout
    assert "cublas" not in needed.lower()
    undefined = subprocess.run(["nm", "-D", "--undefined-only", fa_build.LIB_PATH],
                               capture_output=True, text=True, check=True).stdout
    assert "cublas" not in undefined.lower()
