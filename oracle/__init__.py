"""CPU oracle for the fused causal GQA attention forward and the q4_0 K/V cache.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this package; the product library never imports it.  The arithmetic lives in
``fa_oracle.c`` (plain f64 loops, scalar IEEE f32 quantizer); this module compiles it with gcc
and marshals numpy arrays through ctypes.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against facts that do not
come from the oracle itself (closed forms, invariants, a high-precision brute-force evaluator,
hand-worked q4_0 blocks, and numpy's binary16 conversion).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: the quantizer's multiply and add are separately rounded f32 operations.
CFLAGS = ["-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into liboracle.so next to it (only when stale or missing)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i = ctypes.c_int
            i64 = ctypes.c_int64
            lib.oracle_f32_to_f16_rn.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_f16_rn.restype = ctypes.c_uint16
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = ctypes.c_double
            lib.oracle_quantize_q4_0.argtypes = [p, i64, p, p]
            lib.oracle_quantize_q4_0.restype = None
            lib.oracle_dequantize_q4_0.argtypes = [p, p, i64, p]
            lib.oracle_dequantize_q4_0.restype = None
            common = [i, i, i, i, i, i, i, i, ctypes.c_double, p, i64, i]
            lib.oracle_attention_rows.argtypes = [p, p, p, p, p] + common
            lib.oracle_attention_rows.restype = i
            lib.oracle_attention_rows_q4_0.argtypes = [p, p, p, p, p, p, p] + common
            lib.oracle_attention_rows_q4_0.restype = i
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    return os.cpu_count() or 1


# --------------------------------------------------------------------------------------------
# binary16 helpers
# --------------------------------------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    """Round f32 values to binary16 (ties to even); returns the uint16 bit patterns."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_f16_rn(float(v)) for v in x], dtype=np.uint16)


def f16_bits_to_f64(h) -> np.ndarray:
    lib = _load()
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f64(int(v)) for v in h], dtype=np.float64)


# --------------------------------------------------------------------------------------------
# q4_0
# --------------------------------------------------------------------------------------------

def quantize_q4_0(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantize ``x[..., D]`` (D a multiple of 32) along its last axis.

    Returns ``(nib, scale)``: ``nib[..., D/2]`` uint8 (byte j of each 32-block holds element j in
    the low nibble and element j+16 in the high nibble) and ``scale[..., D/32]`` uint16 (fp16
    bits of d)."""
    lib = _load()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    D = x.shape[-1]
    if D % 32:
        raise ValueError("last dimension must be a multiple of 32")
    nblocks = x.size // 32
    nib = np.empty(x.shape[:-1] + (D // 2,), dtype=np.uint8)
    scale = np.empty(x.shape[:-1] + (D // 32,), dtype=np.uint16)
    lib.oracle_quantize_q4_0(_ptr(x), nblocks, _ptr(nib), _ptr(scale))
    return nib, scale


def dequantize_q4_0(nib: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """Exact f64 values (q - 8) * d of a q4_0 tensor given as (nib, scale) planes."""
    lib = _load()
    nib = np.ascontiguousarray(nib, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint16)
    D = nib.shape[-1] * 2
    out = np.empty(nib.shape[:-1] + (D,), dtype=np.float64)
    lib.oracle_dequantize_q4_0(_ptr(nib), _ptr(scale), scale.size, _ptr(out))
    return out


# --------------------------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------------------------

def _rows_arg(rows, B, Hq, Sq):
    if rows is None:
        return np.arange(B * Hq * Sq, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    if rows.size and (rows.min() < 0 or rows.max() >= B * Hq * Sq):
        raise ValueError("row index out of range")
    return rows


def attention(q, k, v, *, causal: bool, q_pos_offset: int = 0, scale: float,
              rows=None, return_probs: bool = False, threads: int | None = None):
    """f64 attention on dense inputs.

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Sk, D] (any real dtype; upcast exactly to f64).
    rows: optional flat indices (b*Hq + h)*Sq + i of the query rows to evaluate.
    Returns o[nrows, D] (or [B, Hq, Sq, D] when rows is None), plus the probability rows
    [nrows, Sk] when return_probs is set."""
    lib = _load()
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    k = np.ascontiguousarray(np.asarray(k, dtype=np.float64))
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    _check_shapes(q.shape, k.shape, v.shape, causal, q_pos_offset)
    idx = _rows_arg(rows, B, Hq, Sq)
    o = np.empty((idx.size, D), dtype=np.float64)
    prob = np.empty((idx.size, Sk), dtype=np.float64) if return_probs else None
    lib.oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(prob), B, Hq, Hkv, Sq,
                              Sk, D, int(q_pos_offset), int(bool(causal)), float(scale),
                              _ptr(idx), idx.size, threads or default_threads())
    if rows is None:
        o = o.reshape(B, Hq, Sq, D)
    return (o, prob) if return_probs else o


def attention_q4_0(q, k_planes, v_planes, *, causal: bool, q_pos_offset: int = 0,
                   scale: float, rows=None, threads: int | None = None):
    """f64 attention with K and V given as q4_0 (nib, scale) planes [B, Hkv, Sk, D/2|D/32];
    each element is dequantized exactly before use."""
    lib = _load()
    q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
    kn, ks = (np.ascontiguousarray(a) for a in k_planes)
    vn, vs = (np.ascontiguousarray(a) for a in v_planes)
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = kn.shape
    _check_shapes(q.shape, kn.shape[:-1] + (D,), vn.shape[:-1] + (D,), causal, q_pos_offset)
    idx = _rows_arg(rows, B, Hq, Sq)
    o = np.empty((idx.size, D), dtype=np.float64)
    lib.oracle_attention_rows_q4_0(_ptr(q), _ptr(kn), _ptr(ks.view(np.uint16)), _ptr(vn),
                                   _ptr(vs.view(np.uint16)), _ptr(o), None, B, Hq, Hkv, Sq, Sk,
                                   D, int(q_pos_offset), int(bool(causal)), float(scale),
                                   _ptr(idx), idx.size, threads or default_threads())
    if rows is None:
        o = o.reshape(B, Hq, Sq, D)
    return o


def _check_shapes(qs, ks, vs, causal, q_pos_offset):
    B, Hq, Sq, D = qs
    if len(ks) != 4 or ks[0] != B or ks[3] != D or tuple(vs) != tuple(ks):
        raise ValueError("k/v must be [B, Hkv, Sk, D] matching q")
    Hkv, Sk = ks[1], ks[2]
    if Hkv <= 0 or Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if causal and (q_pos_offset < 0 or q_pos_offset + Sq > Sk):
        raise ValueError("causal rows need 0 <= q_pos_offset and q_pos_offset + Sq <= Sk")
