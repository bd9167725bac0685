"""Python binding of libfa_gb300.so: the fused causal GQA flash-attention forward for sm_103a,
with an optional q4_0 K/V cache.

Argument marshalling only: each function here turns torch tensors into the pointers, sizes and
stream handle of the C entry point of the same name (declared in ``include/fa.h``) and raises
``FaError`` on a non-OK status.  Every step of the computation runs in the CUDA kernels; there is
no CPU path.  The library must have been built (``build.build()`` or ``__graft_entry__.build()``);
if it is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import dataclasses
import functools
import os
import threading

import torch

from . import build as _build

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_F16, FA_BF16 = 0, 1
FA_KV_DENSE, FA_KV_Q4_0 = 0, 1

EXPORTED = (
    "fa_fwd", "fa_fwd_ex", "fa_workspace_bytes", "fa_q4_0_bytes", "fa_q4_0_scale_offset",
    "fa_quantize_q4_0", "fa_get_status", "fa_status_string", "fa_debug_wait_timeout",
    "fa_version", "fa_fwd_decode_noalloc", "fa_fwd_kv", "fa_append_q4_0", "fa_decode_paged",
    "fa_decode_paged_workspace_bytes", "fa_fwd_explicit", "fa_explicit_workspace_bytes",
    "fa_prefill_schedule", "fa_decode_schedule", "fa_fwd_kv_stats",
    "fa_prefill_append_workspace_bytes", "fa_prefill_append_q4_0",
)

_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)}")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the CUDA library once per process (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_from(path or _build.LIB_PATH)
        return _lib


def load_from(p: str) -> ctypes.CDLL:
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it first (quantized_kv_cache_sm_gb300.build)")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fwd = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i]
    lib.fa_fwd.argtypes = fwd + [vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_ex.argtypes = fwd + [vp, sz, vp, vp]
    lib.fa_fwd_ex.restype = i
    lib.fa_workspace_bytes.argtypes = [i] * 8
    lib.fa_workspace_bytes.restype = sz
    lib.fa_q4_0_bytes.argtypes = [i] * 4
    lib.fa_q4_0_bytes.restype = sz
    lib.fa_q4_0_scale_offset.argtypes = [i] * 4
    lib.fa_q4_0_scale_offset.restype = sz
    lib.fa_quantize_q4_0.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.fa_quantize_q4_0.restype = i
    lib.fa_get_status.argtypes = [vp]
    lib.fa_get_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_debug_wait_timeout.argtypes = [ctypes.c_int64, vp]
    lib.fa_debug_wait_timeout.restype = i
    lib.fa_version.argtypes = []
    lib.fa_version.restype = i
    lib.fa_prefill_schedule.argtypes = [i] * 10 + [vp, vp, ctypes.c_int64]
    lib.fa_prefill_schedule.restype = ctypes.c_int64
    lib.fa_decode_schedule.argtypes = [vp] + [i] * 8 + [vp, ctypes.c_int64]
    lib.fa_decode_schedule.restype = ctypes.c_int64
    lib.fa_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_decode_noalloc.restype = i
    lib.fa_fwd_kv.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, i, i, vp, sz, vp,
                              vp]
    lib.fa_fwd_kv.restype = i
    lib.fa_fwd_kv_stats.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, i, i, vp, sz,
                                    vp, vp, vp]
    lib.fa_fwd_kv_stats.restype = i
    lib.fa_append_q4_0.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.fa_append_q4_0.restype = i
    lib.fa_prefill_append_workspace_bytes.argtypes = [i] * 7
    lib.fa_prefill_append_workspace_bytes.restype = sz
    lib.fa_prefill_append_q4_0.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp,
                                           sz, vp]
    lib.fa_prefill_append_q4_0.restype = i
    lib.fa_decode_paged_workspace_bytes.argtypes = [i] * 6
    lib.fa_decode_paged_workspace_bytes.restype = sz
    lib.fa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, i, vp,
                                    sz, vp]
    lib.fa_decode_paged.restype = i
    lib.fa_explicit_workspace_bytes.argtypes = [i] * 8
    lib.fa_explicit_workspace_bytes.restype = sz
    lib.fa_fwd_explicit.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, i, i, vp, sz,
                                    vp]
    lib.fa_fwd_explicit.restype = i
    return lib


def status_name(s: int) -> str:
    names = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
             4: "FA_ERR_TIMEOUT"}
    return names.get(int(s), f"status {int(s)}")


def _check(status: int, where: str):
    if status != FA_OK:
        raise FaError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return FA_F16
    if t == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t}: use float16 or bfloat16")


@dataclasses.dataclass
class Q4Tensor:
    """A q4_0 tensor of logical shape [B, H, S, D]: one uint8 device buffer holding the nibble
    plane [B, H, S, D/2] and, at a 256-byte aligned offset, the fp16 scale plane [B, H, S, D/32]."""
    buf: torch.Tensor
    B: int
    H: int
    S: int
    D: int

    @property
    def shape(self):
        return (self.B, self.H, self.S, self.D)

    def nibbles(self) -> torch.Tensor:
        n = self.B * self.H * self.S * self.D // 2
        return self.buf[:n].view(self.B, self.H, self.S, self.D // 2)

    def scales(self) -> torch.Tensor:
        off = fa_q4_0_scale_offset(self.B, self.H, self.S, self.D)
        n = self.B * self.H * self.S * (self.D // 32) * 2
        return self.buf[off:off + n].view(torch.float16).view(self.B, self.H, self.S, self.D // 32)

    def data_ptr(self) -> int:
        return self.buf.data_ptr()


def _check_q4(t: Q4Tensor, what: str):
    """A Q4Tensor's buffer must be one contiguous uint8 vector holding both planes."""
    if t.buf.dtype != torch.uint8 or t.buf.dim() != 1 or not t.buf.is_contiguous():
        raise ValueError(f"{what}: the q4_0 buffer must be a contiguous uint8 vector")
    need = fa_q4_0_bytes(t.B, t.H, t.S, t.D)
    if need == 0 or t.buf.numel() < need:
        raise ValueError(f"{what}: a q4_0 tensor of shape {t.shape} needs {need} bytes, "
                         f"its buffer holds {t.buf.numel()}")


def _on_device(*tensors):
    """The kernels run on the current CUDA device and take raw pointers: every tensor argument
    (None skipped) must live there."""
    cur = None
    for t in tensors:
        if t is None:
            continue
        if isinstance(t, Q4Tensor):
            t = t.buf
        idx = t.get_device()  # -1 for host memory
        if idx < 0:
            raise ValueError(f"tensor arguments must be CUDA tensors (one is on {t.device})")
        if cur is None:
            cur = torch.cuda.current_device()
        if idx != cur:
            raise ValueError(f"a tensor is on cuda:{idx} but the current device is cuda:{cur}")


def _kv_args(k, v):
    if isinstance(k, Q4Tensor) != isinstance(v, Q4Tensor):
        raise TypeError("k and v must both be dense tensors or both be Q4Tensor")
    if isinstance(k, Q4Tensor):
        if k.shape != v.shape:
            raise ValueError("k and v shapes differ")
        _check_q4(k, "k")
        _check_q4(v, "v")
        return FA_KV_Q4_0, k.shape
    if k.shape != v.shape or k.dim() != 4:
        raise ValueError("k and v must both be [B, Hkv, Sk, D]")
    if not (k.is_contiguous() and v.is_contiguous()):
        raise ValueError("k and v must be contiguous")
    return FA_KV_DENSE, tuple(k.shape)


def _fwd_args(q, k, v, o, causal, q_pos_offset, scale):
    if q.dim() != 4 or not q.is_contiguous() or not o.is_contiguous() or o.shape != q.shape:
        raise ValueError("q and o must be contiguous [B, Hq, Sq, D] tensors of the same shape")
    if o.dtype != q.dtype:
        raise TypeError("o must have the dtype of q")
    kv_format, (Bk, Hkv, Sk, Dk) = _kv_args(k, v)
    B, Hq, Sq, D = q.shape
    if Bk != B or Dk != D:
        raise ValueError("k/v batch or head dim does not match q")
    if kv_format == FA_KV_DENSE and k.dtype != q.dtype:
        raise TypeError("dense k/v must have the dtype of q")
    if scale is None:
        scale = D ** -0.5
    if q_pos_offset is None:
        q_pos_offset = Sk - Sq
    _on_device(q, k, v, o)
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sq, Sk, D,
            int(q_pos_offset), int(bool(causal)), float(scale), _dtype_code(q.dtype), kv_format)


def fa_fwd(q, k, v, o=None, *, causal: bool = True, q_pos_offset: int | None = None,
           scale: float | None = None, stream=None) -> torch.Tensor:
    """O = softmax(scale Q K^T + causal mask) V.  q [B,Hq,Sq,D]; k, v [B,Hkv,Sk,D] dense (dtype of
    q) or Q4Tensor.  q_pos_offset defaults to Sk - Sq (bottom-right aligned chunk), scale to
    1/sqrt(D).  Returns o (allocated when not given)."""
    if o is None:
        o = torch.empty_like(q)
    lib = load()
    args = _fwd_args(q, k, v, o, causal, q_pos_offset, scale)
    _check(lib.fa_fwd(*args, _stream(stream)), "fa_fwd")
    return o


def fa_fwd_ex(q, k, v, o=None, *, causal: bool = True, q_pos_offset: int | None = None,
              scale: float | None = None, workspace: torch.Tensor | None = None,
              rescale_count: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """fa_fwd with caller-provided scratch (uint8 device tensor of at least fa_workspace_bytes)
    and an optional int32 [B, Hq, Sq] rescale counter."""
    if o is None:
        o = torch.empty_like(q)
    lib = load()
    args = _fwd_args(q, k, v, o, causal, q_pos_offset, scale)
    _on_device(workspace, rescale_count)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc_ptr = None
    if rescale_count is not None:
        rows = q.shape[0] * q.shape[1] * q.shape[2]
        if rescale_count.dtype != torch.int32 or rescale_count.numel() != rows:
            raise ValueError("rescale_count must be int32 [B, Hq, Sq]")
        rc_ptr = rescale_count.data_ptr()
    _check(lib.fa_fwd_ex(*args, ws_ptr, ws_bytes, rc_ptr, _stream(stream)), "fa_fwd_ex")
    return o


def fa_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal) -> int:
    return int(load().fa_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, int(bool(causal))))


@functools.lru_cache(maxsize=256)
def _q4_0_bytes(B: int, H: int, S: int, D: int) -> int:
    return int(load().fa_q4_0_bytes(B, H, S, D))


def fa_q4_0_bytes(B, H, S, D) -> int:
    # a pure function of the shape, asked on every call that takes a q4_0 tensor: cached
    return _q4_0_bytes(int(B), int(H), int(S), int(D))


def fa_q4_0_scale_offset(B, H, S, D) -> int:
    return int(load().fa_q4_0_scale_offset(B, H, S, D))


def fa_quantize_q4_0(x: torch.Tensor, out: Q4Tensor | None = None, *, stream=None) -> Q4Tensor:
    """Build the q4_0 tensor of x [B, H, S, D] (float16/bfloat16, D % 32 == 0)."""
    if x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [B, H, S, D] tensor")
    B, H, S, D = x.shape
    lib = load()
    if out is not None:
        if out.shape != (B, H, S, D):
            raise ValueError("out must be a q4_0 tensor of the shape of x")
        _check_q4(out, "out")
    _on_device(x, out)
    if out is None:
        nbytes = fa_q4_0_bytes(B, H, S, D)
        if nbytes == 0:
            raise ValueError("D must be a positive multiple of 32")
        out = Q4Tensor(torch.empty(nbytes, dtype=torch.uint8, device=x.device), B, H, S, D)
    _check(lib.fa_quantize_q4_0(x.data_ptr(), out.data_ptr(), B, H, S, D, _dtype_code(x.dtype),
                                _stream(stream)), "fa_quantize_q4_0")
    return out


def fa_get_status(stream=None) -> int:
    return int(load().fa_get_status(_stream(stream)))


def fa_status_string(s: int) -> str:
    return load().fa_status_string(int(s)).decode()


def fa_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(load().fa_debug_wait_timeout(int(limit_ns), _stream(stream)), "fa_debug_wait_timeout")


def fa_version() -> int:
    return int(load().fa_version())


SCHEDULE_COLUMNS = ("cta", "b", "h", "q0A", "nbA", "nbB", "nbmax", "j0", "j1", "unit_start",
                    "slot")


def fa_prefill_schedule(B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal, num_sms, *,
                        force_cut: bool = False):
    """The prefill's work schedule for a call of this shape on `num_sms` SMs, as the kernel
    computes it (host only).  Returns (plan, rows): plan = dict(cut, ctas, W, units,
    workspace_bytes); rows = int64 array [segments, 11] with columns SCHEDULE_COLUMNS, empty when
    the launch runs one unit per CTA.  Raises FaError(FA_ERR_INVALID_ARG) for invalid arguments
    and FaError(FA_ERR_UNSUPPORTED) when a CTA's range does not fit the segment table."""
    import numpy as np
    lib = load()
    plan = (ctypes.c_int64 * 5)()
    args = [int(B), int(Hq), int(Hkv), int(Sq), int(Sk), int(D), int(q_pos_offset),
            int(bool(causal)), int(num_sms), int(bool(force_cut))]
    n = lib.fa_prefill_schedule(*args, plan, None, 0)
    if n == -2:
        raise FaError(FA_ERR_INVALID_ARG, "fa_prefill_schedule")
    if n == -1:
        raise FaError(FA_ERR_UNSUPPORTED, "fa_prefill_schedule")
    rows = np.zeros((n, len(SCHEDULE_COLUMNS)), dtype=np.int64)
    if n > 0:
        got = lib.fa_prefill_schedule(*args, plan, rows.ctypes.data, n)
        assert got == n
    info = dict(zip(("cut", "ctas", "W", "units", "workspace_bytes"), (int(x) for x in plan)))
    info["cut"] = bool(info["cut"])
    return info, rows


def fa_decode_schedule(B, Hkv, num_sms, *, Sk: int | None = None, seq_lens=None,
                       page_size: int = 0, pages_per_seq: int = 0, k_format: str = "q4_0",
                       v_format: str = "q4_0"):
    """The decode kernels' work split (host only): an int32 array [rows, 5] of (sequence, split,
    splits of that sequence, first key, end key).  Uniform batch: give Sk (one row per sequence
    and split).  Paged batch: give seq_lens (B lengths), page_size and pages_per_seq (one row per
    CTA of a kv head; sequence -1 for a CTA with no work).  Raises FaError(FA_ERR_INVALID_ARG)
    for invalid arguments."""
    import numpy as np
    lib = load()
    fmt = {"dense": FA_KV_DENSE, "q4_0": FA_KV_Q4_0}
    lens = None
    if seq_lens is not None:
        lens = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        if lens.shape != (int(B),):
            raise ValueError("seq_lens must hold B lengths")
    args = [lens.ctypes.data if lens is not None else None, int(B), int(Hkv),
            int(Sk or 0), int(page_size), int(pages_per_seq), fmt[k_format], fmt[v_format],
            int(num_sms)]
    n = lib.fa_decode_schedule(*args, None, 0)
    if n < 0:
        raise FaError(FA_ERR_INVALID_ARG, "fa_decode_schedule")
    rows = np.zeros((n, 5), dtype=np.int32)
    if n > 0:
        assert lib.fa_decode_schedule(*args, rows.ctypes.data, n) == n
    return rows


def fa_fwd_decode_noalloc(q, k, v, o=None, *, causal: bool = True,
                          q_pos_offset: int | None = None, scale: float | None = None,
                          stream=None) -> torch.Tensor:
    """Decode (Sq = 1) without any device allocation by the library: the split-K scratch comes
    from a fixed area the library keeps on each GPU (FA_NOALLOC_SCRATCH_BYTES), for callers that
    must not allocate on the call path.  Calls that overlap on the GPU race on that area."""
    if o is None:
        o = torch.empty_like(q)
    lib = load()
    a = _fwd_args(q, k, v, o, causal, q_pos_offset, scale)
    if a[7] != 1:
        raise ValueError("fa_fwd_decode_noalloc takes one query token per sequence (Sq == 1)")
    _check(lib.fa_fwd_decode_noalloc(*a[:7], *a[8:], _stream(stream)), "fa_fwd_decode_noalloc")
    return o


def _side(t):
    """(format code, [B, H, S, D]) of one K or V operand: a dense tensor or a Q4Tensor."""
    if isinstance(t, Q4Tensor):
        _check_q4(t, "k/v")
        return FA_KV_Q4_0, tuple(t.shape)
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError("dense k/v must be contiguous [B, Hkv, S, D] tensors")
    return FA_KV_DENSE, tuple(t.shape)


def fa_fwd_kv(q, k, v, o=None, *, Sk: int | None = None, causal: bool = True,
              q_pos_offset: int | None = None, scale: float | None = None,
              workspace: torch.Tensor | None = None, rescale_count: torch.Tensor | None = None,
              p_max: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Attention over K/V caches whose formats are chosen independently (each a dense tensor in
    q's dtype or a Q4Tensor) and whose token capacity (their third dimension) may exceed the Sk
    tokens filled (default: the capacity).  q_pos_offset defaults to Sk - Sq.  With p_max (f32
    [B, Hq, Sq]) the call goes through fa_fwd_kv_stats, which writes each row's largest P."""
    if o is None:
        o = torch.empty_like(q)
    if q.dim() != 4 or not q.is_contiguous() or not o.is_contiguous() or o.shape != q.shape:
        raise ValueError("q and o must be contiguous [B, Hq, Sq, D] tensors of the same shape")
    kf, (Bk, Hkv, Scap, Dk) = _side(k)
    vf, vshape = _side(v)
    if vshape != (Bk, Hkv, Scap, Dk):
        raise ValueError("k and v must have the same [B, Hkv, capacity, D]")
    B, Hq, Sq, D = q.shape
    if Bk != B or Dk != D:
        raise ValueError("k/v batch or head dim does not match q")
    for t, f in ((k, kf), (v, vf)):
        if f == FA_KV_DENSE and t.dtype != q.dtype:
            raise TypeError("dense k/v must have the dtype of q")
    Sk = Scap if Sk is None else int(Sk)
    if q_pos_offset is None:
        q_pos_offset = Sk - Sq
    if scale is None:
        scale = D ** -0.5
    _on_device(q, k, v, o, workspace, rescale_count, p_max)
    lib = load()
    if workspace is None:
        need = lib.fa_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(q_pos_offset), int(bool(causal)))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc_ptr = None
    if rescale_count is not None:
        if rescale_count.dtype != torch.int32 or rescale_count.numel() != B * Hq * Sq:
            raise ValueError("rescale_count must be int32 [B, Hq, Sq]")
        rc_ptr = rescale_count.data_ptr()
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, Sq, Sk, Scap, D,
            int(q_pos_offset), int(bool(causal)), float(scale), _dtype_code(q.dtype), kf, vf,
            ws_ptr, ws_bytes, rc_ptr)
    if p_max is None:
        _check(lib.fa_fwd_kv(*args, _stream(stream)), "fa_fwd_kv")
    else:
        if (p_max.dtype != torch.float32 or p_max.numel() != B * Hq * Sq
                or not p_max.is_contiguous()):
            raise ValueError("p_max must be a contiguous float32 [B, Hq, Sq] tensor")
        _check(lib.fa_fwd_kv_stats(*args, p_max.data_ptr(), _stream(stream)), "fa_fwd_kv_stats")
    return o


def fa_fwd_kv_stats(q, k, v, o=None, *, p_max: torch.Tensor, **kw) -> torch.Tensor:
    """fa_fwd_kv that also writes, per query row, the largest softmax numerator P it produced
    (p_max: f32 [B, Hq, Sq]; see fa.h)."""
    return fa_fwd_kv(q, k, v, o, p_max=p_max, **kw)


def q4_0_cache(B: int, H: int, capacity: int, D: int, device="cuda") -> Q4Tensor:
    """An empty (uninitialised) q4_0 cache of logical shape [B, H, capacity, D]."""
    nbytes = fa_q4_0_bytes(B, H, capacity, D)
    if nbytes == 0:
        raise ValueError("D must be a positive multiple of 32")
    return Q4Tensor(torch.empty(nbytes, dtype=torch.uint8, device=device), B, H, capacity, D)


def fa_append_q4_0(k_new: torch.Tensor, k_cache: Q4Tensor, pos0: int,
                   v_new: torch.Tensor | None = None, v_cache: Q4Tensor | None = None, *,
                   stream=None) -> None:
    """Quantize k_new (and v_new) [B, H, S_new, D] into tokens pos0 .. pos0 + S_new - 1 of the
    q4_0 caches, in one launch."""
    if k_new.dim() != 4 or not k_new.is_contiguous():
        raise ValueError("k_new must be a contiguous [B, H, S_new, D] tensor")
    B, H, S_new, D = k_new.shape
    if (k_cache.B, k_cache.H, k_cache.D) != (B, H, D):
        raise ValueError("k_cache does not match k_new")
    if (v_new is None) != (v_cache is None):
        raise ValueError("give both v_new and v_cache, or neither")
    if v_new is not None:
        if tuple(v_new.shape) != tuple(k_new.shape) or not v_new.is_contiguous():
            raise ValueError("v_new must match k_new")
        if v_cache.shape != k_cache.shape:
            raise ValueError("v_cache must match k_cache")
        _check_q4(v_cache, "v_cache")
    _check_q4(k_cache, "k_cache")
    _on_device(k_new, k_cache, v_new, v_cache)
    _check(load().fa_append_q4_0(k_new.data_ptr(), v_new.data_ptr() if v_new is not None else None,
                                 k_cache.data_ptr(),
                                 v_cache.data_ptr() if v_cache is not None else None, B, H, S_new,
                                 k_cache.S, int(pos0), D, _dtype_code(k_new.dtype),
                                 _stream(stream)), "fa_append_q4_0")


def fa_prefill_append_workspace_bytes(B: int, Hq: int, Hkv: int, S_new: int, kv_capacity: int,
                                      D: int, pos0: int) -> int:
    return int(load().fa_prefill_append_workspace_bytes(B, Hq, Hkv, S_new, kv_capacity, D, pos0))


def fa_prefill_append_q4_0(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                           k_cache: Q4Tensor, v_cache: Q4Tensor, pos0: int,
                           o: torch.Tensor | None = None, *, scale: float | None = None,
                           workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Append a chunk (k_new, v_new [B, Hkv, S_new, D]) to q4_0 caches at pos0 and run the
    chunk's causal prefill (q [B, Hq, S_new, D] at positions pos0 ..) over the whole cache, in
    one launch where the shape allows (see fa.h)."""
    if o is None:
        o = torch.empty_like(q)
    if q.dim() != 4 or not q.is_contiguous() or not o.is_contiguous() or o.shape != q.shape:
        raise ValueError("q and o must be contiguous [B, Hq, S_new, D] tensors of the same shape")
    B, Hq, S_new, D = q.shape
    for name, t in (("k_new", k_new), ("v_new", v_new)):
        if t.dim() != 4 or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous [B, Hkv, S_new, D] tensor of q's dtype")
    Bk, Hkv, Sn, Dk = k_new.shape
    if (Bk, Sn, Dk) != (B, S_new, D) or tuple(v_new.shape) != tuple(k_new.shape):
        raise ValueError("k_new / v_new do not match q")
    _check_q4(k_cache, "k_cache")
    _check_q4(v_cache, "v_cache")
    if k_cache.shape != v_cache.shape or (k_cache.B, k_cache.H, k_cache.D) != (B, Hkv, D):
        raise ValueError("the caches must be [B, Hkv, capacity, D] q4_0 tensors")
    if scale is None:
        scale = D ** -0.5
    _on_device(q, k_new, v_new, k_cache, v_cache, o, workspace)
    lib = load()
    if workspace is None:
        need = lib.fa_prefill_append_workspace_bytes(B, Hq, Hkv, S_new, k_cache.S, D, int(pos0))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.fa_prefill_append_q4_0(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                      k_cache.data_ptr(), v_cache.data_ptr(), o.data_ptr(), B, Hq,
                                      Hkv, S_new, k_cache.S, D, int(pos0), float(scale),
                                      _dtype_code(q.dtype), ws_ptr, ws_bytes, _stream(stream)),
           "fa_prefill_append_q4_0")
    return o


def fa_decode_paged(q, k_pages, v_pages, block_table: torch.Tensor, seq_lens: torch.Tensor,
                    o=None, *, scale: float | None = None,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode one token per sequence over paged K/V pools.  q [B, Hq, 1, D]; k_pages, v_pages
    [num_pages, Hkv, page_size, D] each dense (dtype of q) or a Q4Tensor of that shape;
    block_table int32 [B, pages_per_seq] and seq_lens int32 [B] on the device."""
    if o is None:
        o = torch.empty_like(q)
    if q.dim() != 4 or q.shape[2] != 1 or not q.is_contiguous() or o.shape != q.shape:
        raise ValueError("q and o must be contiguous [B, Hq, 1, D] tensors")
    kf, (NP, Hkv, page, Dk) = _side(k_pages)
    vf, vshape = _side(v_pages)
    if vshape != (NP, Hkv, page, Dk):
        raise ValueError("k_pages and v_pages must have the same [num_pages, Hkv, page_size, D]")
    B, Hq, _, D = q.shape
    if Dk != D:
        raise ValueError("head dim of the pools does not match q")
    for t, f in ((k_pages, kf), (v_pages, vf)):
        if f == FA_KV_DENSE and t.dtype != q.dtype:
            raise TypeError("dense pools must have the dtype of q")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B \
            or not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [B, pages_per_seq] tensor")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be an int32 [B] tensor")
    pps = block_table.shape[1]
    _on_device(q, k_pages, v_pages, o, block_table, seq_lens, workspace)
    lib = load()
    if workspace is None:
        need = lib.fa_decode_paged_workspace_bytes(B, Hq, Hkv, D, page, pps)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = D ** -0.5
    _check(lib.fa_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), o.data_ptr(),
                               block_table.data_ptr(), seq_lens.data_ptr(), B, Hq, Hkv, D, NP,
                               page, pps, float(scale), _dtype_code(q.dtype), kf, vf,
                               workspace.data_ptr(), workspace.numel(), _stream(stream)),
           "fa_decode_paged")
    return o


def fa_fwd_explicit(q, k, v, o=None, *, causal: bool = True, q_pos_offset: int | None = None,
                    scale: float | None = None, workspace: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """The explicit (non-flash) path: dense K/V (q4_0 sides expanded first), S = scale Q K^T in
    f32, softmax, O = P V.  Same arguments as fa_fwd_kv without a capacity."""
    if o is None:
        o = torch.empty_like(q)
    if q.dim() != 4 or not q.is_contiguous() or not o.is_contiguous() or o.shape != q.shape:
        raise ValueError("q and o must be contiguous [B, Hq, Sq, D] tensors of the same shape")
    kf, (Bk, Hkv, Sk, Dk) = _side(k)
    vf, vshape = _side(v)
    if vshape != (Bk, Hkv, Sk, Dk):
        raise ValueError("k and v must have the same [B, Hkv, Sk, D]")
    B, Hq, Sq, D = q.shape
    if Bk != B or Dk != D:
        raise ValueError("k/v batch or head dim does not match q")
    if q_pos_offset is None:
        q_pos_offset = Sk - Sq
    if scale is None:
        scale = D ** -0.5
    _on_device(q, k, v, o, workspace)
    lib = load()
    if workspace is None:
        need = lib.fa_explicit_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, kf, vf)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(lib.fa_fwd_explicit(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv,
                               Sq, Sk, D, int(q_pos_offset), int(bool(causal)), float(scale),
                               _dtype_code(q.dtype), kf, vf, workspace.data_ptr(),
                               workspace.numel(), _stream(stream)), "fa_fwd_explicit")
    return o
