"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention or quantization arithmetic: it only draws N(0,1) tensors from a
seeded CPU generator, rounds them to the input dtype and (for the score-ramp case) writes a
deterministic pattern into one column of Q and K.

Recipe (the same for every consumer):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed draws f32 N(0,1) for Q, then K,
    then V, in that order, each then rounded to f16 or bf16;
  * layouts are head-major: Q, O ``[B, Hq, Sq, D]``; K, V ``[B, Hkv, Sk, D]``;
  * the score ramp sets Q[..., 0] = 8 and K[..., j, 0] = 2 * floor(j / 128) / (8 * scale), both
    rounded to the input dtype, so each key block of 128 adds about 2.0 to every row's scaled
    score and a row's maximum outgrows a 10-point frame roughly every five blocks.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    dtype: str            # "f16" | "bf16"
    kv_format: str        # "dense" | "q4_0"
    causal: bool = True
    ramp: bool = False
    seed: int = 0

    @property
    def q_pos_offset(self) -> int:
        # query chunk at the end of the key range (bottom-right aligned causal mask)
        return self.Sk - self.Sq

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def visible_pairs(self) -> int:
        """Sum over query rows of the number of visible keys (causal, diagonal included)."""
        if not self.causal:
            return self.Sq * self.Sk
        off = self.q_pos_offset
        return sum(min(self.Sk, off + i + 1) for i in range(self.Sq))

    def flops(self) -> int:
        """4 * D * Hq * B * (visible query-key pairs): QK^T and PV, masked pairs not counted."""
        return 4 * self.D * self.Hq * self.B * self.visible_pairs()


# The five workloads: dense self-attention (head dim 64), chunked prefill at 2K/8K/16K keys with
# GQA 32/8 (f16 and bf16, with and without the score ramp), q4_0 chunked prefill, q4_0 decode.
WORKLOADS = {
    "selfattn_b2_s512_h8_d64_f16": Workload("selfattn_b2_s512_h8_d64_f16", 2, 8, 8, 512, 512,
                                            64, "f16", "dense", seed=1001),
    "prefill_gqa32x8_d128_sq2048_sk2048_f16": Workload(
        "prefill_gqa32x8_d128_sq2048_sk2048_f16", 1, 32, 8, 2048, 2048, 128, "f16", "dense",
        seed=1002),
}
for _sk in (8192, 16384):
    for _dt in ("f16", "bf16"):
        _n = f"prefill_gqa32x8_d128_sq2048_sk{_sk}_{_dt}"
        WORKLOADS[_n] = Workload(_n, 1, 32, 8, 2048, _sk, 128, _dt, "dense", seed=1003)
    _n = f"prefill_gqa32x8_d128_sq2048_sk{_sk}_f16_ramp"
    WORKLOADS[_n] = Workload(_n, 1, 32, 8, 2048, _sk, 128, "f16", "dense", ramp=True, seed=1003)
WORKLOADS["prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16"] = Workload(
    "prefill_q4_0_gqa32x8_d128_sq2048_sk16384_f16", 1, 32, 8, 2048, 16384, 128, "f16", "q4_0",
    seed=1004)
WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"] = Workload(
    "decode_q4_0_b4_gqa32x8_d128_sk65536_f16", 4, 32, 8, 1, 65536, 128, "f16", "q4_0",
    seed=1005)


def torch_dtype(name: str) -> torch.dtype:
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


def make_qkv(w: Workload, *, seed: int | None = None, device: str = "cpu",
             generate_on_device: bool = False):
    """Q, K, V for workload ``w`` (dense values, in the workload dtype), generated on the CPU from
    the seed and then moved to ``device``.  For q4_0 workloads K and V are the values that get
    quantized."""
    return make_tensors(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.dtype,
                        seed=w.seed if seed is None else seed, ramp=w.ramp, scale=w.scale,
                        device=device, generate_on_device=generate_on_device)


def make_tensors(B, Hq, Hkv, Sq, Sk, D, dtype="f16", *, seed=0, ramp=False, scale=None,
                 device="cpu", generate_on_device=False):
    """Q, K, V drawn from one seeded generator in Q, K, V order.  By default the draw happens on
    the CPU (the stream the parity tests and the oracle share) and the tensors are then moved to
    ``device``; with ``generate_on_device`` a CUDA generator with the same seed draws them in
    place (same distribution, different stream; used for large benchmark inputs)."""
    gdev = device if generate_on_device else "cpu"
    g = torch.Generator(device=gdev).manual_seed(int(seed))
    dt = torch_dtype(dtype)
    q = torch.randn(B, Hq, Sq, D, generator=g, dtype=torch.float32, device=gdev).to(dt)
    k = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float32, device=gdev).to(dt)
    v = torch.randn(B, Hkv, Sk, D, generator=g, dtype=torch.float32, device=gdev).to(dt)
    if ramp:
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        q[..., 0] = 8.0
        j = torch.arange(Sk, dtype=torch.float64, device=gdev)
        col = (2.0 * torch.floor(j / 128.0) / (8.0 * scale)).to(dt)
        k[..., 0] = col
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v
