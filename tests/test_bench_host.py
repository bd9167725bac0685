"""Host logic of bench.py without a GPU: the algorithmic byte count, clock parsing, the max-over-
ranks reduction on two gloo ranks, and the CPU reference arm on a small workload."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import fa_inputs


def test_decode_kv_bytes():
    w = fa_inputs.WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"]
    # 4 sequences x 8 kv heads x 65536 keys x (64 + 8) bytes, for K and for V
    assert bench.kv_bytes_q4_0(w) == 301_989_888


def test_decode_workloads_report_kv_bandwidth():
    w = fa_inputs.WORKLOADS["decode_q4_0_b4_gqa32x8_d128_sk65536_f16"]
    # 301 989 888 bytes in 0.06 ms: 5033.2 GB/s; a quarter of the rows: a quarter of the bytes
    v, unit = bench.rate(w, 0.06)
    assert unit == "GB/s" and abs(v - 301_989_888 / 0.06e-3 / 1e9) < 1e-6
    assert abs(bench.rate(w, 0.06, 0.25)[0] - v / 4) < 1e-6
    p = fa_inputs.WORKLOADS["prefill_gqa32x8_d128_sq2048_sk16384_f16"]
    v, unit = bench.rate(p, 0.5)
    assert unit == "TFLOP/s" and abs(v - p.flops() / 0.5e-3 / 1e12) < 1e-9
    assert not bench.is_decode(p) and bench.is_decode(w)


def test_parse_clocks():
    lines = [
        "0, 1965, 2070, 1012.3, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1905, 2070, 1300.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1935, 2070, 1250.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage",
    ]
    c = bench.parse_clocks(lines)
    assert c["sm_mhz"] == 1935 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    got = bench.aggregate(float(rank + 1) * 1.5, world)
    bench.barrier(world)
    out[rank] = got
    dist.destroy_process_group()


def test_aggregate_is_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 3.0, 1: 3.0}


def test_reference_arm_line(capsys):
    rc = bench.main(["--impl", "reference", "--workload", "selfattn_b2_s512_h8_d64_f16",
                     "--steps", "3", "--warmup", "3"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["unit"] == line["unit"]


def test_traffic_table_entries_match_what_bench_looks_up():
    """Every line of profiles/dram_traffic.txt names a kernel key bench.py asks for (kernel,
    dtype, K/V format) and an existing workload, so a capture cannot be silently orphaned by a
    typo (whether its source hash is current is a separate matter: a stale one reports null)."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                        "dram_traffic.txt")
    entries = [ln.split() for ln in open(path) if ln.strip() and not ln.startswith("#")]
    assert entries
    asked = {("decode_split_kernel_f16_q4_0", bench.DECODE_WORKLOAD)}
    for kernel in ("prefill_kernel", "prefill_seg_kernel"):
        for name, w in fa_inputs.WORKLOADS.items():
            asked.add((f"{kernel}_{w.dtype}_{w.kv_format}", name))
    for e in entries:
        assert len(e) >= 5, e
        key, srcs, sha, nbytes, workload = e[:5]
        assert (key, workload) in asked, e
        assert len(sha) == 16 and int(nbytes) > 0
        for f in srcs.split("+"):
            src = os.path.join(bench.ROOT, "quantized_kv_cache_sm_gb300", "csrc", f)
            assert os.path.exists(src)
