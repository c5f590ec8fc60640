"""Host-side arithmetic of bench.py, on the CPU: the algorithmic bytes behind
the roofline fraction, checked against the stored tile layout, and the rule
that a DRAM-traffic record counts only for the decode sources it was
measured on."""

import importlib.util
import json
import pathlib
import types

import numpy as np

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _case(B, Hq, Hkv, GS, P, hist, sink, rec):
    return types.SimpleNamespace(B=B, Hq=Hq, Hkv=Hkv, GS=GS, P=P, hist_len=np.asarray(hist),
                                 sink_len=np.asarray(sink), rec_len=np.asarray(rec))


def test_algorithmic_bytes_of_the_100k_workload():
    b = _bench()
    total, parts = b.algorithmic_bytes(_case(1, 32, 8, 128, 16, [99680], [64], [256]))
    # one stored 16-token tile of one KV head: 512 B of K codes, 512 B of V
    # codes and 16 records of (s_k, z_k, s_v, z_v) in fp16
    tile = 512 + 512 + 16 * 4 * 2
    assert tile == 1152
    assert parts["hist"] == (99680 // 16) * tile * 8
    assert parts["tiers"] == (64 + 256) * 8 * 2 * 128 * 2          # K and V rows, bf16
    assert parts["rot"] == 8 * 2 * 128 * 128 * 4                    # R_k and R_v^T, fp32
    assert parts["page_table"] == (99680 // 16) * 4 * 8             # every KV head reads the page ids
    assert parts["q_out"] == 32 * 128 * 2 + 32 * 128 * 4            # bf16 q in, fp32 out
    assert total == sum(parts.values()) == 59_998_912


def test_group_64_history_bytes_and_ragged_pages():
    b = _bench()
    _, parts = b.algorithmic_bytes(_case(2, 8, 2, 64, 16, [100, 17], [64, 3], [256, 0]))
    # group 64: two (s, z) pairs per tensor and token, a tile of 1280 B
    assert parts["hist"] == (100 + 17) * 2 * (1280 // 16)
    assert parts["page_table"] == (7 + 2) * 4 * 2                  # ceil(100/16) + ceil(17/16) pages
    assert parts["tiers"] == (64 + 256 + 3) * 2 * 512


def test_bf16_path_bytes():
    b = _bench()
    c = _case(1, 32, 8, 128, 16, [99680], [64], [256])
    # the BF16 pool holds all 100,000 tokens: 512 B per token per KV head
    assert b.bf16_bytes(c) == 100000 * 8 * 512 + (100000 // 16) * 4 * 8 + 32 * 128 * 6


def test_traffic_record_counts_only_for_its_sources(tmp_path):
    b = _bench()
    rec = {"workload": "w", "dram_bytes_read": 1000, "dram_bytes_write": 24,
           "source_sha256": b.kernel_source_digest()}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    b.TRAFFIC_RECORD = str(path)
    assert b.measured_traffic("w") == 1024
    assert b.measured_traffic("another workload") is None
    rec["source_sha256"] = "0" * 64                               # measured on other sources
    path.write_text(json.dumps(rec))
    assert b.measured_traffic("w") is None
    b.TRAFFIC_RECORD = str(tmp_path / "missing.json")
    assert b.measured_traffic("w") is None


def test_append_bytes_and_flops_of_the_append_workload():
    """64 sequences x 4096 tokens x 8 KV heads: K and V rows in (bf16, 256 B
    each), and out per token the K and V share of a stored page tile (1,280 B
    per 16 tokens at group 64, 1,152 B at group 128); the rotation is one
    128 x 128 product per row and tensor."""
    b = _bench()
    n = 64 * 4096 * 8
    alg, flops = b.append_bytes_flops(n, 64)
    assert alg == n * (2 * 256 + 1280 // 16) == 1_241_513_984
    assert b.append_bytes_flops(n, 128)[0] == n * (2 * 256 + 1152 // 16)
    assert flops == 2 * 2 * 128 * 128 * n
