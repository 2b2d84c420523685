"""bench.py's host-side rules on CPU: which workloads flush L2 between timed
steps, what the JSON config says about it, the warm-up floor, and the
stored DRAM-traffic table (every entry names a known workload and is used
only while its pass's sources are unchanged)."""
import os

import pytest

import bench
from exact_tiled_attention_04_gb300 import inputs as I


def test_flush_only_when_the_inputs_fit_in_l2():
    W = I.WORKLOADS
    # q, k, v of the headline shape: 402 MB, more than the 129 MB L2
    assert bench.input_bytes(W["b2h32_n8192_d128"]) == 3 * 2 * 32 * 8192 * 128 * 2
    assert not bench.needs_flush(W["b2h32_n8192_d128"])
    assert not bench.needs_flush(W["decode_b8h32kv8_n16384_d128"])
    assert not bench.needs_flush(W["bwd_b2h32_n8192_d128"])
    for name in ("single_head_n512", "tail_n1000", "b4h16_n2048", "long_n16384", "bwd_b4h16_n2048"):
        assert bench.needs_flush(W[name]), name
    # the backward pass reads q, k, v, o, dO and lse
    w = W["bwd_b4h16_n2048"]
    per = w.B * w.H * w.N * w.d * 2
    assert bench.input_bytes(w) == 5 * per + 4 * w.B * w.H * w.N


@pytest.mark.parametrize("name,flushed", [("b2h32_n8192_d128", False), ("b4h16_n2048", True)])
def test_config_states_the_l2_rule(name, flushed):
    cfg = bench.config_of(I.WORKLOADS[name], 1, 0)
    assert ("written before every timed step" in cfg["l2"]) == flushed
    assert ("larger than L2" in cfg["l2"]) == (not flushed)
    assert cfg["workload"] == name and "model" not in cfg


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2", "--steps", "1"])


def test_traffic_table_names_known_workloads():
    """An entry is used only while its pass's sources hash to the stored
    value; a stale entry reads as no measurement (None)."""
    path = os.path.join(bench.ROOT, "profiles", "traffic.txt")
    seen = []
    with open(path) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            kv = dict(item.split("=", 1) for item in line.split())
            name = kv["workload"]
            assert name in I.WORKLOADS, name
            backward = I.WORKLOADS[name].backward
            assert float(kv["dram_bytes_per_launch"]) > 0
            fresh = kv["kernel_hash"] == bench.kernel_source_hash(backward)
            expect = float(kv["dram_bytes_per_launch"]) if fresh else None
            assert bench.stored_traffic(name, backward) == expect, name
            seen.append(name)
    assert "b2h32_n8192_d128" in seen
    assert bench.stored_traffic("no_such_workload") is None
