"""Host-side pieces of bench.py, on CPU: the timed region runs exactly the
requested number of steps for any --steps, the clock pre-roll is bounded,
launch counts follow the plan, and recorded ncu traffic is reported only for
the sources it was measured on."""
import json

import pytest

import bench


@pytest.mark.parametrize("steps", [1, 20, 64, 65, 20000])
def test_timed_region_runs_exactly_the_requested_steps(steps):
    calls, marks = [], []
    bench.timed_loop(lambda: calls.append(len(marks)), steps, marks.append)
    assert marks == [0, 1]
    assert len(calls) == steps
    assert set(calls) == {1}          # every call between the two marks


def test_clock_preroll_is_bounded():
    assert bench.preroll_calls(None) == 0
    assert bench.preroll_calls(0) == 0
    assert bench.preroll_calls(600.0) == 1000           # 0.6 s of 600 us calls
    assert bench.preroll_calls(0.001) == 20000          # capped


def test_launch_count_follows_the_plan():
    assert bench.decode_launches(1, 3) == 2             # stream form + merge
    assert bench.decode_launches(4, 1) == 2             # split + log-sum-exp reduce
    assert bench.decode_launches(8, 2) == 1             # cluster form merges in place
    assert bench.decode_launches(1, 1) == 1
    assert bench.decode_launches(1, 0) == 1


def test_traffic_is_reported_only_for_unchanged_sources(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    h = bench.src_hash(bench.DECODE_SOURCES)
    f.write_text(json.dumps({"w": {"sources_sha256_16": h, "dram_bytes_per_launch": 123},
                             "old": {"sources_sha256_16": "0" * 16,
                                     "dram_bytes_per_launch": 456}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.stored_traffic("w", bench.DECODE_SOURCES) == 123
    assert bench.stored_traffic("old", bench.DECODE_SOURCES) is None
    assert bench.stored_traffic("missing", bench.DECODE_SOURCES) is None


def test_headline_bytes_match_the_workload():
    from paged_kv_decode_22_gb300.workloads import decode_configs
    cfg = decode_configs()[bench.HEADLINE]
    S, H, Hk, D, B = (cfg["num_seqs"], cfg["num_heads"], cfg["num_kv_heads"], cfg["head_size"],
                      cfg["block_size"])
    assert (S, H, Hk, D, B, cfg["dtype"]) == (256, 64, 8, 128, 16, "bf16")
    assert set(cfg["context_lens"]) == {4096}
    kv = S * 4096 * Hk * D * 2 * 2
    assert kv == 4294967296                             # 4.3 GB of K and V per call
    assert kv > 30 * bench.L2_BYTES


def test_oracle_sample_is_a_prefix_of_the_workload():
    c = bench._oracle_sample_case("mqa_ragged_b64", 3)
    from paged_kv_decode_22_gb300.workloads import decode_configs
    cfg = decode_configs()["mqa_ragged_b64"]
    assert list(c.context_lens) == list(cfg["context_lens"][:3])
    assert (c.num_heads, c.num_kv_heads, c.head_size, c.block_size, c.dtype) == (
        cfg["num_heads"], cfg["num_kv_heads"], cfg["head_size"], cfg["block_size"], cfg["dtype"])
