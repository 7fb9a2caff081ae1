"""Host arithmetic of the benchmark line, on CPU: the roofline object, the
algorithmic bytes, the DRAM-counter lookup keyed to each kernel's sources,
and the two-level chain's per-stage rooflines."""

import json

import numpy as np
import pytest

import bench


def test_hbm_roofline_is_bytes_over_time_against_the_peak():
    peak, _ = bench.measured_peak()
    r = bench.hbm_roofline(2 * 10**9, 1000.0, traffic=123.0)  # 2 GB in 1 ms = 2000 GB/s
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(2000.0)
    assert r["peak"] == peak and r["frac"] == pytest.approx(2000.0 / peak)
    assert r["traffic"] == 123.0 and r["algorithmic_bytes_per_launch"] == 2 * 10**9


def test_algorithmic_bytes_clamp_lengths_to_the_row():
    lengths = np.array([-5, 0, 10, 100, 1000], dtype=np.int32)
    # scores read: 0 + 0 + 10 + 100 + 100 (clamped to stride 100); indices written: 5 x 8
    assert bench.algorithmic_bytes(lengths, 100, 5, 8) == 4 * 210 + 4 * 5 * 8


def test_two_level_rooflines():
    nb = np.array([0, 1, 9, 4096], dtype=np.int64)
    res = {name: {"us_per_call": 10.0} for name in ("amax8_varlen", "topk_over_keys",
                                                    "sort_candidate_blocks")}
    bench.two_level_rooflines(res, nb, 4096, 4, 512, "B1024_w262144_k512_paged64")
    # keys: 32 bytes per block but the newest of each row, 4 bytes per key written
    assert res["amax8_varlen"]["roofline"]["algorithmic_bytes_per_launch"] == \
        32 * (0 + 0 + 8 + 4095) + 4 * (0 + 1 + 9 + 4096)
    assert res["topk_over_keys"]["roofline"]["algorithmic_bytes_per_launch"] == \
        4 * (0 + 1 + 9 + 4096) + 4 * 4 * 512
    assert res["sort_candidate_blocks"]["roofline"]["algorithmic_bytes_per_launch"] == 4 * 4 * 512 * 4
    for stage in res.values():
        r = stage["roofline"]
        assert r["achieved"] == pytest.approx(r["algorithmic_bytes_per_launch"] / 10e-6 / 1e9)
    assert "kernel alone" in res["sort_candidate_blocks"]["note"]


def test_dram_counters_follow_their_kernels_sources(tmp_path, monkeypatch):
    """A recorded entry counts only while the hash of its kernel's sources is
    the one recorded; a comment edit leaves the hash alone, a code edit does
    not; every listed source exists."""
    csrc = tmp_path / "sparse_attention_indexer_fp32_gb300" / "csrc"
    csrc.mkdir(parents=True)
    real = bench.os.path.join(bench.ROOT, "sparse_attention_indexer_fp32_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        for name in files:
            assert bench.os.path.exists(bench.os.path.join(real, name)), name
            (csrc / name).write_text(open(bench.os.path.join(real, name)).read())
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h_rows = bench.kernel_source_hash("topk_rows_kernel")
    h_short = bench.kernel_source_hash("topk_short_kernel")
    doc = {"workloads": {
        "a": {"kernel": "topk_rows_kernel", "kernel_source_hash": h_rows, "dram_bytes_per_launch": 5.0},
        "b": {"kernel": "topk_short_kernel", "kernel_source_hash": "0" * 16, "dram_bytes_per_launch": 6.0},
        "c": {"kernel": "no_such_kernel", "kernel_source_hash": h_rows, "dram_bytes_per_launch": 7.0}}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(doc))
    assert bench.profiled_traffic("a") == 5.0
    assert bench.profiled_traffic("b") is None and bench.profiled_traffic("c") is None
    assert bench.profiled_traffic("missing") is None
    short = csrc / "topk_short.cuh"
    short.write_text(short.read_text() + "\n// a comment\n\n")
    assert bench.kernel_source_hash("topk_short_kernel") == h_short
    short.write_text(short.read_text() + "constexpr int kNewConstant = 1;\n")
    assert bench.kernel_source_hash("topk_short_kernel") != h_short
    assert bench.kernel_source_hash("topk_rows_kernel") == h_rows  # not one of its sources
    assert bench.profiled_traffic("a") == 5.0


def test_reference_arm_prints_the_gpu_arms_config(capsys):
    """The reference arm (the host oracle) reports on the same workload
    config, metric and unit as the GPU arm, with dtype f32."""
    from synth import CONFIGS

    bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["dtype"] == "f32"
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    want = dict(bench.workload_config(CONFIGS[bench.WORKLOADS["w262144_k512_paged"]]),
                parallelism="replicas x1")
    assert line["config"] == want
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_summary_lists_every_timed_workload_last():
    roof = bench.hbm_roofline(10**9, 200.0)
    line = {"config": {"workload": "A"}, "value": 200.0, "roofline": roof,
            "also": [{"workload": "B", "us_per_call": 100.0, "roofline": roof}],
            "prefill": [{"workload": "C", "us_per_call": 50.0, "roofline": roof}],
            "two_level": {"workload": "A", "stages": {"amax8_varlen": {"us_per_call": 1.0,
                                                                       "roofline": roof}}},
            "latency": {"workload": "L", "eager_us_per_call": 9.0, "graph_replay_us_per_call": 8.0,
                        "cold_l2_eager_us_per_call": 12.0,
                        "cold_l2_graph_replay_us_per_call": 11.0}}
    summ = bench.summary_of(line)
    assert [e["w"] for e in summ] == ["A", "B", "C", "amax8_varlen_A", "L"]
    assert summ[1]["us"] == 100.0 and summ[1]["frac"] == round(roof["frac"], 3)
    assert len(json.dumps(summ)) < 1500


def test_sweep_paths_and_summary_tables():
    """The dispatch sweep's path list per shape, and its markdown summary on
    a made-up measurement."""
    names = [n for n, _ in bench.sweep_paths(8192, 64, 152)]
    assert names[:3] == ["auto", "short", "short_regs"] and "G2_sampled" in names
    assert "G4_full" not in names  # 8192 / 4 < one stage
    names = [n for n, _ in bench.sweep_paths(262144, 1024, 152)]
    assert "G16_sampled" in names and "G1_split112" in names and "G1_split_all" not in names
    assert bench._sweep_split_rows(1024, 152) == 112
    paths = {n: 10.0 + i for i, (n, _) in enumerate(bench.sweep_paths(262144, 4, 152))}
    doc = {"gpu": "test", "sm_count": 152, "reps": 20, "warmup": 3, "command": "cmd",
           "results": [{"width": 262144, "B": 4, "lengths": "ragged", "k": 512, "paths": paths,
                        "algorithmic_bytes": 10 ** 6, "auto_counters": {}}]}
    md = bench.sweep_markdown(doc)
    assert "| 512 | 262144 | 4 | 10.0 |" in md and "G1_split4" in md
