"""bench.py's DRAM-traffic record: parsing an ncu launch list (CSV) into the
median bytes per launch of each phase's kernel, stored with a hash of the
CUDA sources and reported only while that hash still matches."""

import json

import pytest

import bench


def _csv(rows):
    head = '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",' \
           '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
    lines = ["==PROF== a line ncu prints before the table\n", head]
    for i, name, rd, wr in rows:
        for metric, val in (("dram__bytes_read.sum", rd), ("dram__bytes_write.sum", wr),
                            ("gpu__time_duration.sum", 1000)):
            lines.append(f'"{i}","1","python3","h","{name}","1","7","(576, 1, 1)","(152, 1, 1)","0","10.3",'
                         f'"Command line profiler metrics","{metric}","byte","{val:,}"\n')
    return "".join(lines)


def test_record_and_load(tmp_path, monkeypatch):
    traffic = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(traffic))
    rows = [(0, "void w4a16_tc_kernel<256, 64, 0, 3, 1>(W4Params)", 500_000_000, 300_000_000),
            (1, "void w4a16_tc_kernel<256, 64, 0, 3, 1>(W4Params)", 520_000_000, 300_000_000),
            (2, "void w4a16_tc_kernel<256, 64, 0, 3, 1>(W4Params)", 900_000_000, 300_000_000),
            (3, "w4_decode_nvf4_kernel(W4Params)", 126_000_000, 4_000_000),
            (4, "nvfp4_encode_kernel(Nvfp4Batch)", 400_000_000, 140_000_000),
            (5, "void w4a16_tc_kernel<64, 256, 1, 3, 0>(W4Params)", 131_000_000, 1_000_000)]
    src = tmp_path / "launches.csv"
    src.write_text(_csv(rows))
    bench.record_traffic(str(src))
    d = json.loads(traffic.read_text())
    assert d["source_sha256"] == bench.source_hash()
    assert d["phases"]["prefill"]["dram_bytes_per_launch"] == 820_000_000  # median of three launches
    assert d["phases"]["prefill"]["launches"] == 3
    assert d["phases"]["decode_m1"]["dram_bytes_per_launch"] == 130_000_000
    assert d["phases"]["decode_m8"]["dram_bytes_per_launch"] == 130_000_000
    assert d["phases"]["decode_m64"]["dram_bytes_per_launch"] == 132_000_000
    assert d["phases"]["requant"]["dram_bytes_per_launch"] == 540_000_000
    assert "fp8_gemm" not in d["phases"]
    assert bench.load_traffic("prefill") == 820_000_000
    assert bench.load_traffic("fp8_gemm") is None
    # a record taken from other sources is not reported
    d["source_sha256"] = "0" * 64
    traffic.write_text(json.dumps(d))
    assert bench.load_traffic("prefill") is None


def test_missing_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.load_traffic("prefill") is None


def test_replica_value_units():
    assert bench.whole_job(None, 1, 128_090_140, 0.0512) == pytest.approx(128_090_140 / 0.0512 / 1e6)
