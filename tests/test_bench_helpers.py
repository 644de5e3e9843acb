"""bench.py's byte models and its ncu traffic recorder, on CPU."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import kda_inputs as ki  # noqa: E402


def test_sector_model():
    # row i of a chunk reads its first i elements, rounded up to 32-byte sectors
    assert bench.sector_read_bytes(1, 4) == 0
    assert bench.sector_read_bytes(2, 4) == 32
    assert bench.sector_read_bytes(64, 4) == sum(-(-(4 * i) // 32) * 32 for i in range(64)) == 8960
    assert bench.sector_read_bytes(64, 2) == 4992


@pytest.mark.parametrize("bt", [16, 32, 64])
def test_algorithmic_bytes_per_chunk_length(bt):
    wl = ki.Workload("b", "packed", H=2, in_dtype="f32", out_dtype="bf16", seed=1, seqlens=(bt, 3), bt=bt)
    inp = ki.build(wl)
    want = 2 * (bench.sector_read_bytes(bt, 4) + bt * bt * 2 + bench.sector_read_bytes(3, 4) + 3 * bt * 2)
    assert bench.algorithmic_bytes(inp, 4, 2) == want


def test_kgb_bytes():
    wl = ki.Workload("k", "packed", H=3, in_dtype="bf16", out_dtype="f32", seed=2, seqlens=(70, 5))
    x = ki.build_kgb(wl, K=32)
    rows = 75
    assert bench.kgb_bytes(x, 2, 4) == rows * 3 * (32 * 2 + 32 * 4 + 2) + rows * 3 * 64 * 4


def test_l2_flush_rule():
    small = ki.build(ki.WORKLOADS["dense_1x64_h4_f32"])
    assert bench.flushes_l2(small) and bench.l2_policy(small) == ("flush", 1)
    bt16 = ki.build(ki.WORKLOADS["packed_16x512_h64_f32"].with_(bt=16))      # 67 MB
    kind, r = bench.l2_policy(bt16)
    fp = bench.full_tensor_bytes(bt16, 4, 4)
    assert kind == "rotate" and (r - 1) * fp >= 2 * bench.L2_BYTES and (r - 2) * fp < 2 * bench.L2_BYTES
    assert bench.l2_policy(ki.build(ki.WORKLOADS["packed_16x512_h64_f32"])) == ("none", 1)
    assert bench.workload_key(ki.WORKLOADS["packed_16x512_h64_f32"]) == "packed_16x512_h64_f32"
    assert bench.workload_key(ki.WORKLOADS["packed_16x512_h64_f32"].with_(bt=16)) == "packed_16x512_h64_f32_bt16"


CSV = '''==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python3.12","127.0.0.1","void kda_bt16_kernel<float, float>(SmallParams)","1","7","(64, 1, 1)","(2128, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","33,569,792"
"0","1","python3.12","127.0.0.1","void kda_bt16_kernel<float, float>(SmallParams)","1","7","(64, 1, 1)","(2128, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","0.07"
"0","1","python3.12","127.0.0.1","void kda_bt16_kernel<float, float>(SmallParams)","1","7","(64, 1, 1)","(2128, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","ns","14944"
'''


def test_record_traffic(tmp_path, monkeypatch):
    p = tmp_path / "t.csv"
    p.write_text(CSV)
    store = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(store))
    e = bench.record_traffic(str(p), "w_bt16", "kda_bt16_kernel", "ncu ...")
    assert e["dram_read"] == 33569792 and e["dram_write"] == 70000
    assert e["dram_bytes_per_launch"] == 33639792
    assert e["source_hash"] == bench.kernel_source_hash("kda_bt16_kernel")
    assert json.load(open(store))["w_bt16"]["kda_bt16_kernel"] == e
    # the record is used only while the kernel's sources are unchanged
    assert bench.ncu_traffic("kda_bt16_kernel", "w_bt16") == 33639792
    d = json.load(open(store))
    d["w_bt16"]["kda_bt16_kernel"]["source_hash"] = "stale"
    json.dump(d, open(store, "w"))
    assert bench.ncu_traffic("kda_bt16_kernel", "w_bt16") is None


def test_record_traffic_averages_consecutive_launches(tmp_path, monkeypatch):
    """Several consecutive launches: the record is their mean per launch."""
    lines = CSV.splitlines()
    second = [l.replace('"0","1","python', '"1","1","python').replace('"33,569,792"', '"33,569,800"')
              .replace('"0.07"', '"0.09"').replace('"14944"', '"14956"') for l in lines[2:]]
    p = tmp_path / "t.csv"
    p.write_text("\n".join(lines + second))
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "traffic.json"))
    e = bench.record_traffic(str(p), "w", "kda_bt16_kernel", "ncu ...")
    assert e["launches"] == 2
    assert e["dram_read"] == 33569796 and e["dram_write"] == 80000
    assert abs(e["ncu_us_per_launch"] - 14.95) < 1e-9
    assert abs(e["physical_gbs"] - (33569796 + 80000) / 14950) < 1e-6


def test_record_traffic_needs_a_launch(tmp_path):
    p = tmp_path / "t.csv"
    p.write_text(CSV.splitlines()[0] + "\n" + CSV.splitlines()[1] + "\n")
    with pytest.raises(ValueError):
        bench.record_traffic(str(p), "w", "kda_bt16_kernel", "")


def test_kernel_families_hash_their_own_sources():
    a = bench.kernel_source_hash("kda_tril_kernel<MODE_FUSED>")
    b = bench.kernel_source_hash("kda_bt16_kernel")
    c = bench.kernel_source_hash("kda_kgb_kernel")
    assert len({a, b, c}) == 3
    assert bench.kernel_source_hash("kda_bt32_kernel") == b


def test_source_hash_ignores_comments_only():
    a = "int f(int x) {  // add one\n    return x + 1; /* done */\n}\n"
    b = "int f(int x) {\n    /* a different note */ return x + 1;\n}  // end\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_smi_timestamps_keep_their_milliseconds():
    import time
    base = time.mktime(time.strptime("2026/12/03 09:40:26", "%Y/%m/%d %H:%M:%S"))
    assert bench.parse_smi_time("2026/12/03 09:40:26.250") == pytest.approx(base + 0.25)
    assert bench.parse_smi_time("2026/12/03 09:40:26") == base


def _sampler_with(tmp_path, rows):
    s = bench.ClockSampler(0)
    s.proc = object()                       # as if nvidia-smi had run
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        for ts, mhz, reason in rows:
            f.write(f"{ts}, {mhz}, 2070, 500.0, 0x0, {reason}, Not Active, Not Active, Not Active\n")
    return s


def test_clock_summary_uses_the_timed_region(tmp_path):
    import time
    t = lambda s: time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(1.8e9)) + s
    t0 = bench.parse_smi_time(t(".100"))
    rows = [(t(".000"), 1000, "Not Active"), (t(".150"), 2070, "Not Active"), (t(".200"), 2070, "Not Active"),
            (t(".250"), 2060, "Not Active"), (t(".900"), 500, "Active")]
    got = _sampler_with(tmp_path, rows).summary(t0, t0 + 0.2)
    # only the three samples inside [0.1, 0.3] count: the idle one before and the
    # slowed one after the timed region do not
    assert got["samples"] == 3 and got["window"] == "timed region"
    assert got["sm_mhz"] == 2070 and got["reasons"] == []


def test_clock_summary_widens_a_short_window(tmp_path):
    import time
    t = lambda s: time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(1.8e9)) + s
    t0 = bench.parse_smi_time(t(".500"))
    rows = [(t(".300"), 2070, "Not Active"), (t(".900"), 2070, "Active")]
    got = _sampler_with(tmp_path, rows).summary(t0, t0 + 0.01)
    assert got["window"] == "timed region +- 0.25 s" and got["samples"] == 1
    assert got["reasons"] == []
