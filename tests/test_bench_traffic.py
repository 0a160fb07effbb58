"""bench.py's DRAM-traffic record: the per-call bytes are read from an ncu
CSV log (per launch, read + write, units converted, median over launches,
summed over the kernels of one call) and kept with the kernel sources' hash;
a stale hash gives no traffic figure."""
import json

import bench

CSV = '''==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void ssu::ssu_verify_fold_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","10.00"
"0","1","python","h","void ssu::ssu_verify_fold_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","2.50"
"1","1","python","h","void ssu::ssu_verify_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","1.20"
"1","1","python","h","void ssu::ssu_verify_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","100.00"
"1","1","python","h","void ssu::ssu_verify_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","700.00"
"2","1","python","h","void ssu::ssu_verify_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","1.30"
"2","1","python","h","void ssu::ssu_verify_kernel<float, 32>(ssu::KParams, int)","1","7","(256, 1, 1)","(256, 128, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","100.00"
"3","1","python","h","void at::native::vectorized_elementwise_kernel<4>(int)","1","7","(128, 1, 1)","(8, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","99.00"
'''


def test_traffic_from_csv(tmp_path):
    p = tmp_path / "v.csv"
    p.write_text(CSV)
    rec = bench.traffic_from_ncu_csv(str(p), "verify")
    assert rec["kernels"]["ssu_verify_fold_kernel"] == {"launches": 1, "median_bytes": 12.5e6}
    assert rec["kernels"]["ssu_verify_kernel"]["launches"] == 2
    assert rec["kernels"]["ssu_verify_kernel"]["median_bytes"] == 1.35e9
    assert rec["bytes_per_call"] == int(12.5e6 + 1.35e9)


def test_record_and_lookup(tmp_path, monkeypatch):
    p = tmp_path / "v.csv"
    p.write_text(CSV)
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    bench.record_traffic(str(p), "verify_b256_t4_fp32", "ncu ...")
    assert bench.profiled_traffic("verify", "verify_b256_t4_fp32") == int(12.5e6 + 1.35e9)
    # a run at another batch is not the recorded workload
    assert bench.profiled_traffic("verify", "verify_b256_t4_fp32", batch=32) is None
    rec = json.loads(out.read_text())
    rec["verify/verify_b256_t4_fp32"]["kernel_source_sha256_16"] = "0" * 16
    out.write_text(json.dumps(rec))
    assert bench.profiled_traffic("verify", "verify_b256_t4_fp32") is None
