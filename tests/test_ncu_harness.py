"""CPU tests of the ncu evidence harness's summarising half, on small ncu
`--csv` logs written here (same columns as ncu's metrics logs)."""
import pytest

from self_attention_backward_gb300 import ncu_harness as H

HDR = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
       '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"')


def _row(lid, kernel, metric, unit, value):
    return (f'"{lid}","1","python3","127.0.0.1","{kernel}","1","7","(448, 1, 1)","(800, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"')


MAIN = "void psa::<unnamed>::bwd_main_kernel<32>(CUtensorMap_st, CUtensorMap_st, const float *, int)"
PRE = "void unnamed>::pre_kernel<32>(const __nv_bfloat16 *, float *, long long)"
FILL = "void at::native::vectorized_elementwise_kernel<4, at::native::FillFunctor<unsigned char>>(int, T2)"


def _write(tmp_path, rows, name="log.csv"):
    p = tmp_path / name
    p.write_text("==PROF== Connected to process 1\n" + HDR + "\n" + "\n".join(rows) + "\n")
    return str(p)


def test_short_names():
    assert H.short_name(MAIN) == "bwd_main_kernel<32>"
    assert H.short_name(PRE) == "pre_kernel<32>"
    assert H.short_name(FILL) == "vectorized_elementwise_kernel<4, at::native::FillFunctor<unsigned char>>"
    assert H.short_name("void (anonymous namespace)::dq_kernel<64>(int)") == "dq_kernel<64>"


def test_launch_list_shares(tmp_path):
    rows = [_row(0, MAIN, "gpu__time_duration.sum", "usecond", "600"),
            _row(1, PRE, "gpu__time_duration.sum", "ns", "7,500"),
            _row(2, MAIN, "gpu__time_duration.sum", "msecond", "0.6"),
            _row(3, FILL, "gpu__time_duration.sum", "usecond", "92.5")]
    table, total = H.summarize_launches(H.read_metric_rows(_write(tmp_path, rows)))
    assert total == pytest.approx(1300.0)
    assert table[0][:3] == ("bwd_main_kernel<32>", 2, pytest.approx(1200.0))
    assert sum(r[3] for r in table) == pytest.approx(100.0)
    assert dict((r[0], r[4]) for r in table)["pre_kernel<32>"] == pytest.approx(7.5)
    md = H.launches_markdown(table, total)
    assert "| bwd_main_kernel<32> | 2 | 1200.0 | 92.3 % | 600.0 |" in md


def test_kernel_bandwidth_and_tensor_pipe(tmp_path):
    rows = [_row(0, MAIN, "gpu__time_duration.sum", "usecond", "500"),
            _row(0, MAIN, "dram__bytes_read.sum", "Mbyte", "50"),
            _row(0, MAIN, "dram__bytes_write.sum", "byte", "1000000"),
            _row(0, MAIN, "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", "%", "22.5"),
            _row(1, PRE, "gpu__time_duration.sum", "usecond", "10"),
            _row(1, PRE, "dram__bytes_read.sum", "Kbyte", "40000"),
            _row(1, PRE, "dram__bytes_write.sum", "Mbyte", "0.4")]
    items = H.summarize_kernels(H.read_metric_rows(_write(tmp_path, rows)), hbm_gbs=6000.0)
    main, pre = items
    assert main["kernel"] == "bwd_main_kernel<32>"
    assert main["gbs"] == pytest.approx(51e6 / 500e-6 / 1e9)          # 102 GB/s
    assert main["tensor_pct"] == pytest.approx(22.5)
    assert pre["gbs"] == pytest.approx(40.4e6 / 10e-6 / 1e9)          # 4040 GB/s
    assert pre["hbm_frac"] == pytest.approx(4040.0 / 6000.0)
    assert pre["tensor_pct"] is None
    md = H.kernels_markdown(items, 6000.0)
    assert "| 1 | pre_kernel<32> | 10.0 | 40.00 | 0.40 | 4040 | 67.3 % | n/a |" in md


def test_measured_peak_is_read():
    assert H.measured_hbm_gbs() > 1000.0


def test_record_traffic(tmp_path):
    import json
    items = [{"kernel": "bwd_main_kernel<32>", "dram_read": 5e7, "dram_write": 1e6},
             {"kernel": "pre_kernel<32>", "dram_read": 2e7, "dram_write": 0.0},
             {"kernel": "vectorized_elementwise_kernel<4>", "dram_read": 1.0, "dram_write": 1.0}]
    path = str(tmp_path / "traffic.json")
    H.record_traffic(items, "wl", "tc", path)
    rec = json.load(open(path))["wl"]["tc"]
    assert set(rec) == {"bwd_main", "bwd_pre"}
    assert rec["bwd_main"]["dram_bytes_per_launch"] == 5.1e7
    import importlib.util, os
    spec = importlib.util.spec_from_file_location("bench", os.path.join(H.ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    assert rec["bwd_main"]["source_hash"] == b.source_hash("tc")


def test_kernel_capture_is_one_kernel_one_launch():
    """Every capture that collects more than the duration names one kernel and
    takes one launch, after the warm-up steps, with the clocks left alone."""
    cmd = H.kernel_capture_cmd("bwd_main_kernel", "/tmp/x.csv", ["python", "bench.py"])
    assert cmd[cmd.index("-c") + 1] == "1"
    assert cmd[cmd.index("-s") + 1] == str(H.WARMUP_STEPS)
    assert cmd[cmd.index("--clock-control") + 1] == "none"
    k = cmd[cmd.index("-k") + 1]
    assert k.startswith("regex:") and "|" in k and all(p.lstrip("^").startswith("bwd_main_kernel")
                                                       for p in k[len("regex:"):].split("|"))
    for fam in H.FAMILY_KERNELS.values():
        assert len(set(fam)) == len(fam)
