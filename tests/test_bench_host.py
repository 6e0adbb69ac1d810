"""Host logic of bench.py that needs no GPU: the clock record, the code
fingerprint that keys recorded ncu traffic, and the workload config both arms
print."""
import bench


class _DoneProcess:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with_rows(tmp_path, rows):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = _DoneProcess()
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    return s


def test_clock_record_takes_the_median_and_every_active_reason(tmp_path):
    rows = [
        "0, 2070 MHz, 2070 MHz, 900.1 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980 MHz, 2070 MHz, 1350.0 W, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2025 MHz, 2070 MHz, 1200.0 W, 0x0, Not Active, Active, Not Active, Not Active",
        "garbage line",
    ]
    clk = _sampler_with_rows(tmp_path, rows).stop()
    assert clk["samples"] == 3
    assert clk["sm_mhz"] == 2025.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_record_without_nvidia_smi():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_fingerprint_ignores_comments_and_whitespace_only():
    code = b"int f(int x) {\n  return x + 1;  // add one\n}\n/* block\n comment */\n"
    same = b"int f(int x) { return x + 1; }  /* other words */"
    changed = b"int f(int x) { return x + 2; }"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(changed)


def test_kernel_fingerprints_are_per_kernel():
    a, b, all_ = (bench.kernel_fingerprint("chunk_local"), bench.kernel_fingerprint("chunk_recur"),
                  bench.kernel_fingerprint())
    assert len({a, b, all_}) == 3 and all(len(x) == 16 for x in (a, b, all_))


def test_both_arms_name_one_workload_config():
    c1, c2 = bench.prefill_config(1), bench.prefill_config(2)
    assert c1["workload"] == c2["workload"]
    assert c1["parallelism"] == "replicas x1" and c2["parallelism"] == "replicas x2"
    assert "4 sequences x 8192 tokens, H=32" in c1["workload"]
    assert "larger than L2" in c1["l2"]
