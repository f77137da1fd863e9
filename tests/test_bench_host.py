"""The benchmark's host-side helpers on CPU: the traffic figures recorded from ncu are used
only while the kernel's code is unchanged (comments aside), the clock record flags the
throttle reasons that void a run, and the audit-mode block count."""
import os

import pytest

import bench


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _sampler_on(path):
    s = bench.ClockSampler(0)
    s.path = str(path)
    s.proc = _FakeProc()
    s.fh = open(os.devnull, "w")
    return s


def test_clock_record_median_and_reasons(tmp_path):
    p = tmp_path / "clocks.csv"
    p.write_text(
        "2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "2055, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active\n"
        "2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "garbage line\n")
    r = _sampler_on(p).stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070
    assert r["power_w_max"] == 1100.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_record_flags_slowdowns(tmp_path):
    p = tmp_path / "clocks.csv"
    p.write_text(
        "1500, 2070, 700.0, 0x8, Active, Not Active, Not Active, Not Active\n"
        "1400, 2070, 700.0, 0x48, Not Active, Active, Active, Not Active\n")
    r = _sampler_on(p).stop()
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert r["sm_mhz"] == 1450


def test_clock_record_without_nvidia_smi():
    s = bench.ClockSampler(0)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_code_only_ignores_comments_and_spacing():
    a = "int f(int x) { // the argument\n  return x + 1; /* one\n more */ }\n"
    b = "int f(int x)\n{\n    return x + 1;\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def _fake_tree(root, kernel_src):
    csrc = root / bench._CSRC
    csrc.mkdir(parents=True)
    (csrc / "k_reduce.cuh").write_text(kernel_src)
    (csrc / "common.cuh").write_text("// shared\nconstexpr int kChunk = 4096;\n")
    (csrc / "kernels.h").write_text("struct ReduceArgs { int n; };\n")
    (root / "profiles").mkdir()


def test_traffic_is_used_only_for_the_profiled_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_tree(tmp_path, "__global__ void k_reduce() { /* v1 */ }\n")
    h = bench.kernel_source_hash("k_reduce")
    (tmp_path / "profiles" / "k_reduce_case.md").write_text(
        "# summary\n\n"
        f"traffic_per_launch: kernel=k_reduce bytes=123456789 source_hash={h}\n"
        "traffic_per_launch: kernel=k_adamw bytes=5 source_hash=0000000000000000\n")
    assert bench.profiled_traffic("k_reduce") == 123456789
    # a comment edit keeps the figure; a code edit drops it
    csrc = tmp_path / bench._CSRC
    (csrc / "k_reduce.cuh").write_text("__global__ void k_reduce() { /* v2, reworded */ }\n")
    assert bench.profiled_traffic("k_reduce") == 123456789
    (csrc / "k_reduce.cuh").write_text("__global__ void k_reduce() { int x = 1; }\n")
    assert bench.profiled_traffic("k_reduce") is None
    # a change to a shared header drops it too
    (csrc / "k_reduce.cuh").write_text("__global__ void k_reduce() { /* v1 */ }\n")
    assert bench.profiled_traffic("k_reduce") == 123456789
    (csrc / "common.cuh").write_text("constexpr int kChunk = 2048;\n")
    assert bench.profiled_traffic("k_reduce") is None


def test_committed_traffic_lines_parse():
    """Every traffic line in profiles/ names a known kernel, a byte count and a 16-digit
    source hash (whether or not it matches the current code)."""
    import re
    pdir = os.path.join(bench.ROOT, "profiles")
    found = 0
    for fn in sorted(os.listdir(pdir)):
        for line in open(os.path.join(pdir, fn)):
            if "traffic_per_launch:" not in line:
                continue
            m = re.match(r"\s*traffic_per_launch:\s*kernel=(\S+)\s+bytes=(\d+)\s+"
                         r"source_hash=([0-9a-f]{16})\s*$", line)
            assert m, line
            assert m.group(1) in bench.KERNEL_SOURCES
            found += 1
    assert found >= 2


@pytest.mark.parametrize("n,blocks", [(0, 1), (1, 4), (32, 4), (33, 7), (4096, 385)])
def test_audit_block_count(n, blocks):
    assert bench.b2_blocks(n) == blocks
