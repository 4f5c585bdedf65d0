"""bench.py's bookkeeping on the CPU: the device-code digest that keys the
recorded ncu traffic, and the kernel each bench call is reported under."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_drops_comments_and_spacing():
    a = "int f(int x) { // one\n  return x + 1; /* two\n three */ }\n"
    b = "int f(int x)\n{\n    return x + 1;\n}  // other words\n"
    assert bench.code_only(a) == bench.code_only(b) == "int f(int x) { return x + 1; }"
    assert bench.code_only("return x + 2;") != bench.code_only("return x + 1;")


def test_digest_follows_code_not_comments():
    names = bench.KERNEL_SOURCES["w4a16_tc_kernel"]
    csrc = os.path.join(ROOT, "speculative_verify_gb300", "csrc")
    text = {n: open(os.path.join(csrc, n)).read() for n in names}
    base = bench.kernel_source_digest("w4a16_tc_kernel", lambda n: text[n])
    assert base == bench.kernel_source_digest("w4a16_tc_kernel")
    commented = dict(text)
    commented[names[2]] = "// a new comment line\n" + text[names[2]]
    assert bench.kernel_source_digest("w4a16_tc_kernel", lambda n: commented[n]) == base
    changed = dict(text)
    changed[names[2]] = text[names[2]] + "\nstatic int sv_extra_symbol;\n"
    assert bench.kernel_source_digest("w4a16_tc_kernel", lambda n: changed[n]) != base
    # a kernel's digest covers only its own sources
    assert bench.kernel_source_digest("w4a16_stream_kernel", lambda n: changed[n] if n in changed else text[n]) == \
        bench.kernel_source_digest("w4a16_stream_kernel")


def test_traffic_lookup_needs_the_current_digest(tmp_path, monkeypatch):
    d = tmp_path / "profiles"
    d.mkdir()
    cur = bench.kernel_source_digest("w4a16_tc_kernel")
    (d / "traffic.txt").write_text("# comment\nlmhead_verify_4x8_T32 %s 123   # x\n"
                                   "lmhead_verify_4x8_T32 0000000000000000 456\n" % cur)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc_src = os.path.join(ROOT, "speculative_verify_gb300")
    os.symlink(csrc_src, tmp_path / "speculative_verify_gb300")
    assert bench.recorded_traffic("lmhead_verify_4x8_T32", "w4a16_tc_kernel") == 123
    assert bench.recorded_traffic("lmhead_verify_4x8_T32", "w4a16_stream_kernel") is None
    assert bench.recorded_traffic("gemm_qkv_T1", "w4a16_tc_kernel") is None


@pytest.mark.parametrize("T,kind,vm,kernel", [
    (1, "gemm", None, "w4a16_stream_kernel"),
    (8, "head", None, "w4a16_stream_kernel"),
    (16, "head", None, "w4a16_wide_kernel"),
    (16, "gemm", None, "w4a16_stream_kernel"),
    (16, "head", object(), "w4a16_stream_kernel"),
    (32, "head", None, "w4a16_tc_kernel"),
    (32, "gemm", None, "w4a16_tc_kernel"),
])
def test_kernel_of_follows_the_dispatch_rule(T, kind, vm, kernel):
    assert bench.kernel_of({"T": T, "kind": kind, "vm": vm}) == kernel


def test_committed_traffic_rows_are_well_formed():
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        assert len(parts) >= 3 and len(parts[1]) == 16 and int(parts[2]) > 0, line
