"""Host logic of bench.py that needs no GPU: the recorded DRAM traffic of the
dominant kernel is reported only while the kernel sources it was captured on
are unchanged (otherwise the roofline's traffic is null)."""
import os
import shutil

import bench

KERNEL_FILES = ("kq_umma.cu", "kq_device.cuh", "kq_internal.h", "kq_records.h", "kq_api.cu")


def _tree(tmp_path):
    """A copy of the kernel sources and the build script bench.py hashes,
    under a scratch root."""
    pkg = os.path.join(bench.ROOT, "w4a4_mxfp4_activation_gb300")
    dst = tmp_path / "w4a4_mxfp4_activation_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in KERNEL_FILES:
        shutil.copy(os.path.join(pkg, "csrc", f), dst / f)
    shutil.copy(os.path.join(pkg, "build.py"), dst.parent / "build.py")
    (tmp_path / "profiles").mkdir()
    return dst


def test_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    assert len(h) == 16
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# comment line\n"
        f"flux_ffn_down_umma    {h}  dram_bytes     122196480   115631616   6564864\n"
        "flux_ffn_down_dual    0000000000000000  dram_bytes     1   1   0\n")
    assert bench.recorded_traffic("flux_ffn_down_umma") == 122196480.0
    assert bench.recorded_traffic("flux_ffn_down_dual") is None      # other sources
    assert bench.recorded_traffic("flux_3072_umma") is None          # no such line
    # any edit of a hashed source makes the record stale
    with open(csrc / "kq_umma.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.kernel_source_hash() != h
    assert bench.recorded_traffic("flux_ffn_down_umma") is None


def test_traffic_follows_the_launcher_and_the_compile_command(tmp_path, monkeypatch):
    """The tensor maps and the dispatch live in kq_api.cu and the nvcc flags in
    build.py: an edit of either also makes the traffic record stale."""
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for path in (csrc / "kq_api.cu", csrc.parent / "build.py"):
        h = bench.kernel_source_hash()
        (tmp_path / "profiles" / "traffic.txt").write_text(
            f"flux_ffn_down_umma    {h}  dram_bytes     122196480   115631616   6564864\n")
        assert bench.recorded_traffic("flux_ffn_down_umma") == 122196480.0
        with open(path, "a") as f:
            f.write("\n# edited\n")
        assert bench.recorded_traffic("flux_ffn_down_umma") is None


def test_round_structure_does_not_depend_on_steps():
    """The timed region runs rounds of min(steps left, 32) launches per layer
    graph, so 20 steps time one 20-launch graph per layer, not 20 one-launch
    graphs, and every step count is covered exactly."""
    assert bench.round_lengths(20) == [20]
    assert bench.round_lengths(32) == [32]
    assert bench.round_lengths(70) == [32, 32, 6]
    assert bench.round_lengths(0) == []
    for k in (1, 5, 31, 33, 40000):
        r = bench.round_lengths(k)
        assert sum(r) == k and all(0 < n <= 32 for n in r) and r[:-1] == [32] * (len(r) - 1)


def test_missing_traffic_file_reads_as_null(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("flux_ffn_down_umma") is None


def test_algorithmic_bytes_per_element():
    """2 B read + 1/2 B of codes + 1/32 B of scales per element (the metric's
    byte count); the dual output adds 2 B of bf16."""
    assert bench.algo_bytes(4608, 12288) == 4608 * 12288 * 2.53125
    assert bench.algo_bytes_dual(4608, 12288) == 4608 * 12288 * 4.53125
