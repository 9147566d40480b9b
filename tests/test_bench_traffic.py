"""The bench's roofline traffic on CPU: DRAM bytes per launch come from the
committed traffic file only while its digest matches the kernel sources, so
a capture taken on other kernels is reported as null, never as the current
kernels' traffic."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(path, digest, lines):
    with open(path, "w") as f:
        f.write("# a comment line\n")
        f.write(f"kernel_sources_sha256: {digest}\n")
        for line in lines:
            f.write(line + "\n")


def test_matching_digest_gives_the_values(tmp_path, monkeypatch):
    p = tmp_path / "traffic.txt"
    _write(p, bench.kernel_digest(), ["wl_a kernel_x 123", "wl_a kernel_y 45",
                                      "wl_b kernel_x 7"])
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    got, why = bench.read_traffic("wl_a")
    assert got == {"kernel_x": 123, "kernel_y": 45}
    assert why == "ncu capture of the current kernels"
    assert bench.read_traffic("wl_c")[0] == {}


def test_stale_digest_gives_nothing(tmp_path, monkeypatch):
    p = tmp_path / "traffic.txt"
    stale = ("0" if bench.kernel_digest()[0] != "0" else "1") + \
        bench.kernel_digest()[1:]
    _write(p, stale, ["wl_a kernel_x 123"])
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(p))
    assert bench.read_traffic("wl_a") == ({}, "kernels changed since the "
                                                "capture")


def test_missing_file_gives_nothing(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.txt"))
    assert bench.read_traffic("wl_a") == ({}, "no capture")


def test_digest_covers_every_kernel_source(tmp_path, monkeypatch):
    """Changing any one of the digested sources changes the digest."""
    import shutil
    src = os.path.join(ROOT, "kv_cache_transform_gb300", "csrc")
    fake = tmp_path / "kv_cache_transform_gb300" / "csrc"
    fake.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), fake / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_digest()
    assert base == bench.kernel_digest()
    for name in bench.KERNEL_SOURCES:
        with open(fake / name, "ab") as f:
            f.write(b"\n")
        assert bench.kernel_digest() != base
        base = bench.kernel_digest()
