"""Host-side helpers of bench.py (CPU only)."""
import builtins
import io
import os

import bench


def test_gpu_local_cpus_parses_sysfs_lists(monkeypatch):
    """The sysfs local_cpulist format ("0-3,8,10-11") becomes a set, limited to
    the CPUs this process may use; a missing file gives the empty set."""
    allowed = os.sched_getaffinity(0)
    real_open = builtins.open

    def fake_open(path, *a, **k):
        if str(path).endswith("/0000:1a:00.0/local_cpulist"):
            return io.StringIO("0-3,8,10-11\n")
        if str(path).startswith("/sys/bus/pci/devices/"):
            raise OSError("no such device")
        return real_open(path, *a, **k)

    monkeypatch.setattr(builtins, "open", fake_open)
    got = bench.gpu_local_cpus("00000000:1A:00.0")
    assert got == {0, 1, 2, 3, 8, 10, 11} & allowed
    assert bench.gpu_local_cpus("00000000:FF:00.0") == set()


def test_recorded_traffic_records_are_read():
    """Every record of the committed DRAM traffic file names a kernel source that
    exists and a positive byte count; a record whose hash matches the source is
    returned, a stale hash or an unknown kernel gives None."""
    import hashlib
    import json
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.json")
    records = json.load(open(path))["records"]
    assert {r["kernel"] for r in records} >= {"attn_fwd", "attn_bwd"}
    for r in records:
        src = os.path.join(bench.ROOT, "packed_resolution_diffusion_pack_b300", "csrc", r["source"])
        assert os.path.exists(src)
        assert len(r["sha16"]) == 16 and int(r["dram_bytes_per_launch"]) > 0
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", r["summary"]))
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        got = bench._recorded_traffic(r["kernel"])
        assert got == (int(r["dram_bytes_per_launch"]) if sha == r["sha16"] else None)
    assert bench._recorded_traffic("no_such_kernel") is None
