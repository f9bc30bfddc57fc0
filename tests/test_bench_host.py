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


def test_recorded_traffic_lines_are_read():
    """Every traffic line of the committed DRAM summary names a kernel source
    file that exists, and an unknown kernel gives None."""
    path = os.path.join(bench.ROOT, "profiles", "dram_mixed_50k.md")
    lines = [ln.split() for ln in open(path).read().splitlines() if ln.startswith("traffic ")]
    assert {ln[1] for ln in lines} >= {"attn_fwd", "attn_bwd", "attn_fwd_f8"}
    for ln in lines:
        assert os.path.exists(os.path.join(bench.ROOT, "packed_resolution_diffusion_pack_b300",
                                           "csrc", ln[2]))
        assert len(ln[3]) == 16 and int(ln[4]) > 0
    assert bench._recorded_traffic("no_such_kernel") is None
