"""The committed traffic summaries under profiles/ describe the kernels as they
are: each one names the source files holding its kernel's code and their hash,
which must match the tree (a changed kernel needs a new capture, not a new
hash), and the benchmark's default workload has a current one for its
dominant kernel (the roofline "traffic" field)."""
import glob
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def summaries():
    out = []
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt"))):
        vals = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals.setdefault(k.strip(), v.strip())
        if "source_sha256" in vals:
            out.append((os.path.basename(path), vals))
    return out


def test_every_traffic_summary_matches_its_sources():
    found = summaries()
    assert found, "no traffic summary under profiles/"
    for name, vals in found:
        files = vals["source_files"].split()
        assert bench.kernel_source_hash(files) == vals["source_sha256"], (
            f"{name}: the kernel changed since this capture; capture it again")
        read, write = float(vals["dram__bytes_read.sum"]), float(vals["dram__bytes_write.sum"])
        assert float(vals["dram_bytes_per_launch"]) == read + write, name


def test_default_workload_has_current_traffic():
    assert bench.profile_traffic("moe_w13", bench.DEFAULT_WORKLOAD) is not None
