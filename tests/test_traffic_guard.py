"""The bench reports a kernel's recorded DRAM traffic only while the sources
it was captured from are unchanged (a hash of them, profiles/traffic.json).
That guard is only as good as its file list: every file a kernel's source
includes, directly or through another header, must be hashed."""
import os
import re

import bench

CSRC = os.path.join(bench.ROOT, "bwd_tcgen05_tma_gb300", "csrc")
INCLUDE = re.compile(r'^\s*#\s*include\s+"([^"]+)"', re.M)


def local_includes(name, seen=None):
    seen = set() if seen is None else seen
    path = os.path.normpath(os.path.join(CSRC, name))
    if path in seen or not os.path.exists(path):
        return seen
    seen.add(path)
    with open(path) as f:
        for inc in INCLUDE.findall(f.read()):
            local_includes(os.path.relpath(os.path.join(os.path.dirname(path), inc), CSRC), seen)
    return seen


def test_every_included_kernel_file_is_hashed():
    for kernel, sources in bench.KERNEL_SOURCES.items():
        hashed = {os.path.normpath(os.path.join(CSRC, n)) for n in sources + bench.COMMON_SOURCES}
        closure = set()
        for s in sources:
            closure |= local_includes(s)
        missing = sorted(os.path.relpath(p, CSRC) for p in closure - hashed)
        assert not missing, f"{kernel}: {missing} change the kernel but not its traffic hash"


def test_traffic_records_name_known_kernels():
    import json

    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for workload, kernels in rec.items():
        for k, r in kernels.items():
            assert k in bench.KERNEL_SOURCES, (workload, k)
            assert r["bytes_per_launch"] > 0 and len(r["source_hash"]) == 16
