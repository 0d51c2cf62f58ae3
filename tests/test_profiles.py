"""The committed ncu summaries that bench.py reads its roofline traffic from:
each names its full command, a kernel-source hash and a traffic figure per
launch that is the mean of its captured launches, and that figure is the
workload's algorithmic K/V bytes plus a small excess (the page table, q,
partials, outputs and the ragged tail of the last box), never less: a figure
below the algorithmic bytes, or far above them, would mean a wrong capture or
K/V rows read twice.  (Whether the hash is the current one decides only
whether bench.py reports the figure; that is not asserted here.)"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# algorithmic K/V bytes per step of the workloads (their generators are
# seeded; the figures are what bench.py prints as kv_bytes_per_step)
ALGORITHMIC = {"long": 2147483648, "batched": 1229225984, "many_short": 1077587968}
# allowed excess: the partials and outputs, and for many short sequences the
# 16-token boxes past each length
EXCESS = {"long": 1.01, "batched": 1.02, "many_short": 1.06}


def read(name):
    with open(os.path.join(ROOT, "profiles", name)) as f:
        return f.read()


@pytest.mark.parametrize("workload", sorted(ALGORITHMIC))
def test_traffic_summary_is_consistent(workload):
    text = read(f"split_kernel_{workload}.md")
    assert f"python bench.py --workload {workload}" in text
    assert "ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum" in text
    assert "--clock-control none" in text
    rows = re.findall(r"^\| (\d+) \| (\d+) \| (\d+) \| ([0-9.]+) us \|$", text, re.M)
    assert len(rows) >= 1
    per_launch = [int(r) + int(w) for _, r, w, _ in rows]
    mean = sum(per_launch) // len(per_launch)
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    assert m and int(m.group(1)) == mean
    alg = ALGORITHMIC[workload]
    assert alg <= mean <= EXCESS[workload] * alg, (mean, alg)
    assert re.search(r"kernel_source_sha256:\s*[0-9a-f]{16}", text)


def test_summaries_share_one_kernel_source():
    hashes = set()
    for name in os.listdir(os.path.join(ROOT, "profiles")):
        hashes.update(re.findall(r"kernel_source_sha256[`:\s]+([0-9a-f]{16})", read(name)))
    assert len(hashes) == 1, hashes


@pytest.mark.parametrize("workload", sorted(ALGORITHMIC))
def test_traffic_applies_only_to_the_captured_kernel(workload):
    """bench.py reports a summary's traffic only for runs of the kernel the
    summary captured (and only with the default options, for which the
    caller passes that kernel's name)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    kernel = re.search(r"^kernel:\s*(\S+)$", read(f"split_kernel_{workload}.md"), re.M)
    assert kernel and kernel.group(1).startswith("split_")
    assert bench.recorded_traffic(workload, "split_simt_kernel_other") is None
    assert bench.recorded_traffic(workload, None) is None
    got = bench.recorded_traffic(workload, kernel.group(1))
    if got is not None:  # the summary was taken on the current kernel sources
        m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", read(f"split_kernel_{workload}.md"))
        assert got == float(m.group(1))


def test_kernel_names_follow_the_plan():
    """The kernel bench.py names for a plan: the one the launcher picks
    (cluster, shallow ring, single pass, or the split kernel)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from types import SimpleNamespace as P
    assert bench.split_kernel_name(P(variant=2, cluster=8, ring_stages=3, split=1), 128) == \
        "split_mma_kernel_cluster"
    assert bench.split_kernel_name(P(variant=2, cluster=0, ring_stages=2, split=0), 128) == \
        "split_mma_kernel_shallow"
    assert bench.split_kernel_name(P(variant=2, cluster=0, ring_stages=3, split=0), 128) == \
        "split_mma_kernel_single"
    assert bench.split_kernel_name(P(variant=2, cluster=0, ring_stages=6, split=1), 64) == \
        "split_mma_kernel"
    assert bench.split_kernel_name(P(variant=1, cluster=0, ring_stages=3, split=1), 128) == \
        "split_simt_kernel"
