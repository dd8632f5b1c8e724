"""Host-side logic of bench.py that needs no GPU: the committed DRAM traffic
is reported only for the kernel source and workload it was captured on, and
each workload's FLOP count is the contraction it times."""
import json
import os

import bench


def test_traffic_only_for_its_source_and_workload():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, e in d.items():
        if kernel.startswith("_"):
            continue
        wl, h, v = e["bench_workload"], e["source_hash"], e["dram_bytes_per_launch"]
        assert bench.ncu_traffic(kernel, h, wl) == v
        others = [w for w in bench.WORKLOADS if w != wl]
        assert all(bench.ncu_traffic(kernel, h, w) is None for w in others)
        assert bench.ncu_traffic(kernel, "0" * 16, wl) is None
    assert bench.ncu_traffic("no_such_kernel", "0" * 16, "llama8b") is None


def test_flop_counts():
    w = bench.WORKLOADS
    assert bench._flops("llama8b") == 2.0 * 8192 * 14336 * 4096
    assert bench._flops("moe") == 2.0 * 64 * 512 * 1536 * 4096
    assert bench._flops("w4a16") == 2.0 * w["w4a16"]["L"] * w["w4a16"]["M"] * 14336 * 4096


def test_every_workload_has_a_sample_and_a_description():
    for name, c in bench.WORKLOADS.items():
        assert c["desc"]
        assert name in bench._CPU_SAMPLE and name in bench._REF_SAMPLE
        assert bench._sample_desc(name, *bench._CPU_SAMPLE[name])
