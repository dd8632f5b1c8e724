"""Host-side logic of bench.py that needs no GPU: the committed DRAM traffic
is reported only for the kernel source and workload it was captured on, and
each workload's FLOP count is the contraction it times."""
import json
import os

import bench


def test_traffic_only_for_its_source_and_workload():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, entries in d.items():
        if kernel.startswith("_"):
            continue
        entries = entries if isinstance(entries, list) else [entries]
        captured = {e["bench_workload"] for e in entries}
        for e in entries:
            wl, h, v = e["bench_workload"], e["source_hash"], e["dram_bytes_per_launch"]
            assert bench.ncu_traffic(kernel, h, wl) == v
            others = [w for w in bench.WORKLOADS if w not in captured]
            assert all(bench.ncu_traffic(kernel, h, w) is None for w in others)
            assert bench.ncu_traffic(kernel, "0" * 16, wl) is None
    assert bench.ncu_traffic("no_such_kernel", "0" * 16, "llama8b") is None


def test_flop_counts():
    w = bench.WORKLOADS
    assert bench._flops("llama8b") == 2.0 * 8192 * 14336 * 4096
    assert bench._flops("moe") == 2.0 * 64 * 512 * 1536 * 4096
    assert bench._flops("w4a16") == 2.0 * w["w4a16"]["L"] * w["w4a16"]["M"] * 14336 * 4096


def test_every_workload_has_an_oracle_sample():
    for name, c in bench.WORKLOADS.items():
        assert c["desc"]
        assert name in bench._ORACLE_SLICES or name in ("moe", "w4a16")


def test_linear_fit_separates_fixed_cost():
    """t(n) = a + b*n from two sizes: the fixed part is recovered, so the
    extrapolation to a large n does not multiply it."""
    a, b = bench._linear_fit(100, 1.0 + 0.01 * 100, 200, 1.0 + 0.01 * 200)
    assert abs(a - 1.0) < 1e-12 and abs(b - 0.01) < 1e-12
    assert bench._linear_fit(10, 2.0, 20, 1.9) == (2.0, 0.0)   # noise never gives a negative slope


def test_oracle_step_pr1_runs_whole_step():
    import oracle
    oracle.build()
    X, W = bench._oracle_inputs("pr1")
    r = bench._oracle_step("pr1", X, W)
    assert r["step_s"] == r["spent_s"] > 0 and "no extrapolation" in r["work"]


def test_operand_copies_exceed_l2():
    for per_set in (1 << 20, 52 * 2**20, 85 * 2**20, 126 * 2**20 - 1):
        n = bench.operand_copies(per_set)
        assert n * per_set > bench.L2_BYTES and (n - 1) * per_set <= bench.L2_BYTES + per_set
    assert bench.operand_copies(bench.L2_BYTES) == 1
    assert bench.operand_copies(500 * 2**20) == 1
