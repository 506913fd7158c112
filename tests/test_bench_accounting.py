"""The bench's algorithmic byte counts (the roofline's numerator), against
hand counts: K and V bytes of the attended tokens (+ fp32 scales for INT8 and
INT4), 4 bytes per block-table entry read, 4 per context length, and q plus
out. Shared blocks count once; under a window only the window counts."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from workloads import Geometry, make_workload  # noqa: E402


def test_bf16_two_sequences():
    w = make_workload("acc", Geometry(n_h=4, n_kv=2, d_h=64), [5, 37], seed=1)
    per_token = 2 * 2 * 64 * 2            # K and V, 2 kv heads, 64 dims, bf16
    tables = 4 * (1 + 3)                  # ceil(5/16) + ceil(37/16) entries
    q_out = 2 * 2 * 4 * 64 * 2            # q and out, 2 sequences, 4 heads, bf16
    d = bench.decode_bytes(w)
    assert d["bytes"] == 42 * per_token + tables + 4 * 2 + q_out == 23576
    assert d["flops"] == 4 * 4 * 64 * 42


def test_quantised_pools_add_scales():
    for dt, code_bytes in (("int8", 64), ("int4", 32)):
        w = make_workload("acc8", Geometry(n_h=4, n_kv=2, d_h=64, kv_dtype=dt), [5, 37], seed=1)
        per_token = 2 * 2 * code_bytes + 2 * 2 * 4   # codes + one fp32 scale per row
        assert bench.decode_bytes(w)["bytes"] == 42 * per_token + 16 + 8 + 2048


def test_shared_prefix_counts_once():
    # two sequences sharing 32 tokens (2 full blocks) of prefix
    w = make_workload("accs", Geometry(n_h=4, n_kv=2, d_h=64), [40, 50], seed=2,
                      prefix_len=[32, 32], group=[0, 0])
    d = bench.decode_bytes(w)
    per_token = 512
    other = 4 * (3 + 4) + 8 + 2048
    assert d["logical_bytes"] == 90 * per_token + other
    assert d["bytes"] == (90 - 32) * per_token + other


def test_window_counts_only_the_window():
    w = make_workload("accw", Geometry(n_h=4, n_kv=2, d_h=64), [100, 20], seed=3, window=40)
    # sequence 0 attends [60, 100): blocks 3..6; sequence 1 attends [0, 20): blocks 0..1
    d = bench.decode_bytes(w)
    assert d["bytes"] == (40 + 20) * 512 + 4 * (4 + 2) + 8 + 2048


def test_oracle_on_all_cores_runs_the_sample():
    # the CPU baseline's all-cores leg: (sequence, kv head) units of the
    # sample dealt to spawned processes, timed by wall clock
    w = bench.named_workload("tiny")
    pool = bench.OracleCores(w, [0, 1])
    try:
        assert 1 <= pool.cores <= 2 * w.geom.n_kv
        assert pool.run() > 0 and pool.run() > 0
    finally:
        pool.close()


def test_probe_bytes_count_every_block():
    w = make_workload("probe", Geometry(n_h=4, n_kv=2, d_h=64, kv_dtype="int8"), [5, 37], seed=1)
    blocks = 1 + 3
    assert bench.probe_bytes(w) == blocks * 2 * (2 * 16 * 64 + 2 * 16 * 4) + 4 * blocks
