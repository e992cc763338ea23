"""Host logic of the benchmark's accounting: algorithmic bytes, the keys and
source hash under which measured DRAM traffic is stored, unique vs logical
K/V bytes of a prefix-sharing batch."""

import json
import os

import bench
from paged_kv_cache_292_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_code_only_ignores_comments_and_spacing():
    a = "int x = 1;  // count\n/* block\n comment */ float y = x * 2;\n"
    b = "int x = 1;\nfloat y = x * 2; // other words\n"
    c = "int x = 2;\nfloat y = x * 2;\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_kernel_hash_is_of_the_listed_sources():
    h = bench.kernel_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert all(os.path.exists(p) for p in bench.KERNEL_SRCS)


def test_traffic_keys():
    assert bench.traffic_key("llama3_8b") == "llama3_8b"
    assert bench.traffic_key("llama3_8b", "fp8") == "llama3_8b/fp8"
    assert bench.traffic_key("llama3_8b", queries=4) == "llama3_8b/q4"
    assert bench.traffic_key("gqa8_70b", block_size=32) == "gqa8_70b/bs32"
    assert bench.traffic_key("llama3_8b", separate=True) == "llama3_8b/separate"


def test_committed_traffic_records_are_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        t = json.load(f)
    assert "llama3_8b" in t
    for key, rec in t.items():
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"], key
        assert len(rec["kernel_sha"]) == 16, key


def test_step_bytes_count_kv_queries_tables_and_write():
    sp = workloads.spec("llama3_8b", num_seqs=5, ctx_lo=1, ctx_hi=100, max_context=112, pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=False)
    by = bench.step_bytes(w)
    ctx = w.context_lens.numpy()
    # One token's K and V over all KV heads: 2 * 8 * 128 * 2 bytes.
    assert by["kv_logical"] == int(ctx.sum()) * 4096
    assert by["decode"] > by["kv_logical"]
    assert by["step"] == by["decode"] + by["write"]
    # Without a shared prefix every slot read is distinct.
    assert bench.unique_kv_bytes(w, 2) == by["kv_logical"]


def test_unique_bytes_count_a_shared_prefix_once():
    sp = workloads.spec("mixed_prefix", num_seqs=6, ctx_median=40.0, ctx_hi=200, max_context=224, prefix_tokens=64)
    w = workloads.make_workload(sp, prewritten=True)
    by = bench.step_bytes(w)
    sharing = (w.context_lens.numpy() >= 64)[::2].sum()  # even sequences share the 64-token prefix
    assert sharing >= 2
    assert bench.unique_kv_bytes(w, 2) == by["kv_logical"] - (sharing - 1) * 64 * 4096


def test_step_bytes_for_fp8_pools_and_several_queries():
    """Hand count for a tiny batch: contexts 1, 3 and 20 tokens, 2 KV heads of
    64 dims (128 elements per row), 4 query heads, 2 queries per sequence."""
    sp = workloads.spec("llama3_8b", num_seqs=3, num_heads=4, num_kv_heads=2, head_size=64, max_context=32,
                        pool_blocks=0)
    w = workloads.make_workload(sp, prewritten=False, context_lens=[1, 3, 20])
    row = 2 * 64
    tables = 4 * (1 + 1 + 2) + 4 * 3
    # bf16 pools, one query: K+V 24 tokens x 2 rows x 2 B; q and out; 3 new rows read and written.
    by = bench.step_bytes(w)
    assert by["decode"] == 24 * 2 * row * 2 + 2 * 3 * 4 * 64 * 2 + tables
    assert by["write"] == 3 * 2 * row * (2 + 2) + 8 * 3
    # FP8 pools, two queries: one byte per pool element; the first sequence
    # has only one position for its two new tokens (5 new rows in all).
    by = bench.step_bytes(w, queries=2, kv_fp8=True)
    assert by["kv_logical"] == 24 * 2 * row
    assert by["decode"] == 24 * 2 * row + 2 * 3 * 2 * 4 * 64 * 2 + tables
    assert by["write"] == 5 * 2 * row * (2 + 1) + 8 * 3 * 2
    assert by["step"] == by["decode"] + by["write"]


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference times the oracle on the host and prints one
    JSON line with the contract's keys (no GPU needed)."""
    import subprocess
    import sys

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_fp32", "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny_fp32"
