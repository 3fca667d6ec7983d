"""Host-side figures the bench reports, checked on small hand-made cases."""

import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step  # noqa: E402


@pytest.mark.parametrize("B", [8, 16, 32])
def test_block_tradeoff_counts_last_block_waste(B):
    # contexts 1, B, B + 1 and 3B: last blocks hold 1, B, 1 and B tokens
    lens = [1, B, B + 1, 3 * B]
    step = make_step([RequestSpec(L - 1, 1) for L in lens], num_q_heads=4, num_kv_heads=2,
                     head_dim=64, block_size=B, seed=1, materialize=False)
    t = bench.block_tradeoff(step)
    blocks = 1 + 1 + 2 + 3
    assert t["table_entries_read"] == blocks
    assert t["blocks_in_use"] == blocks
    assert t["slots_allocated"] == blocks * B
    wasted = (B - 1) + 0 + (B - 1) + 0
    assert t["slots_wasted_frac"] == pytest.approx(wasted / (blocks * B))


def test_block_tradeoff_counts_a_shared_block_once():
    # two requests over one shared 32-token prefix (2 blocks of 16), each
    # with 5 private tokens in a block of its own
    specs = [RequestSpec(36, 1, shares_prefix=True), RequestSpec(36, 1, shares_prefix=True)]
    step = make_step(specs, num_q_heads=4, num_kv_heads=2, head_dim=64, prefix_tokens=32,
                     seed=2, materialize=False)
    t = bench.block_tradeoff(step)
    assert t["table_entries_read"] == 2 * 3
    assert t["blocks_in_use"] == 2 + 2
    assert t["slots_allocated"] == 4 * 16
    assert t["slots_wasted_frac"] == pytest.approx(2 * 11 / 64)


def test_step_work_bytes_do_not_depend_on_block_size():
    works = []
    for B in (8, 16, 32):
        step = make_step([RequestSpec(99, 1), RequestSpec(20, 30)], num_q_heads=8,
                         num_kv_heads=2, head_dim=128, block_size=B, seed=3, materialize=False)
        w = bench.step_work(step)
        w.pop("touched_bytes")  # allocated slots: the one figure that depends on B
        works.append(w)
    assert works[0] == works[1] == works[2]
    assert works[0]["decode_kv_bytes"] == 100 * 2 * 128 * 2 * 2
    assert works[0]["prefill_flops"] == 4 * 128 * 8 * (30 * 20 + 30 * 31 // 2)


def test_decode_bytes_count_a_shared_block_once():
    # two decodes over one shared 32-token prefix (2 blocks of 16), each with
    # 5 private tokens in a block of its own: 32 + 2 * 5 unique tokens
    specs = [RequestSpec(36, 1, shares_prefix=True), RequestSpec(36, 1, shares_prefix=True)]
    step = make_step(specs, num_q_heads=4, num_kv_heads=2, head_dim=64, prefix_tokens=32,
                     seed=2, materialize=False)
    w = bench.step_work(step)
    row = 2 * 64 * 2 * 2
    assert w["decode_kv_bytes"] == (32 + 2 * 5) * row
    assert w["decode_kv_logical_bytes"] == 2 * 37 * row


def test_decode_bytes_without_sharing_equal_the_logical_bytes():
    specs = [RequestSpec(L - 1, 1) for L in (1, 15, 16, 17, 100)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=128, seed=4,
                     materialize=False)
    w = bench.step_work(step)
    assert w["decode_kv_bytes"] == w["decode_kv_logical_bytes"] == (1 + 15 + 16 + 17 + 100) * 2 * 128 * 4


def test_code_hash_ignores_comments_but_not_code():
    src = "int f(int x) {  // add one\n  /* the\n  sum */ return x + 1;\n}\n"
    same = "// a new note\nint f(int x) {\n\n   return x + 1;   \n}\n"
    other = "int f(int x) {\n  return x + 2;\n}\n"
    assert bench.code_sha256(src) == bench.code_sha256(same.replace("   return", "  return"))
    assert bench.code_sha256(src) != bench.code_sha256(other)


def test_committed_decode_traffic_matches_the_current_code():
    """The committed DRAM-traffic summary was taken on the decode kernel's
    current code (else the bench reports no traffic)."""
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "paged_kv_cache_hkv_gb300", "csrc", "decode.cu")
    assert bench.traffic_from_profile(src) is not None


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args):
    import subprocess
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=600, cwd=ROOT)


def test_reference_arm_prints_one_json_line_with_the_contract_keys():
    r = _bench("--impl", "reference", "--workload", "tiny_decode", "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    import json
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["value"] > 0 and d["config"]["workload"] == "tiny_decode"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_native_arm_refuses_to_run_without_a_gpu():
    pytest.importorskip("torch")
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = _bench("--workload", "tiny_decode", "--steps", "3", "--warmup", "3")
    assert r.returncode != 0
    assert "no CUDA device" in (r.stderr + r.stdout)


@pytest.mark.parametrize("clocks,rejected", [
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, False),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, False),
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"]}, True),
    ({"sm_mhz": 1500.0, "sm_max_mhz": 2070.0, "reasons": ["hw_thermal_slowdown"]}, True),
    ({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["sw_thermal_slowdown"]}, True),
    ({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []}, True),  # a leftover clock lock
    ({"sm_mhz": 1950.0, "sm_max_mhz": 2070.0, "reasons": []}, False),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}, False),
])
def test_clock_rejection_rule(clocks, rejected):
    assert bench.clocks_rejected(clocks) == rejected


@pytest.mark.parametrize("workers", [1, 3, 16])
def test_oracle_plan_takes_every_row_of_the_mixed_step_once(workers):
    specs = __import__("paged_kv_cache_hkv_gb300.synth", fromlist=["x"]).mixed_step_specs(3)
    plan = bench.oracle_plan(specs, 3, bench.ORACLE_ROW_CAP, workers)
    seen = set()
    for key, (per, total, taken) in plan.items():
        assert total == taken  # the mixed step is timed whole
        assert len(per) == workers
        rows = [r for w in per for r in w]
        assert len(rows) == len(set(rows)) == total
        assert all(bench.request_class(specs[i]) == key for i, _ in rows)
        seen.update(rows)
    assert len(seen) == sum(s.query_len for s in specs)


def test_oracle_plan_samples_a_class_beyond_its_cap():
    specs = [RequestSpec(6144, 2048) for _ in range(4)]
    plan = bench.oracle_plan(specs, 6, {"decode": 8, "chunk": 100, "prefill": 8}, 4)
    per, total, taken = plan["chunk"]
    assert (total, taken) == (8192, 100)
    rows = [r for w in per for r in w]
    assert len(set(rows)) == 100 and max(len(w) for w in per) - min(len(w) for w in per) <= 1
