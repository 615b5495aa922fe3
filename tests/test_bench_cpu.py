"""Host-side arithmetic of bench.py (no GPU): the algorithmic FLOP count of
the causal prefill attention against a brute-force count of (query, key)
pairs, the per-kernel source hashes the traffic table is keyed by, and the
reference arm's config."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_prefill_flops_counts_causal_pairs():
    rng = np.random.default_rng(3)
    for _ in range(20):
        B = int(rng.integers(1, 5))
        L = [int(x) for x in rng.integers(1, 300, size=B)]
        n = [int(rng.integers(0, l + 1)) for l in L]
        pairs = 0
        for Lb, nb in zip(L, n):
            for j in range(nb):             # chunk row j is token Lb - nb + j
                t = Lb - nb + j
                pairs += sum(1 for key in range(Lb) if key <= t)
        # q.k and p.v: 2 D FLOP each per pair and head
        assert bench.prefill_flops(L, n, Hq=32, D=128) == pairs * 32 * 128 * 4


def test_prefill_flops_fresh_prompt_closed_form():
    P = 2048
    assert bench.prefill_flops([P], [P]) == 4 * 128 * 32 * P * (P + 1) // 2


def test_traffic_entries_name_a_kernel_with_sources():
    for name, tr in bench.TRAFFIC.items():
        assert len(tr["kernel_sha"]) == 16 and tr["bytes_per_launch"] > 0, name
    for k, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, f)), (k, f)


def test_reference_arm_reports_the_full_workload_config():
    """The reference arm times a few layers of a workload on the host but its
    line carries the workload's own config (the full layer count and the
    bytes of a whole step), the same object the GPU arm prints."""
    import argparse
    from gqa_paged_kv_gb300 import workloads as wl
    spec = wl.custom(3, [40, 17, 300], pool_pages=64, layers=2, shared_pool=False)
    w = wl.build(spec, "cpu")
    args = argparse.Namespace(no_graph=False, no_overlap=False, qkv=False, hidden=0)
    few = bench.workload_config(w, args, 1)
    full = bench.workload_config(w, args, 1, layers=36)
    assert few["layers"] == 2 and full["layers"] == 36
    assert full["kv_bytes_per_step"] == 18 * few["kv_bytes_per_step"]
    assert "36 qdec_step" in full["launch"]
    assert {k for k in few} == {k for k in full}


def test_qkv_sample_bytes_of_every_sequence_is_the_block_bytes():
    from gqa_paged_kv_gb300 import workloads as wl
    spec = wl.custom(3, [40, 17, 300], pool_pages=64, layers=1)
    w = wl.build(spec, "cpu")
    assert (bench.qkv_sample_bytes(w, 256, w.seq_lens_host)
            == bench.block_bytes_per_layer(w, 256))


def test_oracle_samples_of_the_qkv_block_and_prefill_run():
    """The host oracle samples behind cpu_baseline and the reference arm of
    --qkv and --prefill run on small inputs and report positive rates."""
    from gqa_paged_kv_gb300 import workloads as wl
    spec = wl.custom(2, [40, 17], pool_pages=16, layers=2)
    w = wl.build(spec, "cpu")
    gbs, n, secs = bench.oracle_qkv_sample(w, 128, 0.0)
    assert gbs > 0 and n == 1 and secs > 0
    ops = bench.oracle_qkv_operands(w, 128)
    assert bench.oracle_steps(w, 3, ops, 128) == sum(
        bench.qkv_sample_bytes(w, 128, [L]) for L in (40, 17, 40))
    for fp8 in (False, True):
        run, flops, Pc = bench.oracle_prefill_sample(48, fp8)
        run()
        assert Pc == 48 and flops == bench.prefill_flops([48], [48])


def test_balanced_parts_cover_every_sequence_once():
    rng = np.random.default_rng(5)
    for parts in (1, 3, 16):
        lens = rng.integers(1, 16384, size=64)
        groups = bench.balanced_parts(lens, parts)
        flat = sorted(b for g in groups for b in g)
        assert flat == list(range(64)) and len(groups) == min(parts, 64)
        loads = [int(lens[g].sum()) for g in groups]
        # greedy longest-first: no group exceeds the mean by more than the longest sequence
        assert max(loads) <= sum(loads) / len(loads) + lens.max()


def test_all_core_oracle_sample_runs_on_threads():
    """The all-core CPU baseline: a layer's sequences split over threads,
    the same oracle call per group; it reports the threads it used."""
    from gqa_paged_kv_gb300 import workloads as wl
    spec = wl.custom(5, [40, 17, 300, 2, 90], pool_pages=64, layers=2)
    w = wl.build(spec, "cpu")
    gbs, used, n, secs = bench.oracle_sample_all_cores(w, 0.0, 3)
    assert gbs > 0 and used == 3 and n == 1 and secs > 0
    gbs1, what, n1, _ = bench.oracle_sample(w, 0.0, per_seq=False)
    assert gbs1 > 0 and n1 == 1


def test_reference_arm_prepares_its_steps_outside_the_clock():
    from gqa_paged_kv_gb300 import workloads as wl
    spec = wl.custom(2, [40, 17], pool_pages=16, layers=2)
    w = wl.build(spec, "cpu")
    prepared = bench.oracle_step_inputs(w, 5)
    assert [b for _, b in prepared] == [0, 1, 0, 1, 0]
    assert bench.oracle_run_steps(w, prepared) == sum(
        bench.sample_bytes(w, [L]) for L in (40, 17, 40, 17, 40))


def test_step_spread_percentiles_by_nearest_rank():
    """Per-step ms over 4 layers: median, p10 and p90 by nearest rank, in µs
    per layer-step; an empty list gives no figures."""
    per = [float(x) for x in range(1, 12)]          # 1 .. 11 ms
    got = bench.step_spread(per, 4)
    assert got == {"median": 6 * 1e3 / 4, "p10": 2 * 1e3 / 4, "p90": 10 * 1e3 / 4}
    assert bench.step_spread([], 4) == {}
    assert bench.step_spread([2.0], 2) == {"median": 1000.0, "p10": 1000.0, "p90": 1000.0}
