"""Host-side pieces of bench.py: the byte and FLOP accounting behind the
roofline figures, the compact pools the CPU-baseline samples run on, the
clock-window filtering and the one-core pinning of the oracle.  CPU only."""
import os

import numpy as np
import pytest

import bench
import oracle
from paged_kv_cache_172_gb300 import workloads


def test_prefill_flops_matches_brute_force():
    # query i of an Lq chunk on a context of n keys sees n - Lq + i + 1 keys;
    # each (query, key) pair costs 2 D (Q K^T) + 2 D (P V) FLOPs, per head
    for ctx, Lq, H, D in (([4096] * 8, 512, 40, 128), ([7, 300, 129], 7, 3, 64), ([1], 1, 1, 64)):
        brute = 0
        for n in ctx:
            for i in range(Lq):
                brute += 4 * D * H * (n - Lq + i + 1)
        assert bench.prefill_flops(ctx, Lq, H, D) == brute
    assert bench.prefill_flops([4096] * 8, 512, 40, 128) == 322164490240


def test_decode_bytes_counts_rows_queries_tables():
    ctx = [1, 16, 17, 2048]
    H, D, bs = 40, 128, 16
    rows = sum(ctx) * H * 2 * D * 2  # K and V rows of every attended (key, head)
    qo = 2 * len(ctx) * H * D * 2
    tables = (1 + 1 + 2 + 128) * 4 + len(ctx) * 4
    assert bench.decode_bytes(ctx, len(ctx), H, D, bs) == rows + qo + tables
    # e4m3 rows with one fp32 scale per (token, head) row of K and of V
    fp8 = bench.decode_bytes(ctx, len(ctx), H, D, bs, elem_bytes=1, scale_bytes=4)
    assert fp8 == sum(ctx) * H * (2 * D + 8) + qo + tables
    assert bench.write_bytes(38, 40, 128) == 2 * 2 * 38 * 40 * 128 * 2 + 38 * 8


def test_unique_kv_bytes_counts_shared_blocks_once():
    bs, H, D = 4, 2, 8
    # two sequences share physical blocks 5 and 6; 6 is partial in seq 0 (ctx 7)
    # and full in seq 1 (ctx 11: blocks 5, 6, 9)
    tables = np.array([[5, 6, -1], [5, 6, 9]], np.int32)
    got = bench.unique_kv_bytes(tables, [7, 11], bs, H, D)
    assert got == (4 + 4 + 3) * H * D * 2 * 2
    lay = workloads.prefix_sharing_layout(seed=2)
    u = bench.unique_kv_bytes(lay.tables, lay.context_lens, 16, 40, 128)
    shared = 16 * 63 * 16  # 16 prompts x 63 shared blocks x 16 tokens
    private = int((lay.context_lens - 63 * 16).sum())  # copy-on-write block + tail, per sample
    assert u == (shared + private) * 40 * 128 * 4


def test_compact_pool_keeps_decode_exact():
    batch = workloads.random_decode(4, 3, 64, 8, [37, 1, 64, 100], seed=9, extra_blocks=5)
    ctx = batch.context_lens.numpy()
    bt = batch.block_tables.numpy()
    full = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(), bt, ctx,
                         batch.scale)
    (kc, vc), bt2, remap = bench.compact_pool(bt, ctx, 8, [batch.k_cache, batch.v_cache])
    used = {int(x) for b in range(4) for x in bt[b, :-(-int(ctx[b]) // 8)]}
    assert kc.shape[0] == len(used) == len(remap)
    comp = oracle.decode(batch.q.numpy(), kc, vc, bt2, ctx, batch.scale)
    assert np.array_equal(full, comp)  # same rows, same arithmetic: identical results


def test_clock_summary_uses_only_samples_inside_windows():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.nvml, s.note = object(), None
    s.samples = [(1.0, 2070.0, 2070.0, 0), (2.0, 1800.0, 2070.0, 0x4),
                 (3.0, 2000.0, 2070.0, 0x40), (4.0, 2060.0, 2070.0, 0)]
    out = s.summary([(0.5, 2.5)])
    assert out["samples"] == 2 and out["sm_mhz"] == 1935.0
    assert out["reasons"] == ["sw_power_cap"]
    out = s.summary([(0.5, 1.5), (2.9, 3.1)])
    assert out["samples"] == 2 and out["reasons"] == ["hw_thermal_slowdown"]
    assert s.summary([(10.0, 11.0)])["samples"] == 0


@pytest.mark.skipif(not hasattr(os, "sched_getaffinity"), reason="no affinity API")
def test_one_core_pins_and_restores():
    before = sorted(os.sched_getaffinity(0))
    with bench.one_core() as info:
        assert info["cpu_count"] == os.cpu_count()
        assert info["affinity"] == before
        assert sorted(os.sched_getaffinity(0)) == [info["pinned_core"]]
    assert sorted(os.sched_getaffinity(0)) == before


def test_config_keys_are_the_workload_only():
    # the same keys in both arms; launch details live outside `config`
    batch = workloads.random_decode(3, 2, 64, 16, [5, 40, 17], seed=3)
    cfg = bench.workload_config(batch)
    assert set(cfg) == {"workload", "B", "H", "head_dim", "block_size", "num_blocks",
                        "sum_context_len"}
    assert cfg["sum_context_len"] == 62 and cfg["B"] == 3 and cfg["head_dim"] == 64
