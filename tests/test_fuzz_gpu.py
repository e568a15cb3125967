"""Seeded random configurations of every attention entry point against the
fp64 oracle: batch size, head count (odd ones included), head dim, block size,
context lengths (empty sequences included), partition length, chunk lengths,
sharing groups.  Each draw is small enough for the oracle; together they walk
the shape space the fixed tests sample at chosen points."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, to_dev, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BLOCK_SIZES = (4, 8, 16, 32)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def draw_decode(rng):
    D = int(rng.choice((64, 128)))
    bs = int(rng.choice(BLOCK_SIZES))
    B = int(rng.integers(1, 10))
    H = int(rng.integers(1, 7))
    ctx = rng.integers(0, 700, size=B)
    ctx[rng.random(B) < 0.15] = 0
    ctx[rng.random(B) < 0.15] = int(rng.integers(1, 2 * bs + 2))
    pt = int(rng.choice((0, bs, 4 * bs, 8 * bs, 32 * bs)))
    return D, bs, B, H, [int(c) for c in ctx], pt


@pytest.mark.parametrize("seed", range(32))
def test_fuzz_decode_fp16_and_append(seed):
    rng = np.random.default_rng(1000 + seed)
    D, bs, B, H, ctx, pt = draw_decode(rng)
    batch = workloads.random_decode(B, H, D, bs, ctx, seed=2000 + seed, device="cpu")
    mx = max(max(ctx), 1)
    ref = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                        batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out = pk.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"], g["context_lens"],
                       batch.scale, mx, partition_tokens=pt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, ref, what=f"decode D={D} bs={bs} B={B} H={H} pt={pt} ctx={ctx}")
    # the fused append on the non-empty sequences
    live = [c for c in ctx if c > 0]
    if live:
        ab = workloads.random_decode(len(live), H, D, bs, live, seed=3000 + seed, device="cpu",
                                     new_tokens=True)
        kc, vc = oracle.kv_cache_write(ab.k_new.numpy(), ab.v_new.numpy(), ab.slot_mapping.numpy(),
                                       ab.k_cache.numpy(), ab.v_cache.numpy())
        ref_a = oracle.decode(ab.q.numpy(), kc.view(np.float16), vc.view(np.float16),
                              ab.block_tables.numpy(), ab.context_lens.numpy(), ab.scale)
        ga = to_dev(ab, DEV)
        out_a = pk.pa_decode_append(ga["q"], ga["k_new"], ga["v_new"], ga["k_cache"], ga["v_cache"],
                                    ga["block_tables"], ga["context_lens"], ab.scale, max(live),
                                    partition_tokens=pt, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(ga["k_cache"].cpu().numpy().view(np.uint16), kc.view(np.uint16))
        assert np.array_equal(ga["v_cache"].cpu().numpy().view(np.uint16), vc.view(np.uint16))
        assert_close(out_a, ref_a, what=f"append D={D} bs={bs} H={H} pt={pt} ctx={live}")


@pytest.mark.parametrize("seed", range(20))
def test_fuzz_decode_fp8(seed):
    rng = np.random.default_rng(1100 + seed)
    D, bs, B, H, ctx, pt = draw_decode(rng)
    batch = workloads.random_decode(B, H, D, bs, ctx, seed=2100 + seed, device="cpu")
    NB = batch.k_cache.shape[0]
    rows = NB * bs
    k8o, v8o, kso, vso = oracle.kv_cache_write_fp8(
        batch.k_cache.reshape(rows, H, D).numpy(), batch.v_cache.reshape(rows, H, D).numpy(),
        np.arange(rows, dtype=np.int64), np.zeros((NB, bs, H, D), np.uint8),
        np.zeros((NB, bs, H, D), np.uint8), np.ones((NB, H, bs), np.float32),
        np.ones((NB, H, bs), np.float32))
    ref = oracle.decode_fp8(batch.q.numpy(), k8o, v8o, kso, vso, batch.block_tables.numpy(),
                            batch.context_lens.numpy(), batch.scale)
    k8 = torch.zeros((NB, bs, H, D), dtype=torch.uint8, device=DEV)
    v8 = torch.zeros_like(k8)
    ks = torch.ones((NB, H, bs), dtype=torch.float32, device=DEV)
    vs = torch.ones_like(ks)
    status = zero_status(DEV)
    pk.pa_kv_cache_write_fp8(batch.k_cache.reshape(rows, H, D).to(DEV),
                             batch.v_cache.reshape(rows, H, D).to(DEV),
                             torch.arange(rows, dtype=torch.int64, device=DEV), k8, v8, ks, vs,
                             status=status)
    out = pk.pa_decode_fp8(batch.q.to(DEV), k8, v8, ks, vs, batch.block_tables.to(DEV),
                           batch.context_lens.to(DEV), batch.scale, max(max(ctx), 1),
                           partition_tokens=pt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(k8.cpu().numpy(), k8o) and np.array_equal(vs.cpu().numpy(), vso)
    assert_close(out, ref, what=f"fp8 D={D} bs={bs} B={B} H={H} pt={pt} ctx={ctx}")


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_prefill_and_varlen(seed):
    rng = np.random.default_rng(1200 + seed)
    D = int(rng.choice((64, 128)))
    bs = int(rng.choice(BLOCK_SIZES))
    B = int(rng.integers(1, 4))
    H = int(rng.integers(1, 4))
    Lq = int(rng.integers(1, 300))
    ctx = [Lq + int(rng.integers(0, 500)) for _ in range(B)]
    batch = workloads.random_prefill(B, H, D, bs, Lq, ctx, seed=2200 + seed, device="cpu",
                                     write_chunk=False)
    ref = oracle.prefill(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                         batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    split = bool(rng.integers(0, 2))
    out = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], batch.scale, status=status, tail_split=split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    what = f"prefill D={D} bs={bs} B={B} H={H} Lq={Lq} ctx={ctx} split={split}"
    assert_close(out, ref, what=what)
    # chunk lengths 0..Lq per sequence on the same batch
    q_lens = np.array([int(rng.integers(0, Lq + 1)) for _ in range(B)], np.int32)
    ref_v = oracle.prefill_varlen(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                                  batch.block_tables.numpy(), batch.context_lens.numpy(), q_lens,
                                  batch.scale)
    out_v = pk.pa_prefill_chunk_varlen(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                       g["context_lens"], torch.from_numpy(q_lens).to(DEV),
                                       batch.scale, status=status, tail_split=split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out_v, ref_v, what=f"varlen {what} q_lens={q_lens.tolist()}")


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_shared_prefix(seed):
    rng = np.random.default_rng(1300 + seed)
    D = int(rng.choice((64, 128)))
    bs = int(rng.choice(BLOCK_SIZES))
    H = int(rng.integers(1, 5))
    gmax = int(rng.choice((2, 4, 8, 16)))
    tables, ctx, NB = workloads.fork_forest_layout(2300 + seed, B=int(rng.integers(6, 24)),
                                                   block_size=bs, max_blocks=int(rng.integers(12, 32)),
                                                   p_root=float(rng.uniform(0.05, 0.25)))
    pt = bs * int(rng.choice((2, 4)))
    sg, off, seqs, pref = pk.pa_shared_prefix_groups(torch.from_numpy(tables),
                                                     torch.from_numpy(ctx), bs, pt, gmax)
    gen = torch.Generator().manual_seed(2400 + seed)
    kc = torch.randn((NB, bs, H, D), generator=gen).half()
    vc = torch.randn((NB, bs, H, D), generator=gen).half()
    q = torch.randn((len(ctx), H, D), generator=gen).half()
    scale = 1.0 / np.sqrt(D)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), tables, ctx, scale)
    status = zero_status(DEV)
    max_pref = int(pref.max()) if pref.numel() else 0
    out = pk.pa_decode_shared_prefix(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                     torch.from_numpy(tables).to(DEV), torch.from_numpy(ctx).to(DEV),
                                     sg.to(DEV), off.to(DEV), seqs.to(DEV), pref.to(DEV), scale,
                                     int(ctx.max()), gmax, max_pref, partition_tokens=pt,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, ref, what=f"shared prefix D={D} bs={bs} H={H} gmax={gmax} pt={pt}")
