"""Parity of pa_prefill_chunk (tcgen05 tensor-core kernel) with the fp64 oracle.

The chunk's Lq queries are the last Lq positions of each sequence; query i
sees keys 0 .. ctx-Lq+i.  Cases go from one 128x128 tile up to the
8-sequence, 512-query chunk on a 3,584-token paged context.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, errors, to_dev, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def run_prefill(g, scale, status=None, out=None):
    return pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                               g["context_lens"], scale, status=status, out=out)


def check_against_oracle(B, H, bs, Lq, ctx, seed, what, D=128):
    batch = workloads.random_prefill(B, H, D, bs, Lq, ctx, seed=seed, device="cpu",
                                     write_chunk=False)
    ref = oracle.prefill(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                         batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out = run_prefill(g, batch.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return assert_close(out, ref, what=what)


def test_prefill_one_tile():
    check_against_oracle(1, 1, 16, 128, [128], seed=40, what="one 128x128 tile")


def test_prefill_two_key_tiles():
    check_against_oracle(1, 2, 16, 128, [256], seed=41, what="two key tiles")


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("Lq,ctx", [(1, [1, 77]), (100, [100, 300]), (200, [333, 200]),
                                    (256, [1000, 700]), (37, [4096, 37])])
def test_prefill_ragged(bs, Lq, ctx):
    check_against_oracle(len(ctx), 3, bs, Lq, ctx, seed=42 + Lq, what=f"bs={bs} Lq={Lq} {ctx}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [4, 8, 16, 32])
@pytest.mark.parametrize("Lq,ctx", [(1, [1, 77]), (100, [100, 300]), (200, [333, 200]),
                                    (257, [257, 900]), (37, [1500, 37])])
def test_prefill_head_dims_and_block_sizes(D, bs, Lq, ctx):
    """Every (head_dim, block_size) the library takes: 64-dim rows (one
    swizzle half) and 4-token blocks (gathered by cp.async, two blocks per
    8-row swizzle atom) included, ragged chunks and contexts."""
    check_against_oracle(len(ctx), 3, bs, Lq, ctx, seed=70 + Lq + bs + D, D=D,
                         what=f"D={D} bs={bs} Lq={Lq} {ctx}")


@pytest.mark.parametrize("D,bs", [(64, 16), (64, 4), (128, 4), (128, 8)])
def test_prefill_permutation_invariance_small_blocks_and_d64(D, bs):
    batch = workloads.random_prefill(2, 3, D, bs, 160, [600, 300], seed=53 + bs + D,
                                     device="cpu", write_chunk=False)
    g = to_dev(batch, DEV)
    out = run_prefill(g, batch.scale)
    perm = torch.randperm(batch.num_blocks, generator=torch.Generator().manual_seed(6))
    k2 = torch.empty_like(batch.k_cache)
    v2 = torch.empty_like(batch.v_cache)
    k2[perm] = batch.k_cache
    v2[perm] = batch.v_cache
    bt = batch.block_tables.long()
    t2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], torch.full_like(bt, -1)).int()
    out2 = run_prefill(dict(g, k_cache=k2.to(DEV), v_cache=v2.to(DEV),
                            block_tables=t2.to(DEV)), batch.scale)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("D,bs", [(64, 16), (64, 4), (128, 4)])
def test_prefill_value_ones_and_bad_block_small_blocks_and_d64(D, bs):
    batch = workloads.random_prefill(2, 2, D, bs, 130, [500, 130], seed=54 + bs + D,
                                     device=DEV, write_chunk=False)
    g = to_dev(batch, DEV)
    out = run_prefill(dict(g, v_cache=torch.ones_like(g["v_cache"])), batch.scale)
    assert torch.all(out == 1.0)
    # a block id past the pool: flagged, never dereferenced (read as zeros)
    bt = g["block_tables"].clone()
    bt[0, 3] = batch.num_blocks + 5
    status = zero_status(DEV)
    run_prefill(dict(g, block_tables=bt), batch.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_BLOCK_ID


def test_prefill_lq1_matches_decode():
    batch = workloads.random_prefill(4, 8, 128, 16, 1, [1, 129, 2000, 640], seed=50,
                                     device=DEV, write_chunk=False)
    g = to_dev(batch, DEV)
    a = run_prefill(g, batch.scale)[:, :, 0]
    b = pk.pa_decode(g["q"][:, :, 0].contiguous(), g["k_cache"], g["v_cache"],
                     g["block_tables"], g["context_lens"], batch.scale, 2000)
    assert (a.float() - b.float()).abs().max().item() <= 2e-3


def test_prefill_permutation_invariance_bit_exact():
    batch = workloads.random_prefill(2, 4, 128, 16, 160, [600, 300], seed=51, device="cpu",
                                     write_chunk=False)
    g = to_dev(batch, DEV)
    out = run_prefill(g, batch.scale)
    perm = torch.randperm(batch.num_blocks, generator=torch.Generator().manual_seed(5))
    k2 = torch.empty_like(batch.k_cache)
    v2 = torch.empty_like(batch.v_cache)
    k2[perm] = batch.k_cache
    v2[perm] = batch.v_cache
    bt = batch.block_tables.long()
    t2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], torch.full_like(bt, -1)).int()
    out2 = run_prefill(dict(g, k_cache=k2.to(DEV), v_cache=v2.to(DEV),
                            block_tables=t2.to(DEV)), batch.scale)
    assert torch.equal(out, out2)


@pytest.mark.parametrize("Lq", [130, 300])  # one and two work units per (sequence, head)
def test_prefill_value_ones_and_bad_context(Lq):
    batch = workloads.random_prefill(2, 2, 128, 16, Lq, [Lq + 370, Lq], seed=52, device=DEV,
                                     write_chunk=False)
    g = to_dev(batch, DEV)
    out = run_prefill(dict(g, v_cache=torch.ones_like(g["v_cache"])), batch.scale)
    assert torch.all(out == 1.0)
    status = zero_status(DEV)
    bad = g["context_lens"].clone()
    bad[1] = Lq - 1  # shorter than the chunk
    out = torch.full_like(g["q"], 3.0)
    run_prefill(dict(g, context_lens=bad), batch.scale, status=status, out=out)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_CONTEXT
    assert torch.all(out[1] == 0)


def test_chunked_prefill_workload():
    """8 x 512 queries on 3,584 cached tokens, 40 heads: chunk K/V written by
    pa_kv_cache_write first; oracle on whole (b, h) rows of two heads and on
    sampled rows (tile and mask edges) of every (b, h)."""
    batch = workloads.chunked_prefill(seed=4, device=DEV)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    kc0 = batch.k_cache.cpu().numpy()
    vc0 = batch.v_cache.cpu().numpy()
    pk.pa_kv_cache_write(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"],
                         status=status)
    out = run_prefill(g, batch.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc, vc = oracle.kv_cache_write(batch.k_new.cpu().numpy(), batch.v_new.cpu().numpy(),
                                   batch.slot_mapping.cpu().numpy(), kc0, vc0)
    assert np.array_equal(g["k_cache"].cpu().numpy().view(np.uint16), kc)
    q = batch.q.cpu().numpy()
    tables = batch.block_tables.cpu().numpy()
    ctx = batch.context_lens.cpu().numpy()
    Lq = q.shape[2]
    got = out.float().cpu().numpy()
    errs = []
    for (b, h) in [(0, 0), (5, 33)]:  # whole rows
        for i in range(Lq):
            ref = oracle.attend_row(q[b, h, i], kc, vc, tables[b], ctx[b] - Lq + i + 1, h,
                                    batch.scale)
            errs.append(np.abs(got[b, h, i] - ref))
    rows = [0, 1, 126, 127, 128, 129, 255, 256, 383, 384, 510, 511]
    for b in range(q.shape[0]):
        for h in range(0, q.shape[1], 3):
            for i in rows:
                ref = oracle.attend_row(q[b, h, i], kc, vc, tables[b], ctx[b] - Lq + i + 1, h,
                                        batch.scale)
                errs.append(np.abs(got[b, h, i] - ref))
    err = np.concatenate(errs)
    print(f"chunked prefill: {len(errs)} rows, max|err| {err.max():.2e} mean {err.mean():.2e}")
    assert err.max() <= 5e-3 and err.mean() <= 5e-4


def test_tail_split_matches_whole_units_and_oracle():
    # One sequence, H = SMs + 8 heads, 256 queries: one work unit per head, so
    # the last 8 heads form the partial last round and are split into key ranges.
    nsm = torch.cuda.get_device_properties(DEV).multi_processor_count
    H, Lq, bs = nsm + 8, 256, 16
    ctx = [Lq + 5 * 128 + 37]
    assert pk.pa_prefill_workspace_size(1, H, Lq, 128) > 0
    batch = workloads.random_prefill(1, H, 128, bs, Lq, ctx, seed=95, device="cpu",
                                     write_chunk=False)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out_split = run_prefill(g, batch.scale, status=status)  # the binding allocates the workspace
    out_whole = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                    g["context_lens"], batch.scale, tail_split=False,
                                    status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the split heads against the oracle (heads sliced out of the pool)
    hs = list(range(H - 10, H))
    sl = lambda t: t[:, :, hs].contiguous()
    ref = oracle.prefill(batch.q[:, hs].contiguous().numpy(), sl(batch.k_cache).numpy(),
                         sl(batch.v_cache).numpy(), batch.block_tables.numpy(),
                         batch.context_lens.numpy(), batch.scale)
    assert_close(out_split[:, hs], ref, what="tail-split heads")
    e = errors(out_split, out_whole.float().cpu().numpy().astype(np.float64))
    assert e[0] <= 2e-3, e


@pytest.mark.parametrize("bs", [16, 32])
@pytest.mark.parametrize("Lq,ctx", [(257, [257, 900]), (384, [1000, 500]), (512, [512, 1200]),
                                    (640, [700, 1500]), (1000, [1100, 1000])])
def test_prefill_long_chunks_ragged(bs, Lq, ctx):
    """Chunks of several 256-query work units per (sequence, head), the last one
    ragged inside either of its two Q tiles."""
    check_against_oracle(len(ctx), 2, bs, Lq, ctx, seed=60 + Lq + bs,
                         what=f"long chunk bs={bs} Lq={Lq} {ctx}")


@pytest.mark.parametrize("D,bs", [(64, 16), (64, 8), (128, 4)])
def test_tail_split_d64_and_small_blocks(D, bs):
    # As above for 64-dim heads (the combine's two dims per lane) and for the
    # cp.async gather: H = SMs + 8 heads, one unit per head, the last 8 split.
    nsm = torch.cuda.get_device_properties(DEV).multi_processor_count
    H, Lq = nsm + 8, 256
    ctx = [Lq + 3 * 128 + 21]
    assert pk.pa_prefill_workspace_size(1, H, Lq, D) > 0
    batch = workloads.random_prefill(1, H, D, bs, Lq, ctx, seed=97 + D + bs, device="cpu",
                                     write_chunk=False)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out_split = run_prefill(g, batch.scale, status=status)
    out_whole = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                    g["context_lens"], batch.scale, tail_split=False,
                                    status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    hs = list(range(H - 10, H))
    sl = lambda t: t[:, :, hs].contiguous()
    ref = oracle.prefill(batch.q[:, hs].contiguous().numpy(), sl(batch.k_cache).numpy(),
                         sl(batch.v_cache).numpy(), batch.block_tables.numpy(),
                         batch.context_lens.numpy(), batch.scale)
    assert_close(out_split[:, hs], ref, what=f"tail-split heads D={D} bs={bs}")
    e = errors(out_split, out_whole.float().cpu().numpy().astype(np.float64))
    assert e[0] <= 2e-3, e


def test_tail_split_two_units_per_head():
    # One sequence, 512 queries: two work units per head; SMs / 2 + 6 heads
    # leave a partial last round (12 units), split into key ranges.
    nsm = torch.cuda.get_device_properties(DEV).multi_processor_count
    H, Lq, bs = nsm // 2 + 6, 512, 16
    ctx = [Lq + 3 * 128 + 77]
    batch = workloads.random_prefill(1, H, 128, bs, Lq, ctx, seed=96, device="cpu",
                                     write_chunk=False)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out_split = run_prefill(g, batch.scale, status=status)
    out_whole = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                    g["context_lens"], batch.scale, tail_split=False,
                                    status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    hs = list(range(H - 8, H))
    sl = lambda t: t[:, :, hs].contiguous()
    ref = oracle.prefill(batch.q[:, hs].contiguous().numpy(), sl(batch.k_cache).numpy(),
                         sl(batch.v_cache).numpy(), batch.block_tables.numpy(),
                         batch.context_lens.numpy(), batch.scale)
    assert_close(out_split[:, hs], ref, what="tail-split heads, two units each")
    e = errors(out_split, out_whole.float().cpu().numpy().astype(np.float64))
    assert e[0] <= 2e-3, e


def spiked_batch(D, bs, seed):
    """Scores with jumps far past the softmax's rescale margin: every query is
    u + noise (u = ones) and chosen keys are a * u, so a key's score is about
    a * D above the rest.  Sequence 0: a spike at the last key, masked for all
    queries but the last.  Sequence 1: spikes of growing size in tiles with no
    masked key (the running maximum jumps three times).  Sequence 2: the
    largest score at key 0.  Sequence 3: spikes inside the chunk, each seen
    only by the queries at or after it."""
    Lq, ctx = 256, [1024, 1024, 1024, 600]
    batch = workloads.random_prefill(4, 2, D, bs, Lq, ctx, seed=seed, device="cpu",
                                     write_chunk=False)
    g = torch.Generator().manual_seed(seed)
    batch.q = (1.0 + 0.25 * torch.randn(batch.q.shape, generator=g)).half()
    per_nat = 1.0 / (D * batch.scale)  # key multiple that adds one nat to the score
    spikes = {0: [(ctx[0] - 1, 45)],
              1: [(100, 15), (400, 35), (700, 60)],
              2: [(0, 60)],
              3: [(ctx[3] - Lq + 10, 30), (ctx[3] - Lq + 130, 50), (ctx[3] - Lq + 250, 70)]}
    for b, marks in spikes.items():
        for pos, nats in marks:
            blk = int(batch.block_tables[b, pos // bs])
            batch.k_cache[blk, pos % bs] = torch.full((2, D), nats * per_nat).half()
    return batch


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 16), (128, 4)])
@pytest.mark.parametrize("tail_split", [True, False])
def test_prefill_score_spikes(D, bs, tail_split):
    # the row maximum is taken from the tensor-memory load on tiles with no
    # masked key and from the unmasked keys on diagonal tiles; scores that
    # jump by 15-70 nats check both, and the rescaling of the output
    batch = spiked_batch(D, bs, seed=60 + D + bs)
    ref = oracle.prefill(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                         batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    assert np.all(np.isfinite(ref))
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], batch.scale, status=status,
                              tail_split=tail_split)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, ref, what=f"score spikes D={D} bs={bs} split={tail_split}")
