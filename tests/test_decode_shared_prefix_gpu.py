"""pa_decode_shared_prefix: groups of sequences sharing prefix blocks give the
same result as plain decode (oracle tolerance), with shared partitions read
once per group."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def grouped_batch(sizes, prefix_blocks, tails, H, D, bs, seed):
    """Groups of the given sizes; members share `prefix_blocks[g]` blocks and
    each has a private tail of tails[b] tokens.  Returns tensors + groups."""
    rng = np.random.default_rng(seed)
    B = sum(sizes)
    tables, ctx, seq_group, offsets, seqs, prefix = [], [], [], [0], [], []
    next_blk = 0
    b = 0
    for g, (m, pb) in enumerate(zip(sizes, prefix_blocks)):
        shared = list(range(next_blk, next_blk + pb))
        next_blk += pb
        for _ in range(m):
            t = int(tails[b])
            own = list(range(next_blk, next_blk + -(-t // bs)))
            next_blk += len(own)
            tables.append(shared + own)
            ctx.append(pb * bs + t)
            seq_group.append(g)
            seqs.append(b)
            b += 1
        offsets.append(b)
        prefix.append(pb * bs)
    NB = next_blk + 3
    perm = rng.permutation(NB)
    maxb = max(len(t) for t in tables)
    bt = np.full((B, maxb), -1, np.int32)
    for i, t in enumerate(tables):
        bt[i, :len(t)] = perm[np.asarray(t)]
    gen = torch.Generator().manual_seed(seed)
    kc = torch.randn((NB, bs, H, D), generator=gen).half()
    vc = torch.randn((NB, bs, H, D), generator=gen).half()
    q = torch.randn((B, H, D), generator=gen).half()
    groups = [np.asarray(x, np.int32) for x in (seq_group, offsets, seqs, prefix)]
    return q, kc, vc, bt, np.asarray(ctx, np.int32), groups, max(sizes)


def run_shared(q, kc, vc, bt, ctx, groups, gmax, pt, scale, status=None):
    sg, off, seqs, pref = (torch.from_numpy(x).to(DEV) for x in groups)
    return pk.pa_decode_shared_prefix(q.to(DEV), kc.to(DEV), vc.to(DEV),
                                      torch.from_numpy(bt).to(DEV),
                                      torch.from_numpy(ctx).to(DEV), sg, off, seqs, pref, scale,
                                      int(ctx.max()), gmax, int(groups[3].max()), status=status,
                                      partition_tokens=pt)


@pytest.mark.parametrize("D,bs", [(128, 16), (128, 32), (64, 16), (128, 8), (64, 8), (128, 4),
                                  (64, 4)])
def test_shared_prefix_matches_oracle(D, bs):
    sizes = [1, 3, 16, 2]
    prefix_blocks = [4, 8, 6, 1]
    rng = np.random.default_rng(70 + D + bs)
    tails = rng.integers(1, 5 * bs, size=sum(sizes))
    tails[1] = bs  # a member whose tail fills exactly one block
    q, kc, vc, bt, ctx, groups, gmax = grouped_batch(sizes, prefix_blocks, tails, 4, D, bs,
                                                     seed=71)
    scale = 1.0 / np.sqrt(D)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), bt, ctx, scale)
    status = zero_status(DEV)
    # shared partitions vary, one-partition case included; below 16 tokens per
    # block also partitions that are no multiple of 16 (not shared, per member)
    for pt in sorted({2 * bs, 4 * bs, 8 * bs, 32 * bs}):
        out = run_shared(q, kc, vc, bt, ctx, groups, gmax, pt, scale, status)
        assert_close(out, ref, what=f"shared prefix D={D} bs={bs} pt={pt}")
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_shared_prefix_single_partition_members():
    # every member's whole context is one shared partition (no suffix, no combine)
    sizes = [4, 5]
    prefix_blocks = [8, 8]
    tails = np.zeros(9, dtype=np.int64)
    q, kc, vc, bt, ctx, groups, gmax = grouped_batch(sizes, prefix_blocks, tails, 3, 128, 16,
                                                     seed=72)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), bt, ctx, 0.1)
    out = run_shared(q, kc, vc, bt, ctx, groups, gmax, 128, 0.1)
    assert_close(out, ref, what="single shared partition")


def test_prefix_sharing_workload():
    """16 prompts x 8 samples: copy-on-write copies, then group-aware decode;
    compared with plain decode and with the oracle on a sample of sequences."""
    batch = workloads.prefix_sharing(seed=2, device=DEV)
    lay = batch.meta["layout"]
    pk.pa_block_copy(batch.k_cache, batch.v_cache, batch.copy_pairs)
    groups = workloads.sharing_groups(lay)
    max_ctx = int(lay.context_lens.max())
    pt = 336  # divides the 1,008 shared tokens
    status = zero_status(DEV)
    sg, off, seqs, pref = (torch.from_numpy(x).to(DEV) for x in groups)
    out = pk.pa_decode_shared_prefix(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                                     batch.context_lens, sg, off, seqs, pref, batch.scale,
                                     max_ctx, 8, int(groups[3].max()), partition_tokens=pt,
                                     status=status)
    plain = pk.pa_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                         batch.context_lens, batch.scale, max_ctx, partition_tokens=pt)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (out.float() - plain.float()).abs().max().item() <= 2e-3
    sel = np.arange(1, 128, 5)
    ref = oracle.decode(batch.q.cpu().numpy()[sel], batch.k_cache.cpu().numpy(),
                        batch.v_cache.cpu().numpy(), lay.tables[sel], lay.context_lens[sel],
                        batch.scale)
    assert_close(out[torch.from_numpy(sel).to(DEV)], ref, what="prefix sharing, grouped")


@pytest.mark.parametrize("seed,bs,gmax", [(11, 16, 16), (12, 32, 4), (13, 16, 2)])
def test_groups_from_block_tables(seed, bs, gmax):
    """Groups derived by pa_shared_prefix_groups from a forest of forked
    sequences drive the grouped decode to the oracle's result."""
    H, D = 4, 128
    tables, ctx, NB = workloads.fork_forest_layout(seed, B=48, block_size=bs, max_blocks=40,
                                                   p_root=0.1)
    pt = 4 * bs
    sg, off, seqs, pref = pk.pa_shared_prefix_groups(torch.from_numpy(tables),
                                                     torch.from_numpy(ctx), bs, pt, gmax)
    assert pref.numel() >= 3  # the forest shares prefixes worth grouping
    gen = torch.Generator().manual_seed(seed)
    kc = torch.randn((NB, bs, H, D), generator=gen).half()
    vc = torch.randn((NB, bs, H, D), generator=gen).half()
    q = torch.randn((len(ctx), H, D), generator=gen).half()
    scale = 1.0 / np.sqrt(D)
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), tables, ctx, scale)
    groups = tuple(t.numpy() for t in (sg, off, seqs, pref))
    status = zero_status(DEV)
    out = run_shared(q, kc, vc, tables, ctx, groups, gmax, pt, scale, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out, ref, what=f"derived groups seed={seed} bs={bs} gmax={gmax}")


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 8)])
def test_shared_prefix_score_spikes(D, bs):
    # scores that jump by 15-60 nats inside the shared prefix (the group's
    # MMA partitions, one running maximum per member) and in the private
    # tails, merged across partitions by log-sum-exp
    sizes, prefix_blocks = [3, 4], [8, 6]
    tails = np.array([5, 3 * bs, 1, 2 * bs + 3, bs, 7, 4 * bs])
    q, kc, vc, bt, ctx, groups, gmax = grouped_batch(sizes, prefix_blocks, tails, 2, D, bs,
                                                     seed=73 + D)
    gen = torch.Generator().manual_seed(74 + D)
    q = (1.0 + 0.25 * torch.randn(q.shape, generator=gen)).half()
    scale = 1.0 / np.sqrt(D)
    per_nat = 1.0 / (D * scale)
    marks = [(0, 3, 20), (0, 5 * bs, 40), (0, 8 * bs + 2, 60),  # group 0: prefix, then tail
             (3, 2, 60), (3, 4 * bs + 1, 15),                   # group 1: largest first
             (6, 6 * bs + 4 * bs - 1, 45)]                      # a member's last key
    for b, pos, nats in marks:
        assert pos < ctx[b]
        blk = int(bt[b, pos // bs])
        kc[blk, pos % bs] = torch.full((2, D), nats * per_nat).half()
    ref = oracle.decode(q.numpy(), kc.numpy(), vc.numpy(), bt, ctx, scale)
    assert np.all(np.isfinite(ref))
    status = zero_status(DEV)
    for pt in (2 * bs, 4 * bs):
        out = run_shared(q, kc, vc, bt, ctx, groups, gmax, pt, scale, status)
        assert_close(out, ref, what=f"shared prefix spikes D={D} bs={bs} pt={pt}")
    torch.cuda.synchronize()
    assert int(status.item()) == 0
