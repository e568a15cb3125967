"""Parity of pa_prefill_chunk_varlen (chunks of different lengths) with the
fp64 oracle.

Sequence b's q_lens[b] new queries sit in rows 0 .. q_lens[b]-1 of its slice
of q [B, H, Lq_max, D]; query i is at position ctx_b - q_lens[b] + i and sees
keys 0 .. ctx_b - q_lens[b] + i.  Rows past q_lens[b] come back as zeros.
Cases: lengths 0, 1, around the 128-row tile and the 256-query work unit,
head dims 64 and 128, 4- and 16-token blocks, the tail split's partials and
combine, equal lengths against pa_prefill_chunk, and the status bits.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, to_dev, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def varlen_case(H, D, bs, Lq_max, q_lens, extra, seed):
    """A paged batch whose sequence b holds q_lens[b] + extra[b] keys."""
    ctx = [int(a) + int(e) for a, e in zip(q_lens, extra)]
    ctx = [max(c, 1) for c in ctx]  # every sequence keeps at least one block
    batch = workloads.random_prefill(len(ctx), H, D, bs, Lq_max, [max(c, Lq_max) for c in ctx],
                                     seed=seed, device="cpu", write_chunk=False)
    batch.context_lens = torch.tensor(ctx, dtype=torch.int32)
    return batch, torch.tensor(q_lens, dtype=torch.int32)


def run(batch, q_lens, tail_split=True, status=None):
    g = to_dev(batch, DEV)
    out = torch.full_like(g["q"], float("nan"))  # every row must be written
    return pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                               g["context_lens"], batch.scale, out=out, tail_split=tail_split,
                               status=status, q_lens=q_lens.to(DEV))


def oracle_rows(batch, q_lens, seqs=None):
    seqs = list(range(batch.q.shape[0])) if seqs is None else seqs
    return oracle.prefill_varlen(batch.q.numpy()[seqs], batch.k_cache.numpy(),
                                 batch.v_cache.numpy(), batch.block_tables.numpy()[seqs],
                                 batch.context_lens.numpy()[seqs], q_lens.numpy()[seqs],
                                 batch.scale)


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 16), (128, 4), (64, 4)])
def test_varlen_lengths_around_tiles(D, bs):
    q_lens = [0, 1, 100, 128, 129, 255, 256, 257]
    extra = [3, 0, 517, 1, 64, 300, 0, 129]
    batch, ql = varlen_case(2, D, bs, 300, q_lens, extra, seed=300 + D + bs)
    status = zero_status(DEV)
    out = run(batch, ql, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle_rows(batch, ql)
    assert_close(out, ref, what=f"varlen D={D} bs={bs}")
    for b, n in enumerate(q_lens):
        assert torch.all(out[b, :, n:] == 0), f"padded rows of sequence {b}"


def test_varlen_tail_split_matches_whole_units_and_oracle():
    # 8 x 20 heads x 2 work units = 320 units: the last, partial round is
    # split into key ranges (partials merged by the combine kernel)
    q_lens = [512, 300, 0, 1, 257, 128, 511, 64]
    extra = [0, 100, 5, 777, 40, 1000, 2, 300]
    batch, ql = varlen_case(20, 128, 16, 512, q_lens, extra, seed=310)
    assert pk.pa_prefill_workspace_size(8, 20, 512, 128) > 0
    split = run(batch, ql, tail_split=True)
    whole = run(batch, ql, tail_split=False)
    torch.cuda.synchronize()
    d = (split.float() - whole.float()).abs()
    assert d.max().item() <= 2e-3
    seqs = [0, 1, 3, 4, 6]
    ref = oracle_rows(batch, ql, seqs)
    assert_close(split[torch.tensor(seqs, device=DEV)], ref, what="varlen with the tail split")
    for b, n in enumerate(q_lens):
        assert torch.all(split[b, :, n:] == 0) and torch.all(whole[b, :, n:] == 0)


def test_equal_lengths_match_pa_prefill_chunk_bit_for_bit():
    batch = workloads.random_prefill(3, 4, 128, 16, 200, [333, 200, 900], seed=320,
                                     device="cpu", write_chunk=False)
    g = to_dev(batch, DEV)
    a = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                            g["context_lens"], batch.scale)
    b = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                            g["context_lens"], batch.scale,
                            q_lens=torch.full((3,), 200, dtype=torch.int32, device=DEV))
    assert torch.equal(a, b)


def test_varlen_bad_lengths_flagged():
    q_lens = [50, 60, 40]
    batch, ql = varlen_case(2, 128, 16, 64, q_lens, [10, 0, 30], seed=330)
    bad = torch.tensor([65, 60, 40], dtype=torch.int32)  # more than Lq_max
    status = zero_status(DEV)
    out = run(batch, bad, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_CONTEXT
    assert torch.all(out[0] == 0)
    ref = oracle_rows(batch, ql, [1, 2])
    assert_close(out[1:], ref, what="the other sequences")
    status.zero_()
    short = dataclasses.replace(batch, context_lens=torch.tensor([49, 60, 70],
                                                                 dtype=torch.int32))
    out = run(short, ql, status=status)  # 50 new queries on a 49-key context
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_CONTEXT
    assert torch.all(out[0] == 0)
