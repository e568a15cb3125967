"""Degenerate calls through the C ABI: empty batches, zero tokens or pairs,
an empty query chunk, all-empty contexts, the smallest shapes, and a group
larger than the shared-prefix path supports."""
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


def pool(NB=8, bs=16, H=2, D=128, seed=0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((NB, bs, H, D), generator=g).half().to(DEV),
            torch.randn((NB, bs, H, D), generator=g).half().to(DEV))


def test_zero_size_calls_do_nothing():
    kc, vc = pool()
    kc0, vc0 = kc.clone(), vc.clone()
    status = zero_status(DEV)
    # decode of an empty batch
    q = torch.empty((0, 2, 128), dtype=torch.float16, device=DEV)
    bt = torch.empty((0, 4), dtype=torch.int32, device=DEV)
    cl = torch.empty((0,), dtype=torch.int32, device=DEV)
    out = pk.pa_decode(q, kc, vc, bt, cl, 0.1, 64, status=status)
    assert out.shape == (0, 2, 128)
    # cache write of no tokens, copy of no blocks
    kv = torch.empty((0, 2, 128), dtype=torch.float16, device=DEV)
    pk.pa_kv_cache_write(kv, kv, torch.empty((0,), dtype=torch.int64, device=DEV), kc, vc,
                         status=status)
    pk.pa_block_copy(kc, vc, torch.empty((0, 2), dtype=torch.int64, device=DEV), status=status)
    # prefill of an empty query chunk
    qp = torch.empty((1, 2, 0, 128), dtype=torch.float16, device=DEV)
    outp = pk.pa_prefill_chunk(qp, kc, vc, torch.zeros((1, 4), dtype=torch.int32, device=DEV),
                               torch.tensor([16], dtype=torch.int32, device=DEV), 0.1,
                               status=status)
    assert outp.shape == (1, 2, 0, 128)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kc, kc0) and torch.equal(vc, vc0)


def test_all_contexts_empty_give_zero_rows():
    kc, vc = pool(H=3, D=64, bs=4)
    B = 5
    q = torch.randn((B, 3, 64), device=DEV).half()
    bt = torch.full((B, 3), -1, dtype=torch.int32, device=DEV)
    cl = torch.zeros((B,), dtype=torch.int32, device=DEV)
    out = torch.full((B, 3, 64), float("nan"), dtype=torch.float16, device=DEV)
    status = zero_status(DEV)
    pk.pa_decode(q, kc, vc, bt, cl, 0.125, 0, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, torch.zeros_like(out))


def test_smallest_shapes_match_oracle():
    # one sequence, one head, one key; D=64 and block size 4
    batch = workloads.random_decode(1, 1, 64, 4, [1], seed=11, device="cpu")
    ref = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                        batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    out = pk.pa_decode(batch.q.to(DEV), batch.k_cache.to(DEV), batch.v_cache.to(DEV),
                       batch.block_tables.to(DEV), batch.context_lens.to(DEV), batch.scale, 1)
    assert_close(out, ref, what="B=H=ctx=1")
    # with a single key the output is that key's value row
    v0 = batch.v_cache[batch.block_tables[0, 0], 0, 0]
    assert torch.equal(out[0, 0].cpu(), v0)


def test_group_larger_than_supported_is_rejected():
    B, H, D, bs = 17, 2, 128, 16
    kc, vc = pool(NB=40, bs=bs, H=H, D=D)
    q = torch.randn((B, H, D), device=DEV).half()
    bt = torch.arange(2, dtype=torch.int32, device=DEV).repeat(B, 1).contiguous()
    cl = torch.full((B,), 2 * bs, dtype=torch.int32, device=DEV)
    sg = torch.zeros((B,), dtype=torch.int32, device=DEV)
    off = torch.tensor([0, B], dtype=torch.int32, device=DEV)
    seqs = torch.arange(B, dtype=torch.int32, device=DEV)
    pref = torch.tensor([2 * bs], dtype=torch.int32, device=DEV)
    with pytest.raises(pk.PagedKVError) as e:
        pk.pa_decode_shared_prefix(q, kc, vc, bt, cl, sg, off, seqs, pref, 0.1, 2 * bs, B, 2 * bs)
    assert e.value.code == pk.PA_ERR_UNSUPPORTED
