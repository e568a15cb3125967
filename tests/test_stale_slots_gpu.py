"""Pool slots a call must not read may hold anything, NaN included: the
unwritten tail of each sequence's last block and every block no table uses
(a serving pool is allocated without initialisation).  Attention over the
valid keys must not change: decode and chunked prefill
against the oracle, which reads only keys below each context length."""
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


def poison(batch):
    """NaN in every slot no sequence reads (tails of last blocks, unused blocks)."""
    bs = batch.block_size
    used = np.zeros(batch.k_cache.shape[0], dtype=bool)
    tails = []
    for b, n in enumerate(batch.context_lens.tolist()):
        nb = -(-n // bs)
        ids = batch.block_tables[b, :nb].tolist()
        used[ids] = True
        if n % bs:
            tails.append((ids[-1], n % bs))
    nan = float("nan")
    for kc in (batch.k_cache, batch.v_cache):
        kc[torch.from_numpy(~used)] = nan
        for blk, off in tails:
            kc[blk, off:] = nan
    return int((~used).sum()), len(tails)


@pytest.mark.parametrize("Lq", [200, 400])  # one and two work units per (sequence, head)
@pytest.mark.parametrize("bs,D", [(16, 128), (32, 128), (4, 128), (8, 64), (4, 64)])
def test_prefill_ignores_stale_slots(bs, Lq, D):
    ctx = [Lq + 333, Lq + 1007, Lq + 9]  # partial last blocks
    batch = workloads.random_prefill(len(ctx), 3, D, bs, Lq, ctx, seed=300 + bs + Lq + D,
                                     device="cpu", write_chunk=False)
    n_unused, n_tails = poison(batch)
    assert n_tails == len(ctx)
    ref = oracle.prefill(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                         batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out = pk.pa_prefill_chunk(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], batch.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(out).all()
    assert_close(out, ref, what=f"prefill with NaN in unread slots bs={bs} D={D} Lq={Lq}")


@pytest.mark.parametrize("bs", [4, 16, 32])
def test_decode_ignores_stale_slots(bs):
    ctx = [1, bs + 3, 5 * bs - 1, 700 + 3]
    batch = workloads.random_decode(len(ctx), 4, 128, bs, ctx, seed=310 + bs, device="cpu")
    poison(batch)
    ref = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                        batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    for pt in (0, 4 * bs):
        status = zero_status(DEV)
        out = pk.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                           g["context_lens"], batch.scale, max(ctx), partition_tokens=pt,
                           status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.isfinite(out).all()
        assert_close(out, ref, what=f"decode with NaN in unread slots bs={bs} pt={pt}")
