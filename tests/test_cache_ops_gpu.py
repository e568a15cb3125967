"""Bit-exact parity of pa_kv_cache_write and pa_block_copy with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import bits, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def rand16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float16)


@pytest.mark.parametrize("D,bs,H", [(64, 4, 4), (128, 16, 40), (128, 32, 8), (64, 8, 3)])
def test_kv_cache_write_bit_exact(D, bs, H):
    nb = 37
    kc = rand16((nb, bs, H, D), 1)
    vc = rand16((nb, bs, H, D), 2)
    rng = np.random.default_rng(D + bs)
    T = 50
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[[3, 17]] = -1  # padding tokens are skipped
    k = rand16((T, H, D), 3)
    v = rand16((T, H, D), 4)
    kr, vr = oracle.kv_cache_write(k.numpy(), v.numpy(), slots, kc.numpy(), vc.numpy())
    gk, gv = kc.to(DEV), vc.to(DEV)
    status = zero_status(DEV)
    pk.pa_kv_cache_write(k.to(DEV), v.to(DEV), torch.from_numpy(slots).to(DEV), gk, gv,
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(gk), kr) and np.array_equal(bits(gv), vr)


def test_kv_cache_write_bad_slot_flagged_and_skipped():
    nb, bs, H, D = 8, 16, 2, 64
    kc = rand16((nb, bs, H, D), 5)
    gk, gv = kc.to(DEV), kc.to(DEV).clone()
    k = rand16((3, H, D), 6)
    slots = torch.tensor([0, nb * bs, 5], dtype=torch.int64)
    status = zero_status(DEV)
    pk.pa_kv_cache_write(k.to(DEV), k.to(DEV), slots.to(DEV), gk, gv, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_SLOT
    kr, _ = oracle.kv_cache_write(k.numpy()[[0, 2]], k.numpy()[[0, 2]], np.array([0, 5]),
                                  kc.numpy(), kc.numpy())
    assert np.array_equal(bits(gk), kr)


@pytest.mark.parametrize("D,bs,H", [(64, 4, 4), (128, 16, 40), (128, 32, 5)])
def test_block_copy_bit_exact(D, bs, H):
    nb = 64
    kc = rand16((nb, bs, H, D), 7)
    vc = rand16((nb, bs, H, D), 8)
    rng = np.random.default_rng(9)
    ids = rng.permutation(nb)
    pairs = np.stack([ids[:20], ids[20:40]], axis=1).astype(np.int64)
    pairs = np.concatenate([pairs, [[ids[50], ids[50]]]])  # src == dst: no-op
    kr, vr = oracle.block_copy(kc.numpy(), vc.numpy(), pairs)
    gk, gv = kc.to(DEV), vc.to(DEV)
    status = zero_status(DEV)
    pk.pa_block_copy(gk, gv, torch.from_numpy(pairs).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(gk), kr) and np.array_equal(bits(gv), vr)


def test_block_copy_bad_pair_flagged():
    nb, bs, H, D = 6, 16, 2, 128
    kc = rand16((nb, bs, H, D), 10)
    gk, gv = kc.to(DEV), kc.to(DEV).clone()
    pairs = torch.tensor([[0, 1], [2, nb], [-1, 3]], dtype=torch.int64)
    status = zero_status(DEV)
    pk.pa_block_copy(gk, gv, pairs.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_PAIR
    kr, _ = oracle.block_copy(kc.numpy(), kc.numpy(), np.array([[0, 1]]))
    assert np.array_equal(bits(gk), kr)


def test_prefix_sharing_copy_on_write_pairs():
    """The 128 copy-on-write pairs of the 16x8 prefix-sharing layout, on a
    reduced head count (same block count and pair pattern)."""
    lay = workloads.prefix_sharing_layout(seed=2)
    H, D, bs = 4, 128, lay.block_size
    kc = rand16((lay.num_blocks, bs, H, D), 11)
    vc = rand16((lay.num_blocks, bs, H, D), 12)
    kr, vr = oracle.block_copy(kc.numpy(), vc.numpy(), lay.pairs)
    gk, gv = kc.to(DEV), vc.to(DEV)
    pk.pa_block_copy(gk, gv, torch.from_numpy(lay.pairs).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(bits(gk), kr) and np.array_equal(bits(gv), vr)
