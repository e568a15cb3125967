"""FP8 (e4m3) KV storage on the GPU: the quantizing cache write is bit-exact
with the oracle (codes and scales); fp8 decode matches the oracle's fp8
decode on the same codes within the fp16 attention tolerance; and against
the unquantized fp16 data it stays within the bound e4m3 rounding implies."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, spiked_decode_batch, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# Each stored value carries e4m3 rounding of at most 2^-4 relative (half a
# unit in the last of 3 fraction bits).  To first order an output row then
# carries the V rows' error (<= 2^-4 relative) plus the error of its weights,
# which K's rounding perturbs through the scores by about as much: per
# (sequence, head) the relative L2 error against the unquantized fp16 data is
# bounded by 2^-3, and on average (errors of independent elements partly
# cancel) by 2^-4.
FP8_REL_L2_MAX = 2.0 ** -3
FP8_REL_L2_MEAN = 2.0 ** -4


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def quantize_pool(batch):
    """Quantize every row of the batch's fp16 pools on the GPU; returns the
    fp8 pools and scales (device) after one pa_kv_cache_write_fp8 per pool."""
    NB, bs, H, D = batch.k_cache.shape
    k8 = torch.zeros((NB, bs, H, D), dtype=torch.uint8, device=DEV)
    v8 = torch.zeros_like(k8)
    ks = torch.ones((NB, H, bs), dtype=torch.float32, device=DEV)
    vs = torch.ones_like(ks)
    rows_k = batch.k_cache.to(DEV).reshape(NB * bs, H, D)
    rows_v = batch.v_cache.to(DEV).reshape(NB * bs, H, D)
    slots = torch.arange(NB * bs, dtype=torch.int64, device=DEV)
    status = zero_status(DEV)
    pk.pa_kv_cache_write_fp8(rows_k, rows_v, slots, k8, v8, ks, vs, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return k8, v8, ks, vs


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 4), (128, 32)])
def test_fp8_write_bit_exact(D, bs):
    H, nb = 3, 9
    gen = torch.Generator().manual_seed(80 + D)
    k = (torch.randn((20, H, D), generator=gen) * 3).half()
    v = torch.randn((20, H, D), generator=gen).half()
    v[4, 2] = 0  # all-zero row
    k[7, 0, 5] = 60000.0  # large value stays finite
    slots = torch.from_numpy(np.random.default_rng(D + bs).choice(nb * bs, 20, replace=False))
    slots[3] = -1
    k8 = torch.zeros((nb, bs, H, D), dtype=torch.uint8)
    ks = torch.full((nb, H, bs), 7.0)
    rk8, rv8, rks, rvs = oracle.kv_cache_write_fp8(k.numpy(), v.numpy(), slots.numpy(),
                                                   k8.numpy(), k8.numpy(), ks.numpy(), ks.numpy())
    g = [t.to(DEV) for t in (k8, k8.clone(), ks, ks.clone())]
    status = zero_status(DEV)
    pk.pa_kv_cache_write_fp8(k.to(DEV), v.to(DEV), slots.to(DEV), *g, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(g[0].cpu().numpy(), rk8) and np.array_equal(g[1].cpu().numpy(), rv8)
    assert np.array_equal(g[2].cpu().numpy(), rks) and np.array_equal(g[3].cpu().numpy(), rvs)


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 16), (128, 32), (128, 4), (128, 8), (64, 4), (64, 8), (64, 32)])
def test_fp8_decode_parity_and_accuracy(D, bs):
    ctx = [1, bs, bs + 1, 70, 333, 1024]
    batch = workloads.random_decode(len(ctx), 4, D, bs, ctx, seed=90 + D + bs, device="cpu")
    k8, v8, ks, vs = quantize_pool(batch)
    g = {"q": batch.q.to(DEV), "bt": batch.block_tables.to(DEV), "cl": batch.context_lens.to(DEV)}
    ref8 = oracle.decode_fp8(batch.q.numpy(), k8.cpu().numpy(), v8.cpu().numpy(),
                             ks.cpu().numpy(), vs.cpu().numpy(), batch.block_tables.numpy(),
                             batch.context_lens.numpy(), batch.scale)
    for pt in (0, bs, 8 * bs):
        out = pk.pa_decode_fp8(g["q"], k8, v8, ks, vs, g["bt"], g["cl"], batch.scale, 1024,
                               partition_tokens=pt)
        assert_close(out, ref8, what=f"fp8 decode D={D} bs={bs} pt={pt}")
    ref16 = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                          batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    got = out.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref16, axis=-1) / np.linalg.norm(ref16, axis=-1)
    print(f"fp8 vs fp16 data, D={D} bs={bs}: relative L2 max {rel.max():.3e} mean {rel.mean():.3e}")
    assert rel.max() <= FP8_REL_L2_MAX and rel.mean() <= FP8_REL_L2_MEAN


@pytest.mark.parametrize("H,bs", [(3, 16), (5, 32), (1, 4)])
def test_fp8_decode_odd_head_count(H, bs):
    # an odd head count: one head per warp (even counts pair adjacent heads)
    ctx = [1, 15, 16, 17, 300, 777]
    batch = workloads.random_decode(len(ctx), H, 128, bs, ctx, seed=95 + H, device="cpu")
    k8, v8, ks, vs = quantize_pool(batch)
    ref8 = oracle.decode_fp8(batch.q.numpy(), k8.cpu().numpy(), v8.cpu().numpy(),
                             ks.cpu().numpy(), vs.cpu().numpy(), batch.block_tables.numpy(),
                             batch.context_lens.numpy(), batch.scale)
    for pt in (0, 2 * bs):
        out = pk.pa_decode_fp8(batch.q.to(DEV), k8, v8, ks, vs, batch.block_tables.to(DEV),
                               batch.context_lens.to(DEV), batch.scale, 777, partition_tokens=pt)
        assert_close(out, ref8, what=f"fp8 decode H={H} bs={bs} pt={pt}")


def test_fp8_llama13b_batch():
    batch = workloads.llama13b_decode(seed=1, device=DEV)
    k8, v8, ks, vs = quantize_pool(batch)
    out = pk.pa_decode_fp8(batch.q, k8, v8, ks, vs, batch.block_tables, batch.context_lens,
                           batch.scale, 2048)
    sel = np.arange(0, 38, 4)
    ref8 = oracle.decode_fp8(batch.q.cpu().numpy()[sel], k8.cpu().numpy(), v8.cpu().numpy(),
                             ks.cpu().numpy(), vs.cpu().numpy(),
                             batch.block_tables.cpu().numpy()[sel],
                             batch.context_lens.cpu().numpy()[sel], batch.scale)
    assert_close(out[torch.from_numpy(sel).to(DEV)], ref8, what="fp8 llama13b")


def test_fp8_decode_score_spikes():
    # e4m3 keys whose scores jump by up to 60 nats across partitions (the
    # spike rows quantize with their own per-(token, head) scale)
    batch = spiked_decode_batch(128, 16, seed=95)
    k8, v8, ks, vs = quantize_pool(batch)
    ref8 = oracle.decode_fp8(batch.q.numpy(), k8.cpu().numpy(), v8.cpu().numpy(),
                             ks.cpu().numpy(), vs.cpu().numpy(), batch.block_tables.numpy(),
                             batch.context_lens.numpy(), batch.scale)
    assert np.all(np.isfinite(ref8))
    g = {"q": batch.q.to(DEV), "bt": batch.block_tables.to(DEV), "cl": batch.context_lens.to(DEV)}
    for pt in (0, 16, 128):
        status = zero_status(DEV)
        out = pk.pa_decode_fp8(g["q"], k8, v8, ks, vs, g["bt"], g["cl"], batch.scale, 1024,
                               partition_tokens=pt, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(out, ref8, what=f"fp8 score spikes pt={pt}")
