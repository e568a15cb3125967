"""pa_decode_append (cache write fused into decode) against the oracle's
cache write + decode, and against the two-call path on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, bits, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def new_token_batch(B, H, D, bs, ctx, seed):
    """Decode batch whose sequences all grow by one token (ctx >= 1): k_new/v_new
    [B,H,D] for position ctx-1 of every sequence."""
    batch = workloads.random_decode(B, H, D, bs, ctx, seed, device="cpu", new_tokens=True)
    assert batch.slot_mapping.numel() == B
    return batch


def append_vs_oracle(batch, max_ctx, pt=0):
    g = {k: getattr(batch, k).to(DEV) for k in ("q", "k_cache", "v_cache", "block_tables",
                                                "context_lens", "k_new", "v_new")}
    status = zero_status(DEV)
    out = pk.pa_decode_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"],
                              g["block_tables"], g["context_lens"], batch.scale, max_ctx,
                              partition_tokens=pt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc, vc = oracle.kv_cache_write(batch.k_new.numpy(), batch.v_new.numpy(),
                                   batch.slot_mapping.numpy(), batch.k_cache.numpy(),
                                   batch.v_cache.numpy())
    assert np.array_equal(bits(g["k_cache"]), kc) and np.array_equal(bits(g["v_cache"]), vc)
    ref = oracle.decode(batch.q.numpy(), kc, vc, batch.block_tables.numpy(),
                        batch.context_lens.numpy(), batch.scale)
    assert_close(out, ref, what=f"append bs={batch.block_size} pt={pt}")
    return out


@pytest.mark.parametrize("bs", [4, 16, 32])
def test_append_ragged(bs):
    # new token at a block start (ctx-1 % bs == 0), mid-block, first token, long
    ctx = [1, bs + 1, 2 * bs, 3 * bs - 1, 40 * bs + 1, 777]
    batch = new_token_batch(len(ctx), 5, 128, bs, ctx, seed=60 + bs)
    for pt in (0, bs, 8 * bs):
        append_vs_oracle(batch, max(ctx), pt)


def test_append_d64():
    batch = new_token_batch(3, 4, 64, 16, [17, 1, 300], seed=64)
    append_vs_oracle(batch, 300)


def test_append_equals_write_then_decode():
    batch = workloads.llama13b_decode(seed=1, device=DEV)
    g1 = {k: getattr(batch, k).clone() for k in ("k_cache", "v_cache")}
    out_fused = pk.pa_decode_append(batch.q, batch.k_new, batch.v_new, g1["k_cache"],
                                    g1["v_cache"], batch.block_tables, batch.context_lens,
                                    batch.scale, 2048)
    pk.pa_kv_cache_write(batch.k_new, batch.v_new, batch.slot_mapping, batch.k_cache,
                         batch.v_cache)
    out_two = pk.pa_decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                           batch.context_lens, batch.scale, 2048)
    torch.cuda.synchronize()
    assert torch.equal(g1["k_cache"], batch.k_cache) and torch.equal(g1["v_cache"], batch.v_cache)
    assert torch.equal(out_fused, out_two)


def test_append_llama13b_against_oracle():
    batch = workloads.llama13b_decode(seed=1, device="cpu")
    append_vs_oracle(batch, 2048)


def test_append_bad_block_flagged():
    batch = new_token_batch(2, 2, 128, 16, [40, 9], seed=65)
    g = {k: getattr(batch, k).to(DEV) for k in ("q", "k_cache", "v_cache", "block_tables",
                                                "context_lens", "k_new", "v_new")}
    before = g["k_cache"].clone()
    bt = g["block_tables"].clone()
    bt[0, 2] = -5  # the block holding position 39
    status = zero_status(DEV)
    pk.pa_decode_append(g["q"], g["k_new"], g["v_new"], g["k_cache"], g["v_cache"], bt,
                        g["context_lens"], batch.scale, 40, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_BLOCK_ID
    # sequence 0's token was not stored; sequence 1's was
    s1 = int(batch.slot_mapping[1])
    k_rows = g["k_cache"].view(-1, 2, 128)
    assert torch.equal(k_rows[s1], g["k_new"][1])
    s0 = int(batch.slot_mapping[0])
    assert torch.equal(k_rows[s0], before.view(-1, 2, 128)[s0])
