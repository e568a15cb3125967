"""Parity of pa_decode (and the cache write feeding it) with the fp64 oracle.

All through the C ABI on cuda:0, on seeded inputs from the shared workload
generator: the tiny allocator replay, a sweep of head_dim x block_size with
ragged context lengths and several partition sizes, the 38-sequence
LLaMA-13B-shaped batch, the prefix-sharing batch and the 1M-token context.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_172_gb300 as pk
from oracle.allocator import BlockAllocator, Sequence_
from paged_kv_cache_172_gb300 import workloads
from pk_testutil import assert_close, bits, errors, spiked_decode_batch, to_dev, zero_status

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(DEV)


def run_decode(g, scale, max_ctx, pt=0, status=None, out=None):
    return pk.pa_decode(g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                        g["context_lens"], scale, max_context_len=max_ctx,
                        partition_tokens=pt, status=status, out=out)


# ----------------------------------------------------------------------------
# tiny replay: allocator growth, cache writes and decode at every step
# ----------------------------------------------------------------------------
def test_tiny_replay():
    sch = workloads.tiny_schedule(seed=0, device="cpu")
    alloc = BlockAllocator(sch.num_blocks, sch.block_size, sch.free_order)
    seqs = [Sequence_(b, p) for b, p in enumerate(sch.prompt_lens)]
    kc_ref = np.zeros((sch.num_blocks, sch.block_size, sch.H, sch.D), np.float16)
    vc_ref = np.zeros_like(kc_ref)
    kc = torch.zeros(kc_ref.shape, dtype=torch.float16, device=DEV)
    vc = torch.zeros_like(kc)
    status = zero_status(DEV)
    maxb = 4

    def write(tokens):  # tokens: list of (seq, position)
        slots = np.array([alloc.slot(seqs[b], p) for b, p in tokens], np.int64)
        kn = torch.stack([sch.k_tok[b][p] for b, p in tokens])
        vn = torch.stack([sch.v_tok[b][p] for b, p in tokens])
        nonlocal kc_ref, vc_ref
        kc_ref, vc_ref = oracle.kv_cache_write(kn.numpy(), vn.numpy(), slots, kc_ref, vc_ref)
        kc_ref, vc_ref = kc_ref.view(np.float16), vc_ref.view(np.float16)
        pk.pa_kv_cache_write(kn.to(DEV), vn.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc,
                             status=status)

    def attend(r):
        tables = np.full((sch.B, maxb), -1, np.int32)
        for b, s in enumerate(seqs):
            tables[b, :len(s.block_table)] = s.block_table
        ctx = np.array([s.seq_len for s in seqs], np.int32)
        q = sch.queries[r]
        ref = oracle.decode(q.numpy(), kc_ref, vc_ref, tables, ctx, sch.scale)
        g = {"q": q.to(DEV), "k_cache": kc, "v_cache": vc,
             "block_tables": torch.from_numpy(tables).to(DEV),
             "context_lens": torch.from_numpy(ctx).to(DEV)}
        for pt in (0, 4):
            out = run_decode(g, sch.scale, 16, pt=pt, status=status)
            assert_close(out, ref, what=f"round {r} partition {pt}")

    for s in seqs:
        alloc.allocate_for_prefill(s)
    write([(b, p) for b, s in enumerate(seqs) for p in range(s.seq_len)])
    # the notes' worked numbers: 6 tokens -> 2 blocks, 4 tokens -> 1 block
    assert [len(s.block_table) for s in seqs] == [2, 2, 1, 1]
    attend(0)
    for r in range(max(sch.decode_steps)):
        grown = []
        for b, s in enumerate(seqs):
            if r < sch.decode_steps[b]:
                alloc.allocate_for_decode(s)
                grown.append((b, s.seq_len - 1))
        write(grown)
        attend(r + 1)
    # 9th token took a 3rd block; length 5 took a 2nd block
    assert [s.seq_len for s in seqs] == [6, 9, 4, 5]
    assert [len(s.block_table) for s in seqs] == [2, 3, 1, 2]
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(kc), kc_ref.view(np.uint16))
    assert np.array_equal(bits(vc), vc_ref.view(np.uint16))


# ----------------------------------------------------------------------------
# sweep: head_dim x block_size x partition size, ragged lengths
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [4, 8, 16, 32])
def test_decode_sweep(D, bs):
    H = 5  # ragged head group (CTAs hold 4 heads)
    ctx = [0, 1, bs - 1, bs, bs + 1, 3 * bs + 2, 40 * bs + 7, 17, 250]
    maxb = -(-max(ctx) // bs)
    batch = workloads.random_decode(len(ctx), H, D, bs, ctx, seed=100 + D + bs, device="cpu",
                                    max_blocks=maxb + 2)
    ref = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                        batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    max_ctx = max(ctx)
    outs = {}
    for pt in (0, bs, 8 * bs, 32 * bs):
        out = run_decode(g, batch.scale, max_ctx, pt=pt, status=status)
        assert_close(out, ref, what=f"D={D} bs={bs} partition={pt}")
        outs[pt] = out
        assert torch.all(out[0] == 0)  # ctx == 0 row
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_decode_single_key_and_ones():
    batch = workloads.random_decode(3, 4, 128, 16, [1, 300, 33], seed=7, device="cpu")
    g = to_dev(batch, DEV)
    out = run_decode(g, batch.scale, 300, pt=32)
    # one key: output is that key's V row, rounded to fp16 (exactly itself)
    blk = int(batch.block_tables[0, 0])
    assert torch.equal(out[0].cpu(), batch.v_cache[blk, 0])
    g["v_cache"] = torch.ones_like(g["v_cache"])
    out1 = run_decode(g, batch.scale, 300, pt=32)
    assert torch.all(out1 == 1.0)


def test_decode_permutation_invariance_bit_exact():
    batch = workloads.random_decode(6, 8, 128, 16, [5, 77, 160, 1000, 2, 513], seed=8,
                                    device="cpu", extra_blocks=7)
    g = to_dev(batch, DEV)
    out = run_decode(g, batch.scale, 1000)
    perm = torch.randperm(batch.num_blocks, generator=torch.Generator().manual_seed(3))
    k2 = torch.empty_like(batch.k_cache)
    v2 = torch.empty_like(batch.v_cache)
    k2[perm] = batch.k_cache
    v2[perm] = batch.v_cache
    bt = batch.block_tables.long()
    t2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], torch.full_like(bt, -1)).int()
    g2 = dict(g, k_cache=k2.to(DEV), v_cache=v2.to(DEV), block_tables=t2.to(DEV))
    out2 = run_decode(g2, batch.scale, 1000)
    assert torch.equal(out, out2)


def test_decode_partition_consistency():
    batch = workloads.random_decode(4, 8, 128, 16, [2048, 1500, 700, 129], seed=9, device="cpu")
    g = to_dev(batch, DEV)
    a = run_decode(g, batch.scale, 2048, pt=512)
    b = run_decode(g, batch.scale, 2048, pt=128)
    c = run_decode(g, batch.scale, 2048, pt=16)
    assert (a.float() - b.float()).abs().max().item() <= 2e-3
    assert (a.float() - c.float()).abs().max().item() <= 2e-3


def test_decode_status_and_canaries():
    batch = workloads.random_decode(3, 4, 64, 16, [40, 20, 70], seed=10, device="cpu",
                                    max_blocks=6)
    g = to_dev(batch, DEV)
    # output written inside a larger buffer: the canaries around it stay intact
    big = torch.full((3 * 4 * 64 + 2 * 64,), 7.0, dtype=torch.float16, device=DEV)
    out = big[64:64 + 3 * 4 * 64].view(3, 4, 64)
    status = zero_status(DEV)
    run_decode(g, batch.scale, 70, status=status, out=out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.all(big[:64] == 7.0) and torch.all(big[-64:] == 7.0)
    # a needed table entry out of range: flagged, no fault
    bad = g["block_tables"].clone()
    bad[1, 0] = -1
    bad[2, 3] = batch.num_blocks + 5
    status.zero_()
    run_decode(dict(g, block_tables=bad), batch.scale, 70, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_BLOCK_ID
    # entries past ceil(ctx / bs) are never read
    junk = g["block_tables"].clone()
    junk[1, 2:] = 1 << 30
    status.zero_()
    a = run_decode(dict(g, block_tables=junk), batch.scale, 70, status=status)
    b = run_decode(g, batch.scale, 70)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(a, b)
    # context beyond the promised maximum: flagged and clamped
    status.zero_()
    run_decode(g, batch.scale, 48, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pk.PA_DEV_BAD_CONTEXT


# ----------------------------------------------------------------------------
# the full-size workloads
# ----------------------------------------------------------------------------
def test_llama13b_batch():
    batch = workloads.llama13b_decode(seed=1, device=DEV)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    pk.pa_kv_cache_write(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"],
                         status=status)
    out = run_decode(g, batch.scale, 2048, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc = batch.k_cache.cpu().numpy()
    vc = batch.v_cache.cpu().numpy()
    kc_ref, vc_ref = oracle.kv_cache_write(batch.k_new.cpu().numpy(), batch.v_new.cpu().numpy(),
                                           batch.slot_mapping.cpu().numpy(), kc, vc)
    assert np.array_equal(bits(g["k_cache"]), kc_ref)
    assert np.array_equal(bits(g["v_cache"]), vc_ref)
    ref = oracle.decode(batch.q.cpu().numpy(), kc_ref, vc_ref, batch.block_tables.cpu().numpy(),
                        batch.context_lens.cpu().numpy(), batch.scale)
    mx, mean = assert_close(out, ref, what="llama13b")
    print(f"llama13b decode max|err| {mx:.2e} mean {mean:.2e}")


def test_prefix_sharing_batch():
    batch = workloads.prefix_sharing(seed=2, device=DEV)
    lay = batch.meta["layout"]
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    kc0 = batch.k_cache.cpu().numpy()
    vc0 = batch.v_cache.cpu().numpy()
    pk.pa_block_copy(g["k_cache"], g["v_cache"], g["copy_pairs"], status=status)
    out = run_decode(g, batch.scale, int(lay.context_lens.max()), status=status)
    # shared tables (before the copy-on-write repointing) give identical bits
    shared = lay.tables.copy()
    for b in range(lay.prompts * lay.samples):
        shared[b, lay.prompt_len // lay.block_size - 1] = lay.pairs[b][0]
    out_shared = run_decode(dict(g, block_tables=torch.from_numpy(shared).to(DEV)),
                            batch.scale, int(lay.context_lens.max()))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, out_shared)
    kc_ref, vc_ref = oracle.block_copy(kc0, vc0, lay.pairs)
    assert np.array_equal(bits(g["k_cache"]), kc_ref)
    assert np.array_equal(bits(g["v_cache"]), vc_ref)
    # oracle on every 4th sequence (all heads): 32 of 128 sequences
    sel = np.arange(0, lay.prompts * lay.samples, 4)
    ref = oracle.decode(batch.q.cpu().numpy()[sel], kc_ref, vc_ref, lay.tables[sel],
                        lay.context_lens[sel], batch.scale)
    mx, mean = assert_close(out[torch.from_numpy(sel).to(DEV)], ref, what="prefix sharing")
    print(f"prefix sharing decode max|err| {mx:.2e} mean {mean:.2e}")


def test_long_context_1m():
    batch = workloads.long_context(seed=3, device=DEV)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    n = 1 << 20
    out = run_decode(g, batch.scale, n, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    table = batch.block_tables.cpu().numpy()[0]
    for h in (0, 17, 39):
        kh = batch.k_cache[:, :, h:h + 1, :].contiguous().cpu().numpy()
        vh = batch.v_cache[:, :, h:h + 1, :].contiguous().cpu().numpy()
        ref = oracle.attend_row(batch.q[0, h].cpu().numpy(), kh, vh, table, n, 0, batch.scale)
        got = out[0, h]
        mx, mean = errors(got, ref)
        rel = float(np.linalg.norm(got.float().cpu().numpy() - ref) / np.linalg.norm(ref))
        assert mx <= 5e-3 and mean <= 5e-4 and rel <= 1e-2, (h, mx, mean, rel)
        print(f"1M head {h}: max|err| {mx:.2e} rel {rel:.2e}")
    # V = 1 everywhere -> every output is exactly 1 after fp16 rounding
    g["v_cache"].fill_(1.0)
    out1 = run_decode(g, batch.scale, n)
    assert torch.all(out1 == 1.0)


def test_llama13b_batch_block32():
    """The same 38-sequence batch laid out in 32-token blocks (decode stages
    stream each block as two 16-token boxes)."""
    batch = workloads.llama13b_decode(seed=1, device=DEV, block_size=32)
    g = to_dev(batch, DEV)
    status = zero_status(DEV)
    out = run_decode(g, batch.scale, 2048, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sel = np.arange(0, 38, 3)
    ref = oracle.decode(batch.q.cpu().numpy()[sel], batch.k_cache.cpu().numpy(),
                        batch.v_cache.cpu().numpy(), batch.block_tables.cpu().numpy()[sel],
                        batch.context_lens.cpu().numpy()[sel], batch.scale)
    assert_close(out[torch.from_numpy(sel).to(DEV)], ref, what="llama13b bs=32")


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 8)])
def test_decode_score_spikes(D, bs):
    # partitions whose maxima differ by up to 60 nats: the per-partition
    # softmax and the log-sum-exp merge must keep every weight finite
    batch = spiked_decode_batch(D, bs, seed=70 + D + bs)
    ref = oracle.decode(batch.q.numpy(), batch.k_cache.numpy(), batch.v_cache.numpy(),
                        batch.block_tables.numpy(), batch.context_lens.numpy(), batch.scale)
    assert np.all(np.isfinite(ref))
    g = to_dev(batch, DEV)
    for pt in (0, bs, 8 * bs):
        status = zero_status(DEV)
        out = run_decode(g, batch.scale, 1024, pt=pt, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(out, ref, what=f"score spikes D={D} bs={bs} pt={pt}")
