"""The workload generator's block tables are the oracle allocator's tables
(same shuffled free list, same allocation order), and the drawn structure
matches the stated recipes."""
import numpy as np

from oracle.allocator import BlockAllocator, Sequence_
from paged_kv_cache_172_gb300 import workloads


def test_fill_tables_is_allocator_replay():
    rng = np.random.default_rng(0)
    lengths = [int(x) for x in rng.integers(1, 500, size=20)]
    bs = 16
    need = sum(-(-n // bs) for n in lengths)
    order = workloads.shuffled_pool(need + 9, rng)
    tables = workloads.fill_tables(lengths, bs, order, 40)
    alloc = BlockAllocator(need + 9, bs, order)
    for b, n in enumerate(lengths):
        s = Sequence_(b, n)
        alloc.allocate_for_prefill(s)
        row = tables[b]
        assert list(row[:len(s.block_table)]) == s.block_table
        assert np.all(row[len(s.block_table):] == -1)


def test_prefix_sharing_layout_is_fork_and_copy_on_write():
    lay = workloads.prefix_sharing_layout(seed=2)
    assert lay.prompts == 16 and lay.samples == 8 and lay.prompt_len == 1024
    assert lay.tails.min() >= 1 and lay.tails.max() <= 512
    alloc = BlockAllocator(lay.num_blocks, lay.block_size, lay.free_order)
    parents = []
    for p in range(lay.prompts):
        s = Sequence_(-1 - p, lay.prompt_len)
        alloc.allocate_for_prefill(s)
        parents.append(s)
    pblk = lay.prompt_len // lay.block_size
    pairs = []
    for p in range(lay.prompts):
        for k in range(lay.samples):
            b = p * lay.samples + k
            child = alloc.fork(parents[p], b)
            pairs.append(alloc.copy_on_write(child, pblk - 1))
            for _ in range(int(lay.tails[b])):
                alloc.allocate_for_decode(child)
            assert child.seq_len == lay.context_lens[b]
            row = lay.tables[b]
            assert list(row[:len(child.block_table)]) == child.block_table
            assert np.all(row[len(child.block_table):] == -1)
    assert np.array_equal(np.asarray(pairs), lay.pairs)
    # logical blocks 0..62 are shared by the 8 samples of a prompt
    assert alloc.refcount[parents[0].block_table[0]] == 1 + lay.samples
    assert alloc.refcount[parents[0].block_table[pblk - 1]] == 1
    assert lay.num_blocks == int(np.ceil(1.2 * alloc.in_use()))


def test_llama13b_lengths():
    ctx = workloads.llama13b_context_lens(seed=1)
    assert len(ctx) == 38 and ctx.min() >= 128 and ctx.max() <= 2048


def test_tiny_schedule_shapes():
    sch = workloads.tiny_schedule(seed=0)
    assert sch.prompt_lens == [6, 6, 4, 4] and sch.decode_steps == [0, 3, 0, 1]
    assert sorted(sch.free_order.tolist()) == list(range(64))
    assert [t.shape[0] for t in sch.k_tok] == [6, 9, 4, 5]
