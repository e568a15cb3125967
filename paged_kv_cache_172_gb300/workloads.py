"""Seeded synthetic inputs for the paged-attention workloads.

This module is the one piece shared by the oracle side and the CUDA side:
it draws random numbers and lays out block tables, and holds none of the
attention arithmetic.  Values are fp16 N(0, 1) drawn with a seeded
``torch.Generator`` on the requested device; structure (context lengths,
block permutations, tails) is drawn with ``numpy.random.default_rng(seed)``
so that it is identical on every machine.

Block tables follow the allocation pattern of the study notes
"DataWhale组队学习笔记--llm-algo-leetcode(五)" ("代码实现": blocks are taken from the
front of a free list), with the free list shuffled by the seed so that the
physical ids of a sequence are non-contiguous.  Sequences are allocated in
order, each taking ceil(len / block_size) blocks; unused table entries are
-1 (the sentinel of the blog "PagedAttention origin and evolution",
sec. 3.2.2).

Workloads (sizes as stated for each builder):
  tiny_schedule     -- 4 sequences, 4 heads, head_dim 64, block_size 4, 64
                       blocks; prompts {6,6,4,4} then {0,3,0,1} decode steps;
  llama13b_decode   -- 38 sequences, 40 heads, head_dim 128, block_size 16,
                       context lengths uniform in [128, 2048], pool 1.2x need,
                       plus one new token per sequence to write;
  prefix_sharing    -- 16 prompts x 8 samples, 1024-token prompts shared,
                       private tails uniform in [1, 512], one copy-on-write
                       block per sample;
  long_context      -- 1 sequence of 1,048,576 tokens over 65,536 permuted
                       blocks;
  chunked_prefill   -- 8 sequences, 3,584 cached tokens + a 512-query chunk.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import math

import numpy as np
import torch

__all__ = [
    "PagedBatch", "TinySchedule", "tiny_schedule", "llama13b_decode",
    "prefix_sharing", "prefix_sharing_layout", "SharingLayout",
    "llama13b_context_lens", "long_context", "chunked_prefill", "random_decode",
    "sharing_groups", "fork_forest_layout",
    "random_prefill", "shuffled_pool", "fill_tables",
]


@dataclass
class PagedBatch:
    """A paged KV pool plus the per-sequence views onto it.

    q            [B, H, D] (decode) or [B, H, Lq, D] (prefill chunk), fp16
    k_cache      [num_blocks, block_size, H, D] fp16
    v_cache      same shape as k_cache
    block_tables [B, max_blocks] int32, -1 past each sequence's blocks
    context_lens [B] int32, keys per sequence including any new tokens
    k_new/v_new  [T, H, D] fp16 tokens to write before attention (or None)
    slot_mapping [T] int64 flat slots (physical * block_size + offset)
    copy_pairs   [N, 2] int64 (src, dst) blocks to copy before attention
    """
    name: str
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    scale: float
    block_size: int
    k_new: Optional[torch.Tensor] = None
    v_new: Optional[torch.Tensor] = None
    slot_mapping: Optional[torch.Tensor] = None
    copy_pairs: Optional[torch.Tensor] = None
    meta: Dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return self.k_cache.shape[0]

    @property
    def H(self) -> int:
        return self.k_cache.shape[2]

    @property
    def D(self) -> int:
        return self.k_cache.shape[3]

    @property
    def B(self) -> int:
        return self.q.shape[0]


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn16(shape, gen, device):
    """fp16 N(0,1) values from a seeded generator."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float16)


def shuffled_pool(num_blocks: int, rng: np.random.Generator) -> np.ndarray:
    """A seeded permutation of the physical block ids: the free list."""
    return rng.permutation(num_blocks).astype(np.int64)


def fill_tables(lengths: List[int], block_size: int, free_order: np.ndarray,
                max_blocks: int) -> np.ndarray:
    """Block tables for sequences allocated in order from the front of
    ``free_order``; each takes ceil(len / block_size) blocks."""
    tables = np.full((len(lengths), max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(lengths):
        nblk = -(-int(n) // block_size)
        tables[b, :nblk] = free_order[pos:pos + nblk]
        pos += nblk
    return tables


def _slots(tables: np.ndarray, seq: np.ndarray, positions: np.ndarray,
           block_size: int) -> np.ndarray:
    return (tables[seq, positions // block_size].astype(np.int64) * block_size
            + positions % block_size)


# --------------------------------------------------------------------------
# tiny: 4 sequences, allocator replay (prefill then decode growth)
# --------------------------------------------------------------------------
@dataclass
class TinySchedule:
    """Inputs of the tiny replay.  Tables are NOT precomputed: the replay
    runs an allocator over ``free_order``.  ``k_tok[b]``/``v_tok[b]`` hold
    the K/V of every position of sequence b ([final_len, H, D]);
    ``queries[r]`` is the [B, H, D] query batch attended after decode step r
    (step 0 = right after prefill)."""
    B: int
    H: int
    D: int
    block_size: int
    num_blocks: int
    free_order: np.ndarray
    prompt_lens: List[int]
    decode_steps: List[int]
    k_tok: List[torch.Tensor]
    v_tok: List[torch.Tensor]
    queries: List[torch.Tensor]
    scale: float


def tiny_schedule(seed: int = 0, device="cpu") -> TinySchedule:
    B, H, D, bs, NB = 4, 4, 64, 4, 64
    prompt_lens = [6, 6, 4, 4]
    decode_steps = [0, 3, 0, 1]
    rng = np.random.default_rng(seed)
    free_order = shuffled_pool(NB, rng)
    g = _gen(device, seed)
    final = [p + d for p, d in zip(prompt_lens, decode_steps)]
    k_tok = [randn16((n, H, D), g, device) for n in final]
    v_tok = [randn16((n, H, D), g, device) for n in final]
    steps = max(decode_steps)
    queries = [randn16((B, H, D), g, device) for _ in range(steps + 1)]
    return TinySchedule(B, H, D, bs, NB, free_order, prompt_lens, decode_steps,
                        k_tok, v_tok, queries, 1.0 / math.sqrt(D))


# --------------------------------------------------------------------------
# generic random decode / prefill batches (parity sweeps, ragged edges)
# --------------------------------------------------------------------------
def random_decode(B, H, D, block_size, context_lens, seed, device="cpu",
                  pool_factor=1.2, max_blocks=None, extra_blocks=0,
                  new_tokens=False, name="random_decode") -> PagedBatch:
    """Decode batch with the given context lengths.  With ``new_tokens``, the
    last position of every non-empty sequence is written by a cache write
    before attention (k_new/v_new/slot_mapping)."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    need = int(sum(-(-int(c) // block_size) for c in ctx))
    NB = max(1, int(math.ceil(pool_factor * need)) + extra_blocks)
    if max_blocks is None:
        max_blocks = max(1, max(-(-int(c) // block_size) for c in ctx) if len(ctx) else 1)
    free_order = shuffled_pool(NB, rng)
    tables = fill_tables(list(ctx), block_size, free_order, max_blocks)
    g = _gen(device, seed)
    k_cache = randn16((NB, block_size, H, D), g, device)
    v_cache = randn16((NB, block_size, H, D), g, device)
    q = randn16((B, H, D), g, device)
    batch = PagedBatch(name, q, k_cache, v_cache,
                       torch.from_numpy(tables).to(device),
                       torch.from_numpy(ctx.astype(np.int32)).to(device),
                       1.0 / math.sqrt(D), block_size,
                       meta={"seed": seed, "free_order": free_order})
    if new_tokens:
        seqs = np.nonzero(ctx > 0)[0]
        slots = _slots(tables, seqs, ctx[seqs] - 1, block_size)
        batch.k_new = randn16((len(seqs), H, D), g, device)
        batch.v_new = randn16((len(seqs), H, D), g, device)
        batch.slot_mapping = torch.from_numpy(slots).to(device)
    return batch


def random_prefill(B, H, D, block_size, Lq, context_lens, seed, device="cpu",
                   pool_factor=1.2, write_chunk=True,
                   name="random_prefill") -> PagedBatch:
    """Prefill batch: the last ``Lq`` positions of each sequence are the new
    chunk (queries q[B,H,Lq,D]); with ``write_chunk`` their K/V come as
    k_new/v_new [B*Lq, H, D] with slots, to be written before attention."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int64)
    assert (ctx >= Lq).all()
    need = int(sum(-(-int(c) // block_size) for c in ctx))
    NB = max(1, int(math.ceil(pool_factor * need)))
    max_blocks = max(-(-int(c) // block_size) for c in ctx)
    free_order = shuffled_pool(NB, rng)
    tables = fill_tables(list(ctx), block_size, free_order, max_blocks)
    g = _gen(device, seed)
    k_cache = randn16((NB, block_size, H, D), g, device)
    v_cache = randn16((NB, block_size, H, D), g, device)
    q = randn16((B, H, Lq, D), g, device)
    batch = PagedBatch(name, q, k_cache, v_cache,
                       torch.from_numpy(tables).to(device),
                       torch.from_numpy(ctx.astype(np.int32)).to(device),
                       1.0 / math.sqrt(D), block_size,
                       meta={"seed": seed, "Lq": Lq, "free_order": free_order})
    if write_chunk and Lq > 0:
        seqs = np.repeat(np.arange(B), Lq)
        pos = (ctx[seqs] - Lq) + np.tile(np.arange(Lq), B)
        batch.slot_mapping = torch.from_numpy(_slots(tables, seqs, pos, block_size)).to(device)
        batch.k_new = randn16((B * Lq, H, D), g, device)
        batch.v_new = randn16((B * Lq, H, D), g, device)
    return batch


# --------------------------------------------------------------------------
# the four large workloads
# --------------------------------------------------------------------------
def llama13b_context_lens(seed: int = 1) -> np.ndarray:
    """38 context lengths uniform in [128, 2048] (inclusive)."""
    rng = np.random.default_rng(seed)
    return rng.integers(128, 2048, size=38, endpoint=True)


def llama13b_decode(seed: int = 1, device="cpu", block_size: int = 16) -> PagedBatch:
    """LLaMA-13B-shaped decode: B=38, H=40, D=128, block_size=16 (or the
    given one), context lengths uniform in [128, 2048] (inclusive, counting
    the new token), pool sized ceil(1.2 x total blocks), one new token per
    sequence written at position ctx-1 before decode."""
    ctx = llama13b_context_lens(seed)
    return random_decode(38, 40, 128, block_size, ctx, seed, device=device,
                         max_blocks=2048 // block_size, new_tokens=True,
                         name="llama13b_decode_b38")


@dataclass
class SharingLayout:
    num_blocks: int
    tables: np.ndarray
    context_lens: np.ndarray
    pairs: np.ndarray
    free_order: np.ndarray
    prompt_blocks: List[np.ndarray]
    tails: np.ndarray
    prompts: int
    samples: int
    prompt_len: int
    block_size: int


def prefix_sharing_layout(seed: int = 2, prompts: int = 16, samples: int = 8,
                          prompt_len: int = 1024, max_tail: int = 512,
                          block_size: int = 16) -> SharingLayout:
    """Block tables of the prefix-sharing workload (no values).

    Each prompt (prompt_len tokens, a whole number of blocks) is allocated
    once; its samples share its logical blocks 0..n-2 and each receives a
    private copy of the last prompt block (the copy-on-write pair
    (prompt block, fresh block)); each sample's private tail of
    U[1, max_tail] tokens follows in fresh blocks.  Allocation order from
    the shuffled free list: all prompts, then per sample (prompt-major) its
    copy block and its tail blocks.  The pool is ceil(1.2 x blocks used)."""
    rng = np.random.default_rng(seed)
    P, S, bs = prompts, samples, block_size
    assert prompt_len % bs == 0
    pblk = prompt_len // bs
    tails = rng.integers(1, max_tail, size=P * S, endpoint=True)
    used = P * pblk + P * S + int(sum(-(-int(t) // bs) for t in tails))
    NB = int(math.ceil(1.2 * used))
    free_order = shuffled_pool(NB, rng)
    max_blocks = pblk + -(-max_tail // bs)
    tables = np.full((P * S, max_blocks), -1, dtype=np.int32)
    pos = 0
    prompt_blocks = []
    for p in range(P):
        prompt_blocks.append(free_order[pos:pos + pblk].copy())
        pos += pblk
    pairs = []
    for p in range(P):
        for s in range(S):
            b = p * S + s
            tables[b, :pblk] = prompt_blocks[p]
            cow = int(free_order[pos])
            pos += 1
            pairs.append((int(prompt_blocks[p][pblk - 1]), cow))
            tables[b, pblk - 1] = cow
            nt = -(-int(tails[b]) // bs)
            tables[b, pblk:pblk + nt] = free_order[pos:pos + nt]
            pos += nt
    ctx = (prompt_len + tails).astype(np.int32)
    return SharingLayout(NB, tables, ctx, np.asarray(pairs, dtype=np.int64),
                         free_order, prompt_blocks, tails, P, S, prompt_len, bs)


def sharing_groups(lay: "SharingLayout"):
    """CSR description of the prefix-sharing layout's groups: the samples of
    prompt p form group p; they share the prompt's blocks 0..n-2 (the last
    prompt block is each sample's private copy).  Returns numpy int32
    (seq_group[B], group_offsets[G+1], group_seqs[B], group_prefix_len[G])."""
    P, S = lay.prompts, lay.samples
    seq_group = np.repeat(np.arange(P, dtype=np.int32), S)
    offsets = (np.arange(P + 1, dtype=np.int32) * S).astype(np.int32)
    seqs = np.arange(P * S, dtype=np.int32)
    shared = lay.prompt_len - lay.block_size
    prefix = np.full(P, shared, dtype=np.int32)
    return seq_group, offsets, seqs, prefix


def fork_forest_layout(seed: int, B: int, block_size: int, max_blocks: int = 24,
                       p_root: float = 0.2):
    """Block tables of sequences forked from one another (beam search or
    parallel sampling), no values.  Sequence 0 is a root; sequence i > 0 is a
    new root with probability p_root, else it forks from a uniformly chosen
    earlier sequence at a uniform point k in [0, that sequence's full
    blocks]: it maps the parent's first k blocks and takes fresh blocks for
    the rest of its own length, uniform in [k+1, max_blocks] blocks.  Its
    context length ends uniformly inside its last block.  Physical ids come
    from a shuffled pool of exactly the blocks used.  Returns (tables
    [B, max_blocks] int32 padded with -1, context_lens [B] int32,
    num_blocks)."""
    rng = np.random.default_rng(seed)
    bs = block_size
    chains, ctx = [], []
    nxt = 0
    for i in range(B):
        if i == 0 or rng.random() < p_root:
            k, head = 0, []
        else:
            par = int(rng.integers(0, i))
            k = int(rng.integers(0, ctx[par] // bs, endpoint=True))
            head = chains[par][:k]
        n = int(rng.integers(max(k, 1), max_blocks, endpoint=True))
        if n == k:  # ends on the parent's blocks: take one fresh block
            n = k + 1
        chains.append(head + list(range(nxt, nxt + n - k)))
        nxt += n - k
        ctx.append((n - 1) * bs + int(rng.integers(1, bs, endpoint=True)))
    perm = rng.permutation(nxt).astype(np.int32)
    tables = np.full((B, max_blocks + 1), -1, dtype=np.int32)
    for i, c in enumerate(chains):
        tables[i, :len(c)] = perm[np.asarray(c, dtype=np.int64)]
    return tables, np.asarray(ctx, dtype=np.int32), nxt


def prefix_sharing(seed: int = 2, device="cpu", H: int = 40, D: int = 128,
                   **layout_kw) -> PagedBatch:
    """16 prompts x 8 samples = 128 sequences, H=40, D=128, block_size=16,
    1024-token shared prompts, private tails U[1, 512]; one copy-on-write
    pair per sample, to run before decode."""
    lay = prefix_sharing_layout(seed, **layout_kw)
    g = _gen(device, seed)
    bs = lay.block_size
    k_cache = randn16((lay.num_blocks, bs, H, D), g, device)
    v_cache = randn16((lay.num_blocks, bs, H, D), g, device)
    q = randn16((lay.prompts * lay.samples, H, D), g, device)
    return PagedBatch(f"prefix_sharing_{lay.prompts}x{lay.samples}", q, k_cache,
                      v_cache, torch.from_numpy(lay.tables).to(device),
                      torch.from_numpy(lay.context_lens).to(device),
                      1.0 / math.sqrt(D), bs,
                      copy_pairs=torch.from_numpy(lay.pairs).to(device),
                      meta={"seed": seed, "layout": lay})


def long_context(seed: int = 3, device="cpu", context_len: int = 1 << 20,
                 H: int = 40, D: int = 128, bs: int = 16) -> PagedBatch:
    """One sequence of ``context_len`` tokens over exactly
    context_len / block_size randomly permuted physical blocks."""
    rng = np.random.default_rng(seed)
    NB = -(-context_len // bs)
    free_order = shuffled_pool(NB, rng)
    tables = free_order.astype(np.int32).reshape(1, NB)
    g = _gen(device, seed)
    k_cache = randn16((NB, bs, H, D), g, device)
    v_cache = randn16((NB, bs, H, D), g, device)
    q = randn16((1, H, D), g, device)
    return PagedBatch(f"long_context_{context_len}", q, k_cache, v_cache,
                      torch.from_numpy(tables).to(device),
                      torch.tensor([context_len], dtype=torch.int32, device=device),
                      1.0 / math.sqrt(D), bs,
                      meta={"seed": seed, "free_order": free_order})


def chunked_prefill(seed: int = 4, device="cpu", block_size: int = 16) -> PagedBatch:
    """8 sequences, each a 512-query chunk appended to 3,584 cached tokens
    (context 4,096 = 256 blocks of 16), H=40, D=128; the chunk's K/V are
    written into the cache before attention."""
    return random_prefill(8, 40, 128, block_size, 512, [4096] * 8, seed, device=device,
                          name="chunked_prefill_8x512_on_3584")
