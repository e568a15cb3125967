"""Host block allocator of the paged KV cache (oracle side).

TEST INFRASTRUCTURE: the reference behaviour that the worked examples pin.

Follows the study notes "DataWhale组队学习笔记--llm-algo-leetcode(五)",
"代码实现" (KVCacheManager: free list = range(num_blocks) taken from the
front; prefill takes ceil(seq_len / block_size) blocks and raises an OOM
RuntimeError before taking any when the list is short; decode grows the
sequence by one token and takes one new block when the last one is full;
get_physical_cache concatenates the blocks and cuts to seq_len), the
tutorial "4. PagedAttention机制：vLLM的核心创新", section "Block管理策略"
(Block Table / Free List / Allocator; on completion every block returns to
the free list), and the same notes' "4. PagedAttention 带来的核心红利"
(sequences that share a prompt point at the same physical blocks; a new
physical block is taken only when one of them writes: copy-on-write).

Readings (pages silent or inexact):
  * growth: a new block is needed when seq_len > len(block_table) * bs after
    the increment (the notes' ``seq_len % bs == 1`` test says the same for
    bs >= 2 and never fires for bs == 1);
  * a decode OOM leaves the sequence unchanged (the notes leave seq_len
    incremented; no test on the pages observes it);
  * the free list may start in any order (a seeded shuffle gives the
    non-contiguous physical ids of the synthetic workloads); it is FIFO;
  * shared blocks carry a reference count; a block returns to the free list
    when its count reaches zero.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple


class OutOfBlocks(RuntimeError):
    """Raised with a message containing "OOM" when the free list is short."""


@dataclass
class Sequence_:
    seq_id: int
    seq_len: int
    block_table: List[int] = field(default_factory=list)


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Sequence[int]] = None):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("num_blocks >= 0 and block_size > 0 required")
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else list(free_order)
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool")
        self.free_blocks: List[int] = order
        self.refcount = [0] * num_blocks

    # -- allocation ------------------------------------------------------
    def _take(self) -> int:
        blk = self.free_blocks.pop(0)
        self.refcount[blk] = 1
        return blk

    def blocks_needed(self, seq_len: int) -> int:
        return (seq_len + self.block_size - 1) // self.block_size

    def allocate_for_prefill(self, seq: Sequence_) -> None:
        needed = self.blocks_needed(seq.seq_len) - len(seq.block_table)
        if needed > len(self.free_blocks):
            raise OutOfBlocks("OOM")
        for _ in range(max(needed, 0)):
            seq.block_table.append(self._take())

    def allocate_for_decode(self, seq: Sequence_) -> Optional[int]:
        """Grow by one token.  Returns the new physical block, or None when
        the token fits in the last block."""
        new_len = seq.seq_len + 1
        if new_len > len(seq.block_table) * self.block_size:
            if not self.free_blocks:
                raise OutOfBlocks("OOM")
            blk = self._take()
            seq.block_table.append(blk)
            seq.seq_len = new_len
            return blk
        seq.seq_len = new_len
        return None

    def free(self, seq: Sequence_) -> None:
        for blk in seq.block_table:
            self.refcount[blk] -= 1
            if self.refcount[blk] == 0:
                self.free_blocks.append(blk)
        seq.block_table = []

    # -- sharing -----------------------------------------------------------
    def fork(self, parent: Sequence_, child_id: int) -> Sequence_:
        """A new sequence that shares every block of ``parent``."""
        for blk in parent.block_table:
            self.refcount[blk] += 1
        return Sequence_(child_id, parent.seq_len, list(parent.block_table))

    def copy_on_write(self, seq: Sequence_, logical: int) -> Optional[Tuple[int, int]]:
        """Make logical block ``logical`` private to ``seq``.  Returns the
        (src, dst) pair the device copy must perform, or None when the
        block already has a single owner."""
        blk = seq.block_table[logical]
        if self.refcount[blk] <= 1:
            return None
        if not self.free_blocks:
            raise OutOfBlocks("OOM")
        new = self._take()
        self.refcount[blk] -= 1
        seq.block_table[logical] = new
        return (blk, new)

    # -- addressing --------------------------------------------------------
    def slot(self, seq: Sequence_, pos: int) -> int:
        """Flat slot of token position ``pos``: physical * bs + offset."""
        return seq.block_table[pos // self.block_size] * self.block_size + pos % self.block_size

    def wasted_slots(self, seq: Sequence_) -> int:
        return len(seq.block_table) * self.block_size - seq.seq_len

    def in_use(self) -> int:
        return sum(1 for c in self.refcount if c > 0)
