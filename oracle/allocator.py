"""Reference block allocator -- TEST INFRASTRUCTURE ONLY (part of the oracle).

Written independently of the library's C++ allocator; tests require the two to
agree bit for bit (tables, reference counts, free-list order, slots, copy pairs).

Policy, from the pages:
  * CSDN tutorial "PagedAttention实战" §2.2 BlockManager: every page is created up
    front; the free list is a Python list; allocate pops from its END and raises
    MemoryError when it is empty; a page's ref_count rises on allocation; free
    decrements it and appends the page to the free list when it reaches 0.
  * same tutorial §3.1 SequenceManager.append_kv: token position p goes to logical
    page p // page_size at offset p % page_size; an unmapped logical page gets a
    freshly allocated physical page.
  * same tutorial §5.1 clone_sequence: a clone copies the page table and raises the
    ref_count of every shared page.
  * azimuth.plus PagedAttention summary, section "Memory sharing: copy-on-write":
    when a sequence must write into a block that other sequences share, only that
    block is copied to a new location and only the writer's table changes.  (The
    tutorial's append_kv writes into shared pages in place; the summary's
    copy-on-write rule is followed instead.)

Readings where the pages are silent:
  * the initial free list is an explicit permutation (a seeded shuffle of the pool);
    allocation pops its last element;
  * a write into a block whose ref_count is 1 happens in place, so the last holder
    of a once-shared block does not copy it;
  * OOM leaves every piece of state unchanged;
  * freeing a sequence walks its table from logical block 0 upwards;
  * the slot of a token is physical_block * block_size + offset.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple


class OracleOOM(MemoryError):
    """The tutorial's MemoryError("No free pages available")."""


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        if free_order is None:
            free = list(range(num_blocks))
        else:
            free = [int(x) for x in free_order]
            if sorted(free) != list(range(num_blocks)):
                raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free: List[int] = free
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lengths: Dict[int, int] = {}
        self._next_id = 0

    # -- tutorial §2.2 ---------------------------------------------------------
    def _allocate(self) -> int:
        if not self.free:
            raise OracleOOM("no free block")
        b = self.free.pop()
        self.ref[b] += 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequences -------------------------------------------------------------
    def new_seq(self) -> int:
        sid = self._next_id
        self._next_id += 1
        self.tables[sid] = []
        self.lengths[sid] = 0
        return sid

    def fork(self, parent: int) -> int:
        table = list(self.tables[parent])
        sid = self._next_id
        self._next_id += 1
        for b in table:
            self.ref[b] += 1
        self.tables[sid] = table
        self.lengths[sid] = self.lengths[parent]
        return sid

    def append(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow) with cow = (src_block, dst_block) when the target block
        was shared and had to be copied, else None."""
        table = self.tables[seq]
        pos = self.lengths[seq]
        logical, offset = divmod(pos, self.block_size)
        cow = None
        if logical == len(table):
            table.append(self._allocate())
        else:
            src = table[logical]
            if self.ref[src] > 1:
                dst = self._allocate()          # may raise: nothing changed yet
                self.ref[src] -= 1
                table[logical] = dst
                cow = (src, dst)
        self.lengths[seq] = pos + 1
        return table[logical] * self.block_size + offset, cow

    def free_seq(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lengths[seq]

    # -- views -----------------------------------------------------------------
    def block_table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def seq_len(self, seq: int) -> int:
        return self.lengths[seq]

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def num_free(self) -> int:
        return len(self.free)

    def free_list(self) -> List[int]:
        return list(self.free)
