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

  * azimuth.plus summary, section "vLLM": under memory pressure the scheduler pauses
    a request by moving its blocks to CPU memory (swap) and brings them back later.

Readings where the pages are silent:
  * the initial free list is an explicit permutation (a seeded shuffle of the pool);
    allocation pops its last element;
  * a write into a block whose ref_count is 1 happens in place, so the last holder
    of a once-shared block does not copy it;
  * OOM leaves every piece of state unchanged;
  * freeing a sequence walks its table from logical block 0 upwards;
  * the slot of a token is physical_block * block_size + offset.
  * swapping moves whole sequences: each distinct block they hold (sequence order,
    then table order) gets one block of the other pool, taken from the end of that
    pool's free list; the host pool's free list starts as 0..H-1; a block another
    resident sequence still holds keeps its data there, the swapped sequences get
    their own copy; released blocks go to the end of their free list in release
    order; a swapped-out sequence cannot grow or be forked until it is swapped in.
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
        self.swapped: Dict[int, bool] = {}
        self.host_free: List[int] = []
        self.host_ref: List[int] = []
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
        if self.swapped.get(parent):
            raise ValueError("a swapped-out sequence cannot be forked")
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
        if self.swapped.get(seq):
            raise ValueError("a swapped-out sequence cannot grow")
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
        on_host = self.swapped.pop(seq, False)
        for b in self.tables.pop(seq):
            if on_host:
                self.host_ref[b] -= 1
                if self.host_ref[b] == 0:
                    self.host_free.append(b)
            else:
                self._release(b)
        del self.lengths[seq]

    # -- swap space (summary section "vLLM") -------------------------------------
    def set_host_pool(self, num_host_blocks: int) -> None:
        if any(self.swapped.values()):
            raise ValueError("sequences are swapped out")
        self.host_free = list(range(num_host_blocks))
        self.host_ref = [0] * num_host_blocks

    def swap_out(self, seqs: Sequence[int]) -> List[Tuple[int, int]]:
        """Move the sequences to the host pool; (device block, host block) copies."""
        return self._move(seqs, to_host=True)

    def swap_in(self, seqs: Sequence[int]) -> List[Tuple[int, int]]:
        """Move the sequences back; (host block, device block) copies."""
        return self._move(seqs, to_host=False)

    def _move(self, seqs: Sequence[int], to_host: bool) -> List[Tuple[int, int]]:
        seqs = [int(q) for q in seqs]
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence is listed twice")
        for q in seqs:
            if q not in self.tables or self.swapped.get(q, False) == to_host:
                raise ValueError(f"sequence {q} is not live in the source pool")
        if to_host:
            src_ref, src_free, dst_ref, dst_free = self.ref, self.free, self.host_ref, self.host_free
        else:
            src_ref, src_free, dst_ref, dst_free = self.host_ref, self.host_free, self.ref, self.free
        distinct: List[int] = []
        seen = set()
        for q in seqs:
            for b in self.tables[q]:
                if b not in seen:
                    seen.add(b)
                    distinct.append(b)
        if len(distinct) > len(dst_free):
            raise OracleOOM("no free block in the target pool")
        copy_of = {b: dst_free.pop() for b in distinct}
        for q in seqs:
            table = self.tables[q]
            for j, b in enumerate(table):
                dst_ref[copy_of[b]] += 1
                src_ref[b] -= 1
                if src_ref[b] == 0:
                    src_free.append(b)
                table[j] = copy_of[b]
            self.swapped[q] = to_host
        return [(b, copy_of[b]) for b in distinct]

    # -- accounting: summary sections "Results" (waste) and "Memory sharing" ------
    def usage(self) -> Dict[str, int]:
        """used_blocks, logical_blocks, token_slots, tokens over resident sequences
        (tokens: for each used block, the most rows any holder has filled)."""
        filled: Dict[int, int] = {}
        logical = 0
        resident = swapped = 0
        for seq, table in self.tables.items():
            if self.swapped.get(seq):
                swapped += 1
                continue
            resident += 1
            logical += len(table)
            T = self.lengths[seq]
            for j, b in enumerate(table):
                rows = min(self.block_size, T - j * self.block_size)
                filled[b] = max(filled.get(b, 0), rows)
        used = sum(1 for r in self.ref if r > 0)
        return {"used_blocks": used, "logical_blocks": logical, "token_slots": used * self.block_size,
                "tokens": sum(filled.values()), "resident_seqs": resident, "swapped_seqs": swapped}

    def is_swapped(self, seq: int) -> bool:
        return bool(self.swapped.get(seq, False))

    def host_refcount(self, block: int) -> int:
        return self.host_ref[block]

    def num_free_host(self) -> int:
        return len(self.host_free)

    def host_free_list(self) -> List[int]:
        return list(self.host_free)

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
