"""Reference block allocator in plain Python.

TEST INFRASTRUCTURE (see the package docstring).

The cache lives in fixed-size blocks handed out as a sequence grows, with a
per-sequence table from positions to blocks, and sequences that share a
prefix share its blocks ("Serving", section 23.4 Paged Attention); a write
into a shared block copies it first ("Paged Attention: Managing the KV Cache
Like Virtual Memory", inference-serving tag page: sharing with copy-on-write).

The policy details the pages leave open are fixed as follows (the CUDA
library's host allocator must reproduce them bit for bit):
  * free list = FIFO queue, initially ``free_order`` (default 0..N-1);
    allocation pops the front, a block whose count reaches 0 is appended;
  * token p of a sequence: p % bs == 0 takes a new block; otherwise a last
    block with count > 1 is copied on write (new block, old count - 1);
  * fork copies the parent's table and length, every count + 1;
  * free releases the table's blocks in table order;
  * out of blocks -> ``MemoryError`` and no state change.
"""
from collections import deque


class ReferenceAllocator:
    def __init__(self, num_blocks, block_size=16, free_order=None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free_order must be a permutation"
        self.free = deque(order)
        self.refcount = [0] * num_blocks
        self.tables = {}
        self.lengths = {}

    def seq_add(self, seq):
        if seq < 0 or seq in self.tables:
            raise ValueError("bad or duplicate sequence id")
        self.tables[seq] = []
        self.lengths[seq] = 0

    def fork(self, parent, child):
        if parent not in self.tables or child in self.tables or child < 0:
            raise ValueError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def append_slot(self, seq):
        """Returns (slot, cow_src, cow_dst); cow_* are -1 without a copy."""
        table = self.tables[seq]
        pos = self.lengths[seq]
        bs = self.block_size
        cow = (-1, -1)
        if pos % bs == 0:
            if not self.free:
                raise MemoryError("no free block")
            b = self.free.popleft()
            self.refcount[b] = 1
            table.append(b)
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                if not self.free:
                    raise MemoryError("no free block")
                b = self.free.popleft()
                self.refcount[last] -= 1
                self.refcount[b] = 1
                table[-1] = b
                cow = (last, b)
        self.lengths[seq] = pos + 1
        slot = table[pos // bs] * bs + pos % bs
        return slot, cow[0], cow[1]

    def seq_free(self, seq):
        for b in self.tables.pop(seq):
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.lengths[seq]

    def table(self, seq):
        return list(self.tables[seq])

    def num_free(self):
        return len(self.free)
