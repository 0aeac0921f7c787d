"""Reference model of the host block allocator (test infrastructure only).

Semantics follow "Why AI servers waste memory, and how paging fixes it"
(spicyshark.co), sections "The idea: a block table", "A hand-worked example",
"The real implementation" and "Sharing a prefix with copy-on-write":

* The pool is cut into num_blocks blocks of block_size token slots.  The free
  list is a FIFO: blocks are taken from the front and returned to the back.
  Freed blocks are not cleared.
* Each sequence owns a block table (physical block ids in logical order) and a
  token count.  Token position p lives in slot p % B of block table[p // B].
* Appending a token: if the sequence's token count is a multiple of B
  (including 0) the last block is full, so a block is taken from the front of
  the free list and appended to the table.  Otherwise, if the last block is
  shared (refcount > 1), it is copied into a freshly taken block, the old
  block's count drops by one and the table points at the copy
  (copy-on-write).  Then the token is written at offset count % B of the last
  block.  If a block is needed and the free list is empty, OutOfBlocks is
  raised before anything changes.
* Fork: the child gets a copy of the parent's table and token count, and
  every block in it gains one reference.  No key or value moves.
* Free: walk the table in order, drop one reference per block, and put a block
  at the back of the free list when its count reaches zero.

Extensions of the library, each a plain reading:
* append(seq, n) with n > 1 is the same as n single appends, but all or
  nothing: the free-list check covers the whole request before any change.
* The initial free-list order may be given (a seeded permutation of the block
  ids stands in for a pool whose blocks are scattered); the default is
  0 .. num_blocks-1 as on the page.
"""
from collections import deque


class OutOfBlocks(Exception):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks, block_size, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.refs = [0] * num_blocks
        self.tables = {}
        self.lengths = {}

    # -- sequences ---------------------------------------------------------
    def add(self, seq):
        if seq in self.tables:
            raise KeyError(f"sequence {seq} already exists")
        self.tables[seq] = []
        self.lengths[seq] = 0

    def _blocks_needed(self, seq, n):
        table, count = self.tables[seq], self.lengths[seq]
        needed = 0
        for i in range(n):
            pos = count + i
            if pos % self.block_size == 0:
                needed += 1
            elif i == 0 and self.refs[table[-1]] > 1:
                needed += 1
        return needed

    def _take(self):
        blk = self.free.popleft()
        assert self.refs[blk] == 0
        self.refs[blk] = 1
        return blk

    def append(self, seq, n=1):
        """Append n tokens.  Returns (slots, copies): the flat slot
        (block * B + offset) of each new token, and the (src, dst) block copies
        the device must do before writing them (at most one)."""
        if seq not in self.tables:
            raise KeyError(f"unknown sequence {seq}")
        if n < 0:
            raise ValueError("n must be >= 0")
        if self._blocks_needed(seq, n) > len(self.free):
            raise OutOfBlocks(seq)
        table = self.tables[seq]
        slots, copies = [], []
        for _ in range(n):
            count = self.lengths[seq]
            offset = count % self.block_size
            if offset == 0:
                table.append(self._take())
            elif self.refs[table[-1]] > 1:
                old = table[-1]
                new = self._take()
                copies.append((old, new))
                self.refs[old] -= 1
                table[-1] = new
            slots.append(table[-1] * self.block_size + offset)
            self.lengths[seq] = count + 1
        return slots, copies

    def fork(self, parent, child):
        if parent not in self.tables:
            raise KeyError(f"unknown sequence {parent}")
        if child in self.tables:
            raise KeyError(f"sequence {child} already exists")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for blk in self.tables[child]:
            self.refs[blk] += 1

    def release(self, seq):
        """Finish a sequence (the page's free(rid))."""
        if seq not in self.tables:
            raise KeyError(f"unknown sequence {seq}")
        for blk in self.tables.pop(seq):
            self.refs[blk] -= 1
            if self.refs[blk] == 0:
                self.free.append(blk)
        del self.lengths[seq]

    # -- queries -----------------------------------------------------------
    def table(self, seq):
        return list(self.tables[seq])

    def length(self, seq):
        return self.lengths[seq]

    def free_list(self):
        return list(self.free)

    def refcount(self, blk):
        return self.refs[blk]

    def wasted_slots(self):
        """Allocated slots minus stored tokens, summed over sequences (the
        "wasted" column of the page's hand-worked table, where no block is
        shared)."""
        return sum(len(t) * self.block_size - self.lengths[s] for s, t in self.tables.items())
