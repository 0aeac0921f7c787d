"""Reference model of the prefix-caching block pool (test infrastructure only).

Semantics follow "2.1 PagedAttention" (infra-guide), section 9 "Source
walkthrough: KV Cache management in vLLM V1" (9.1 the KVCacheManager /
BlockPool split, 9.2 the doubly linked free queue, 9.3 reference counts and
free order), and "PagedAttention: Treating KV Memory Like Virtual Memory"
(lenatriestounderstand.com), section "A separate mechanism: automatic prefix
caching" and the salt paragraph of "Where the analogy stops":

* Every block is either in use (refcount > 0) or in the free queue, an
  ordered list.  New blocks are taken from its head.  When a request is
  freed, its blocks are visited in reverse order (tail first); each loses one
  reference, and those that reach zero go back to the queue: blocks without
  a hash to the head (reused first), blocks with a hash to the tail (evicted
  last, so cached blocks leave oldest-first).  Freeing does not clear a
  block, and a free hashed block keeps its hash until it is taken again.
* A block is hashed when it fills.  Its hash covers the previous block's
  hash, the block's token ids and, for a request's first block, the request's
  salt, so the hashes of a request's blocks form a chain and a block's
  identity is the whole prefix up to it.  The table of cached blocks maps a
  hash to the block holding that content, in use or free.
* A lookup finds the longest run of a prompt's leading full blocks whose
  chain is in the table, and a hit is not copied: touch() takes a free hit
  block out of the queue and adds one reference.  Only full blocks are ever
  shared, so no block is written while shared and nothing is copied on write.

Readings where the pages leave a step open (each is plain):
* Hash: FNV-1a 64 (Fowler, Noll, Vo; offset basis 14695981039346656037,
  prime 1099511628211) over the bytes of the previous block's hash as a
  little-endian 64-bit word (for the first block: the salt, 0 when the request
  has none) followed by each token id as a little-endian 32-bit word.  A hit
  also compares the stored token ids and previous hash, so a collision can
  only cost a hit, never return wrong content.
* The last prompt token is always computed (its step produces the next
  token), so at most (n - 1) // block_size blocks of an n-token prompt hit:
  a 2,407-token prompt at 16 tokens per block finds 150 blocks, 2,400 tokens.
* A block that fills with content some cached block already holds is not
  registered a second time; it stays unhashed and is freed to the head.
* prepend to the head keeps the group's order: the first freed block without
  a hash becomes the new head.
* A request that needs more new blocks than the queue holds (after its hits
  are taken out) raises OutOfBlocks and changes nothing.
"""
import struct

from .allocator import OutOfBlocks

FNV_OFFSET = 14695981039346656037
FNV_PRIME = 1099511628211
MASK64 = (1 << 64) - 1


def fnv1a64(data, h=FNV_OFFSET):
    for byte in data:
        h ^= byte
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(prev, tokens):
    """Hash of a full block given the previous block's hash (or the salt for
    a request's first block) and the block's token ids."""
    data = struct.pack("<Q", prev & MASK64) + b"".join(struct.pack("<i", int(t)) for t in tokens)
    return fnv1a64(data)


class PrefixCachePoolModel:
    def __init__(self, num_blocks, block_size, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(order)             # head is free[0]
        self.refs = [0] * num_blocks
        self.hash_of = [None] * num_blocks  # hash of a cached block's content
        self.content = [None] * num_blocks  # (previous hash, token ids) of a cached block
        self.cached = {}                    # hash -> block
        self.tables = {}
        self.tokens = {}                    # seq -> token ids written so far
        self.chain = {}                     # seq -> hashes of its full blocks
        self.salts = {}

    # -- hashing ----------------------------------------------------------
    def _find(self, prev, toks):
        h = block_hash(prev, toks)
        b = self.cached.get(h)
        if b is None or self.content[b] != (prev, tuple(toks)):
            return h, None
        return h, b

    def lookup(self, tokens, salt=0):
        """Number of blocks in the longest cached run of the prompt's leading
        full blocks (at most (n - 1) // block_size of them)."""
        return len(self.hits(tokens, salt))

    def hits(self, tokens, salt=0):
        """The blocks of that run."""
        B = self.block_size
        hits, prev = [], salt
        for i in range(max(0, (len(tokens) - 1) // B)):
            h, b = self._find(prev, tokens[i * B:(i + 1) * B])
            if b is None:
                break
            hits.append(b)
            prev = h
        return hits

    def _register(self, seq, i):
        """Block i of seq just filled: hash it and cache it unless the same
        content is cached already."""
        B = self.block_size
        prev = self.chain[seq][i - 1] if i > 0 else self.salts[seq]
        toks = tuple(self.tokens[seq][i * B:(i + 1) * B])
        h, b = self._find(prev, toks)
        self.chain[seq].append(h)
        blk = self.tables[seq][i]
        if b is None and h not in self.cached:
            self.cached[h] = blk
            self.hash_of[blk] = h
            self.content[blk] = (prev, toks)

    def _take(self):
        blk = self.free.pop(0)
        h = self.hash_of[blk]
        if h is not None:  # evicted: its content is about to be overwritten
            del self.cached[h]
            self.hash_of[blk] = None
            self.content[blk] = None
        self.refs[blk] = 1
        return blk

    def _touch(self, blocks):
        for blk in blocks:
            if self.refs[blk] == 0:
                self.free.remove(blk)
            self.refs[blk] += 1

    # -- requests ---------------------------------------------------------
    def add_request(self, seq, tokens, salt=0):
        """New request with its prompt: hit blocks are shared, the rest get
        new blocks.  Returns (number of cached tokens, slot of every prompt
        position)."""
        if seq in self.tables:
            raise KeyError(f"sequence {seq} already exists")
        B = self.block_size
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        hits = self.hits(tokens, salt)
        need = -(-n // B) - len(hits)
        free_hits = sum(1 for b in set(hits) if self.refs[b] == 0)
        if need > len(self.free) - free_hits:
            raise OutOfBlocks(f"need {need} blocks, {len(self.free) - free_hits} free")
        self._touch(hits)
        table = hits + [self._take() for _ in range(need)]
        self.tables[seq] = table
        self.tokens[seq] = tokens
        self.salts[seq] = salt
        self.chain[seq] = []
        prev = salt
        for b in hits:
            h = self.hash_of[b]
            self.chain[seq].append(h)
            prev = h
        for i in range(len(hits), n // B):
            self._register(seq, i)
        slots = [table[p // B] * B + p % B for p in range(n)]
        return len(hits) * B, slots

    def append(self, seq, token):
        """One generated token; returns its slot."""
        B = self.block_size
        L = len(self.tokens[seq])
        if L % B == 0:
            if not self.free:
                raise OutOfBlocks("no free block")
            self.tables[seq].append(self._take())
        self.tokens[seq].append(int(token))
        if (L + 1) % B == 0:
            self._register(seq, L // B)
        return self.tables[seq][L // B] * B + L % B

    def release(self, seq):
        table = self.tables.pop(seq)
        del self.tokens[seq], self.chain[seq], self.salts[seq]
        to_free = []
        for blk in reversed(table):
            self.refs[blk] -= 1
            if self.refs[blk] == 0:
                to_free.append(blk)
        no_hash = [b for b in to_free if self.hash_of[b] is None]
        has_hash = [b for b in to_free if self.hash_of[b] is not None]
        self.free = no_hash + self.free + has_hash

    # -- views ------------------------------------------------------------
    def table(self, seq):
        return list(self.tables[seq])

    def length(self, seq):
        return len(self.tokens[seq])

    def free_list(self):
        return list(self.free)

    def refcount(self, blk):
        return self.refs[blk]

    def block_hash(self, blk):
        return self.hash_of[blk]
