"""Pins of the prefix-caching block pool (no GPU): the pages' worked numbers,
the free-order rule, the hash-chain rules and the published FNV-1a test
vectors.  Each scenario runs on the oracle's model and on the library's
native pool (pa_pcache_*); a randomised trace checks the two operation by
operation."""
import json
import os

import numpy as np
import pytest

from oracle.allocator import OutOfBlocks as ModelOutOfBlocks
from oracle.prefix_cache import PrefixCachePoolModel, block_hash, fnv1a64
from conftest import read_json


@pytest.fixture(params=["model", "native"])
def Pool(request):
    """The pool class under test and the exception it raises when out of
    blocks."""
    if request.param == "model":
        return PrefixCachePoolModel
    from paged_kv_cache_64_gb300 import api, build
    build.build()
    return api.PrefixCachePool


def out_of_blocks():
    from paged_kv_cache_64_gb300 import _lib
    return (ModelOutOfBlocks, _lib.OutOfBlocks)


def test_fnv1a64_published_vectors():
    # FNV-1a 64-bit test vectors (Fowler, Noll, Vo)
    assert fnv1a64(b"") == 0xcbf29ce484222325
    assert fnv1a64(b"a") == 0xaf63dc4c8601ec8c
    assert fnv1a64(b"foobar") == 0x85944171f73967e8


def test_block_hash_encoding():
    # previous hash as 8 little-endian bytes, then int32 little-endian token ids
    data = (7).to_bytes(8, "little") + (1).to_bytes(4, "little") + (-2 & 0xffffffff).to_bytes(4, "little")
    assert block_hash(7, [1, -2]) == fnv1a64(data)
    assert block_hash(0, [1, 2]) != block_hash(1, [1, 2]) != block_hash(0, [2, 1])


def test_pages_2407_token_prefix(Pool, golden_dir):
    g = read_json(os.path.join(golden_dir, "p1_prefix_match.json"))
    B, n = g["block_size"], g["prompt_tokens"]
    rng = np.random.default_rng(0)
    prompt = rng.integers(0, 150000, n).tolist()
    pool = Pool(4096, B)
    found = []
    for r in range(g["requests"]):
        cached, slots = pool.add_request(r, prompt + [10**6 + r])
        found.append(cached)
        assert len(slots) == n + 1
    assert found[0] == 0
    assert found[1:] == [g["tokens_found"]] * (g["requests"] - 1)
    assert g["tokens_found"] == g["full_blocks_found"] * B
    # what each later request computes: its prompt's tail (the page's seven
    # tokens) plus the one token that differs in this test
    assert n - g["tokens_found"] == g["tokens_computed"]
    # nothing is copied on a hit: the 150 blocks are the first request's
    t0 = pool.table(0)[:150]
    for r in range(1, g["requests"]):
        assert pool.table(r)[:150] == t0
    assert all(pool.refcount(b) == g["requests"] for b in t0)


def test_match_ends_on_block_boundary_and_last_token_is_computed(Pool):
    pool = Pool(64, 16)
    p = list(range(100, 148))  # 48 tokens, three full blocks
    pool.add_request(0, p)
    assert pool.add_request(1, p)[0] == 32       # (48 - 1) // 16 = 2 blocks
    assert pool.add_request(2, p + [5])[0] == 48  # one more token: all three
    assert pool.add_request(3, p[:40])[0] == 32   # shorter prompt: two blocks


def test_free_order_hashed_to_tail_reverse_order(Pool):
    """[P4] 9.3: free walks the request's blocks tail first; blocks without a
    hash go to the head of the free queue, hashed ones to the tail."""
    pool = Pool(8, 4)
    cached, slots = pool.add_request(10, list(range(1, 11)))  # 10 tokens: blocks 0, 1 full
    assert cached == 0 and pool.table(10) == [0, 1, 2]
    assert slots == [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]
    assert pool.block_hash(0) is not None and pool.block_hash(1) is not None
    assert pool.block_hash(2) is None
    assert pool.free_list() == [3, 4, 5, 6, 7]
    pool.release(10)
    assert pool.free_list() == [2, 3, 4, 5, 6, 7, 1, 0]
    # freeing does not clear: the same prompt finds blocks 0 and 1, touch
    # takes them out of the middle / tail of the queue
    cached, _ = pool.add_request(11, list(range(1, 11)))
    assert cached == 8 and pool.table(11) == [0, 1, 2]
    assert pool.free_list() == [3, 4, 5, 6, 7]
    assert [pool.refcount(b) for b in (0, 1, 2)] == [1, 1, 1]


def test_cached_blocks_leave_oldest_first(Pool):
    pool = Pool(6, 2)
    pool.add_request(10, [1, 2, 3])   # blocks 0 (hashed), 1
    pool.add_request(11, [7, 8, 9])   # blocks 2 (hashed), 3
    pool.release(10)                  # free: 1 4 5 0
    pool.release(11)                  # free: 3 1 4 5 0 2
    assert pool.free_list() == [3, 1, 4, 5, 0, 2]
    # four fresh blocks take the unhashed ones first, then the oldest cached
    pool.add_request(12, list(range(20, 28)))
    assert pool.table(12) == [3, 1, 4, 5]
    assert pool.lookup([1, 2, 3]) == 1 and pool.lookup([7, 8, 9]) == 1
    pool.add_request(13, [30, 31])    # needs one block: block 0, A's cache, goes
    assert pool.table(13) == [0]
    assert pool.lookup([1, 2, 3]) == 0 and pool.lookup([7, 8, 9]) == 1
    # block 0 now caches D's own full block instead
    assert pool.block_hash(0) == block_hash(0, [30, 31]) and pool.block_hash(2) is not None


def test_hash_chain_identity_and_salt(Pool):
    pool = Pool(32, 4)
    a = [1, 2, 3, 4, 5, 6, 7, 8, 9]
    pool.add_request(0, a)
    # the same second block after a different first block is not a hit
    b = [9, 9, 9, 9, 5, 6, 7, 8, 9]
    assert pool.lookup(b) == 0
    assert pool.lookup(a) == 2
    # a salt is mixed into the first block: different salts never match
    assert pool.lookup(a, salt=3) == 0
    pool.add_request(1, a, salt=3)
    assert pool.lookup(a, salt=3) == 2 and pool.lookup(a, salt=4) == 0
    assert pool.table(1)[:2] != pool.table(0)[:2]


def test_out_of_blocks_changes_nothing(Pool):
    pool = Pool(5, 2)
    pool.add_request(0, [1, 2, 3, 4, 5])  # 3 blocks, two hashed
    pool.release(0)
    pool.add_request(1, [1, 2, 3, 4, 5, 6, 7])  # hits 2 (touch), needs 2 more
    before = (pool.free_list(), [pool.refcount(b) for b in range(5)], pool.table(1))
    with pytest.raises(out_of_blocks()):
        pool.add_request(2, list(range(40, 47)))  # needs 4, 1 free
    with pytest.raises(out_of_blocks()):
        for t in range(10):
            pool.append(1, 100 + t)
    assert pool.refcount(0) == 1
    pool2 = Pool(5, 2)
    pool2.add_request(0, [1, 2, 3, 4, 5])
    pool2.release(0)
    pool2.add_request(1, [1, 2, 3, 4, 5, 6, 7])
    assert before == (pool2.free_list(), [pool2.refcount(b) for b in range(5)], pool2.table(1))


def test_append_fills_and_registers(Pool):
    pool = Pool(8, 4)
    pool.add_request(0, [1, 2, 3])
    assert pool.block_hash(0) is None
    slot = pool.append(0, 4)
    assert slot == 3 and pool.block_hash(0) == block_hash(0, [1, 2, 3, 4])
    assert pool.append(0, 5) == 4  # block 1
    # generated tokens are cached too: a request whose prompt is the first
    # request's text so far finds them
    assert pool.add_request(1, [1, 2, 3, 4, 5])[0] == 4


def test_duplicate_content_is_not_registered_twice(Pool):
    pool = Pool(8, 2)
    pool.add_request(0, [1, 2, 3, 4])     # blocks 0, 1 hashed
    cached, _ = pool.add_request(1, [1, 2, 3, 4])  # (4 - 1) // 2 = 1 hit; block 1 recomputed
    assert cached == 2 and pool.table(1)[0] == 0
    dup = pool.table(1)[1]
    assert pool.block_hash(dup) is None   # same content as block 1: not cached again
    pool.release(1)
    assert pool.free_list()[0] == dup     # unhashed: back to the head


def test_random_invariants():
    rng = np.random.default_rng(5)
    pool = PrefixCachePoolModel(40, 4, free_order=rng.permutation(40))
    prompts = [rng.integers(0, 6, int(rng.integers(1, 20))).tolist() for _ in range(6)]
    live, nxt = set(), 0
    for _ in range(500):
        op = rng.choice(["add", "append", "free"], p=[0.35, 0.4, 0.25])
        if op == "add":
            base = prompts[int(rng.integers(len(prompts)))]
            extra = rng.integers(0, 6, int(rng.integers(0, 6))).tolist()
            try:
                pool.add_request(nxt, base + extra, salt=int(rng.integers(0, 2)))
                live.add(nxt)
            except ModelOutOfBlocks:
                pass
            nxt += 1
        elif op == "append" and live:
            s = sorted(live)[int(rng.integers(len(live)))]
            try:
                pool.append(s, int(rng.integers(0, 6)))
            except ModelOutOfBlocks:
                pass
        elif op == "free" and live:
            s = sorted(live)[int(rng.integers(len(live)))]
            pool.release(s)
            live.discard(s)
        # every block is in use or free, never both; counts match the tables
        refs = [0] * 40
        for s in live:
            for b in pool.table(s):
                refs[b] += 1
            assert len(pool.table(s)) == -(-pool.length(s) // 4)
        assert refs == [pool.refcount(b) for b in range(40)]
        free = pool.free_list()
        assert len(set(free)) == len(free)
        assert sorted(free + [b for b in range(40) if refs[b] > 0]) == list(range(40))
        # every cached hash points at a block that holds it
        for h, b in pool.cached.items():
            assert pool.block_hash(b) == h


def test_native_hash_matches_model():
    from paged_kv_cache_64_gb300 import api, build
    build.build()
    pool = api.PrefixCachePool(4, 4)
    rng = np.random.default_rng(11)
    for _ in range(200):
        prev = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        toks = rng.integers(-2**31, 2**31, int(rng.integers(0, 40))).tolist()
        assert pool.hash_block(prev, toks) == block_hash(prev, toks)


@pytest.mark.parametrize("seed", range(4))
def test_native_matches_model_random(seed):
    """500 mixed operations on both pools: identical cached counts, slots,
    tables, free queues, refcounts and block hashes after every operation."""
    from paged_kv_cache_64_gb300 import _lib, api, build
    build.build()
    rng = np.random.default_rng(200 + seed)
    nb, B = 48, 4
    order = rng.permutation(nb)
    native = api.PrefixCachePool(nb, B, free_order=order)
    model = PrefixCachePoolModel(nb, B, free_order=order)
    prompts = [rng.integers(0, 5, int(rng.integers(1, 22))).tolist() for _ in range(5)]
    live, nxt = [], 0
    for _ in range(500):
        op = rng.choice(["add", "append", "free"], p=[0.3, 0.45, 0.25])
        if op == "add" or not live:
            toks = prompts[int(rng.integers(len(prompts)))] + \
                rng.integers(0, 5, int(rng.integers(0, 7))).tolist()
            salt = int(rng.integers(0, 2))
            assert native.lookup(toks, salt) == model.lookup(toks, salt)
            try:
                want = model.add_request(nxt, toks, salt)
            except ModelOutOfBlocks:
                with pytest.raises(_lib.OutOfBlocks):
                    native.add_request(nxt, toks, salt)
                nxt += 1
                continue
            assert native.add_request(nxt, toks, salt) == want
            live.append(nxt)
            nxt += 1
        elif op == "append":
            s = live[int(rng.integers(len(live)))]
            tok = int(rng.integers(0, 5))
            try:
                want = model.append(s, tok)
            except ModelOutOfBlocks:
                with pytest.raises(_lib.OutOfBlocks):
                    native.append(s, tok)
                continue
            assert native.append(s, tok) == want
        else:
            s = live.pop(int(rng.integers(len(live))))
            native.release(s)
            model.release(s)
        assert native.free_list() == model.free_list()
        assert [native.refcount(b) for b in range(nb)] == [model.refcount(b) for b in range(nb)]
        assert [native.block_hash(b) for b in range(nb)] == [model.block_hash(b) for b in range(nb)]
        for s in live:
            assert native.table(s) == model.table(s)
            assert native.length(s) == model.length(s)
