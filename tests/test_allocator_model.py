"""Pins of the allocator model (oracle/allocator.py) against the tables the
pages print and against invariants that must hold after every operation."""
import json
import os

import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, OutOfBlocks
from conftest import read_json


def replay_hand_table(model, steps):
    for st in steps:
        ev = st["event"]
        if ev[0] == "add":
            model.add(ev[1])
            model.append(ev[1], ev[2])
        elif ev[0] == "append":
            model.append(ev[1], ev[2])
        elif ev[0] == "free":
            model.release(ev[1])
        yield st


def test_hand_worked_table(golden_dir):
    g = read_json(os.path.join(golden_dir, "p2_hand_worked_table.json"))
    model = BlockAllocatorModel(g["num_blocks"], g["block_size"])
    for st in replay_hand_table(model, g["steps"]):
        assert {s: model.table(s) for s in model.tables} == st["tables"], st
        assert model.free_list() == st["free"], st
        assert {s: model.length(s) for s in model.lengths} == st["tokens"], st
        assert model.wasted_slots() == st["wasted"], st


def test_quiz4_new_request(golden_dir):
    g = read_json(os.path.join(golden_dir, "p2_hand_worked_table.json"))
    q = read_json(os.path.join(golden_dir, "p2_quiz4.json"))
    model = BlockAllocatorModel(g["num_blocks"], g["block_size"])
    for _ in replay_hand_table(model, g["steps"]):
        pass
    model.add(q["new_request"])
    slots, copies = model.append(q["new_request"], q["prompt_tokens"])
    table = model.table(q["new_request"])
    assert table == q["expected_table"] and model.free_list() == q["expected_free"]
    assert len(table) * q["block_size"] - q["prompt_tokens"] == q["expected_empty_slots"]
    p = q["position"]
    assert p // q["block_size"] == q["expected_logical_block"]
    assert p % q["block_size"] == q["expected_offset"]
    assert table[p // q["block_size"]] == q["expected_physical_block"]
    assert slots[p] == q["expected_physical_block"] * q["block_size"] + q["expected_offset"]
    assert copies == []


def test_prefix_sharing_copy_on_write(golden_dir):
    g = read_json(os.path.join(golden_dir, "p2_prefix_sharing.json"))
    model = BlockAllocatorModel(g["num_blocks"], g["block_size"])
    for st in g["steps"]:
        ev = st["event"]
        copies = []
        if ev[0] == "prompt":
            model.add(ev[1])
            _, copies = model.append(ev[1], g["prompt_tokens"])
        elif ev[0] == "fork":
            model.fork(ev[1], ev[2])
        elif ev[0] == "append":
            _, copies = model.append(ev[1], ev[2])
        assert {s: model.table(s) for s in model.tables} == st["tables"], st
        assert [model.refcount(b) for b in (0, 1, 2)] == st["refs_0_1_2"], st
        assert model.free_list() == st["free"], st
        assert [list(c) for c in copies] == st["copies"], st


def test_out_of_blocks_changes_nothing():
    """A copy-on-write append with no free block raises and leaves every
    table, count, refcount and the free list as they were."""
    model = BlockAllocatorModel(3, 4)
    model.add("a")
    model.append("a", 6)      # blocks 0, 1
    model.fork("a", "b")      # block 1 shared, half full
    model.add("c")
    model.append("c", 3)      # block 2: pool now empty
    state = (dict(model.tables), dict(model.lengths), list(model.refs), model.free_list())
    with pytest.raises(OutOfBlocks):
        model.append("b", 1)
    with pytest.raises(OutOfBlocks):
        model.append("c", 2)  # needs a new block for position 4
    assert state == (dict(model.tables), dict(model.lengths), list(model.refs), model.free_list())
    model.append("c", 1)      # fits in block 2: fine
    # all-or-nothing: 1 token fits, 5 would not
    with pytest.raises(OutOfBlocks):
        model.append("a", 3)


def test_seeded_free_order():
    model = BlockAllocatorModel(5, 2, free_order=[3, 0, 4, 1, 2])
    model.add(0)
    slots, _ = model.append(0, 3)
    assert model.table(0) == [3, 0] and slots == [6, 7, 0]
    with pytest.raises(ValueError):
        BlockAllocatorModel(3, 2, free_order=[0, 0, 1])


@pytest.mark.parametrize("seed", range(5))
def test_random_operations_invariants(seed):
    """400 mixed operations (add / append / fork / free).  After each one: no
    block is lost, double-booked or listed twice; refcounts equal the number
    of table entries naming the block; every sequence reads back, through its
    table, exactly what was written for it."""
    rng = np.random.default_rng(seed)
    nb, B = 24, 4
    model = BlockAllocatorModel(nb, B)
    pool = np.full(nb * B, -1, dtype=np.int64)   # one "value" per slot
    logical = {}                                 # seq -> values in order
    next_id, next_val = 0, 0
    for _ in range(400):
        op = rng.choice(["add", "append", "fork", "free"], p=[0.2, 0.5, 0.15, 0.15])
        live = sorted(model.tables)
        if op == "add" or not live:
            model.add(next_id)
            logical[next_id] = []
            next_id += 1
        elif op == "append":
            s = live[rng.integers(len(live))]
            n = int(rng.integers(1, 7))
            try:
                slots, copies = model.append(s, n)
            except OutOfBlocks:
                continue
            for src, dst in copies:
                pool[dst * B:(dst + 1) * B] = pool[src * B:(src + 1) * B]
            for slot in slots:
                pool[slot] = next_val
                logical[s].append(next_val)
                next_val += 1
        elif op == "fork":
            s = live[rng.integers(len(live))]
            model.fork(s, next_id)
            logical[next_id] = list(logical[s])
            next_id += 1
        else:
            s = live[rng.integers(len(live))]
            model.release(s)
            del logical[s]
        # invariants
        free = model.free_list()
        assert len(free) == len(set(free))
        counts = np.zeros(nb, dtype=np.int64)
        for t in model.tables.values():
            for b in t:
                counts[b] += 1
        assert counts.tolist() == model.refs
        held = {b for b in range(nb) if counts[b] > 0}
        assert held.isdisjoint(free) and held | set(free) == set(range(nb))
        for s, vals in logical.items():
            t = model.table(s)
            assert model.length(s) == len(vals)
            assert len(t) == -(-len(vals) // B)
            got = [int(pool[t[p // B] * B + p % B]) for p in range(len(vals))]
            assert got == vals
