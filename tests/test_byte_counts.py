"""Host checks of the byte counts the benchmark's roofline divides by.

The closed forms in `workloads` (algorithmic_bytes, cascade_bytes,
cache_write_bytes) are checked against counts made another way: walking a
real layout (the allocator model's tables after the step) position by
position, the way a decode reads it, and counting what is read and written.
The cascade's count reads each shared prefix slot once by its physical
address, so it also checks that the layout really shares the prefix.
"""
import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_64_gb300 import workloads


def _layout(name, **kw):
    plan = workloads.make_plan(name, **kw)
    return plan.spec, workloads.layout(plan, BlockAllocatorModel)


def _elem(spec):
    return workloads.DTYPE_BYTES[spec.dtype]


def walk_plain(spec, lay, kvb=None):
    """Every sequence reads its own positions [0, L) (K and V of each KV
    head), one table entry per block it touches, q in and out, its length."""
    B = spec.block_size
    kvb = kvb or _elem(spec)
    positions, entries = 0, set()
    for s, L in enumerate(lay.seq_lens):
        for pos in range(int(L)):
            positions += 1
            entries.add((s, pos // B))
    per_pos = 2 * spec.num_kv_heads * spec.head_dim * kvb
    qo = 2 * len(lay.seq_lens) * spec.num_q_heads * spec.head_dim * _elem(spec)
    return positions * per_pos + 4 * len(entries) + qo + 4 * len(lay.seq_lens)


def walk_cascade(spec, lay, prefix_len):
    """Positions below prefix_len are read once, by physical slot, through
    sequence 0's table; each tail through its own table."""
    B = spec.block_size
    slots, tail_positions, entries = set(), 0, set()
    for s, L in enumerate(lay.seq_lens):
        for pos in range(int(L)):
            blk = int(lay.block_tables[s, pos // B])
            if pos < prefix_len:
                slots.add(blk * B + pos % B)
                entries.add((0, pos // B))
            else:
                tail_positions += 1
                entries.add((s, pos // B))
    per_pos = 2 * spec.num_kv_heads * spec.head_dim * _elem(spec)
    qo = 2 * len(lay.seq_lens) * spec.num_q_heads * spec.head_dim * _elem(spec)
    return ((len(slots) + tail_positions) * per_pos + 4 * len(entries) + qo +
            4 * len(lay.seq_lens))


def shared_whole_blocks(lay, B):
    """Positions of the leading whole blocks every sequence reaches through
    the same table entry (and fully covers)."""
    n = 0
    min_blocks = int(lay.seq_lens.min()) // B
    while n < min_blocks and np.all(lay.block_tables[:, n] == lay.block_tables[0, n]):
        n += 1
    return n * B


CASES = [("tiny", {}), ("qwen", {"num_seqs": 16}), ("llama", {"num_seqs": 8}),
         ("long", {"num_seqs": 2}), ("prefix", {"num_seqs": 12}),
         ("prefix", {"num_seqs": 12, "cow": True})]


@pytest.mark.parametrize("name,kw", CASES)
def test_algorithmic_bytes_match_a_walk_of_the_layout(name, kw):
    spec, lay = _layout(name, **kw)
    assert workloads.algorithmic_bytes(spec, lay.seq_lens) == walk_plain(spec, lay)
    # E4M3 pools: one byte per K/V element, q and out still 16-bit
    assert workloads.algorithmic_bytes(spec, lay.seq_lens, 1) == walk_plain(spec, lay, 1)


@pytest.mark.parametrize("cow", [False, True])
def test_cascade_bytes_read_the_shared_prefix_once(cow):
    spec, lay = _layout("prefix", num_seqs=12, cow=cow)
    B = spec.block_size
    P = shared_whole_blocks(lay, B)
    # 4,096 positions shared; with the 4,112-token prompt the half-full
    # 129th block was copied on write by all but one fork, so it is not shared
    assert P == 4096
    assert workloads.cascade_bytes(spec, lay.seq_lens, P) == walk_cascade(spec, lay, P)
    plain = workloads.algorithmic_bytes(spec, lay.seq_lens)
    per_pos = 2 * spec.num_kv_heads * spec.head_dim * _elem(spec)
    saved = (len(lay.seq_lens) - 1) * (P * per_pos + 4 * (P // B))
    assert plain - workloads.cascade_bytes(spec, lay.seq_lens, P) == saved


@pytest.mark.parametrize("name,kw", CASES)
def test_cascade_bytes_without_a_prefix_are_the_plain_bytes(name, kw):
    spec, lay = _layout(name, **kw)
    assert (workloads.cascade_bytes(spec, lay.seq_lens, 0) ==
            workloads.algorithmic_bytes(spec, lay.seq_lens))


@pytest.mark.parametrize("name,kw", CASES)
@pytest.mark.parametrize("kvb", [None, 1])
def test_cache_write_bytes_match_the_step_slots(name, kw, kvb):
    """Each new token: K and V of every KV head read from the 16-bit inputs
    and written to its own slot of the pools, plus its 8-byte slot index."""
    spec, lay = _layout(name, **kw)
    slots = [int(x) for x in lay.slot_mapping]
    assert len(set(slots)) == len(slots) == spec.num_seqs
    per_slot = 2 * spec.num_kv_heads * spec.head_dim * (_elem(spec) + (kvb or _elem(spec)))
    assert (workloads.cache_write_bytes(spec, spec.num_seqs, kvb) ==
            len(set(slots)) * (per_slot + 8))


def test_unit_bytes_are_the_per_token_kv_bytes():
    """One cached token of one KV head is 2 d b bytes (K and V): 512 B at
    d = 128 in bf16, 256 B at d = 64 in fp16, half of each over E4M3 pools.
    A one-sequence, one-KV-head batch grows by exactly that per token."""
    for name, unit in (("llama", 512), ("qwen", 256)):
        base = workloads.SPECS[name]
        spec = workloads.Spec(base.name, 1, base.num_q_heads // base.num_kv_heads, 1,
                              base.head_dim, base.block_size, base.dtype, 1, 0, 0, "")
        B = spec.block_size
        for L in (1, B - 1, B, 5 * B + 3):
            # same block count for L and L + 1 inside a block, one more entry across
            grow = (workloads.algorithmic_bytes(spec, [L + 1]) -
                    workloads.algorithmic_bytes(spec, [L]))
            assert grow == unit + (4 if L % B == 0 else 0)
            grow8 = (workloads.algorithmic_bytes(spec, [L + 1], 1) -
                     workloads.algorithmic_bytes(spec, [L], 1))
            assert grow8 == unit // 2 + (4 if L % B == 0 else 0)
