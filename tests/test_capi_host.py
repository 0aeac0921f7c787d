"""Host-side tests of the C ABI (no GPU needed): the library loads and exports
every symbol include/pa.h declares; the native allocator matches the
allocator model operation for operation; argument validation rejects bad
shapes before any launch."""
import ctypes
import json
import os
import re

import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, OutOfBlocks as ModelOutOfBlocks
from paged_kv_cache_64_gb300 import _lib, api, workloads
from conftest import read_json

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_64_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "pa.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, n
    assert set(_lib.SIGNATURES) == set(names)


def test_version_and_status_strings(lib):
    assert lib.pa_version() >= 100
    for code in range(8):
        assert lib.pa_status_string(code)


def test_validation_before_launch(lib):
    vp = ctypes.c_void_p
    # G not an integer -> invalid; head_dim 96 -> unsupported; no device call needed
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 6, 4, 128,
                       16, 1.0, -1, None, 0, 1, None)
    assert rc == 1
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 8, 4, 96,
                       16, 1.0, -1, None, 0, 1, None)
    assert rc == 3
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 8, 4, 128,
                       24, 1.0, -1, None, 0, 1, None)
    assert rc == 3  # block size 24
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 8, 4, 128,
                       16, 1.0, 40, None, 0, 1, None)
    assert rc == 1  # partition not a multiple of 16
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 32, 2, 128,
                       16, 1.0, -1, None, 0, 1, None)
    assert rc == 3  # G = 16 not compiled
    rc = lib.pa_decode(vp(16), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 8, 4, 128,
                       16, float("nan"), -1, None, 0, 1, None)
    assert rc == 1  # non-finite scale
    rc = lib.pa_decode(vp(17), vp(16), vp(16), vp(16), 10, vp(16), 4, vp(16), 64, 2, 8, 4, 128,
                       16, 1.0, -1, None, 0, 1, None)
    assert rc == 1  # misaligned out
    assert lib.pa_cache_write(vp(16), vp(16), vp(16), 3, vp(16), vp(16), 8, 2, 80, 16, 0,
                              None) == 3
    assert lib.pa_cache_write(vp(16), vp(16), vp(16), -1, vp(16), vp(16), 8, 2, 64, 16, 0,
                              None) == 1
    assert lib.pa_cache_write(None, None, None, 0, None, None, 8, 2, 64, 16, 0, None) == 0
    arr = (ctypes.c_void_p * 1)(16)
    assert lib.pa_copy_blocks(arr, arr, 1, None, 0, 8, 4096, None) == 0
    assert lib.pa_copy_blocks(arr, arr, 1, vp(16), 2, 8, 4095, None) == 1
    assert lib.pa_copy_blocks(arr, arr, 0, vp(16), 2, 8, 4096, None) == 1


def test_cascade_validation_before_launch(lib):
    vp = ctypes.c_void_p
    args = lambda P, maxlen=64: (vp(16), vp(16), None, None, None, vp(16), vp(16), 10, vp(16), 4,
                                 vp(16), maxlen, 2, 8, 4, 128, 16, 1.0, P, vp(256), 1 << 20, 1,
                                 None)
    assert lib.pa_decode_cascade(*args(24)) == 1       # not a whole number of blocks
    assert lib.pa_decode_cascade(*args(80)) == 1       # longer than max_seq_len
    assert lib.pa_decode_cascade(*args(-16)) == 1
    assert lib.pa_decode_cascade_workspace_size(2, 8, 4, 128, 16, 64, 24, 1) == 0
    assert lib.pa_decode_cascade_workspace_size(2, 8, 4, 128, 16, 64, 80, 1) == 0


def test_workspace_size_layout(lib):
    # explicit partition: m, l (256-aligned) then O (64 positions: never
    # several partitions a CTA, so one partial per partition)
    S, hq, hkv, d, maxlen, P = 3, 8, 2, 128, 1000, 64
    NP = 16
    rows = S * hq * NP
    a = lambda x: (x + 255) // 256 * 256
    # + the fused combine: a 64-bit counter per (seq, kv head), a 32-bit flag per partition
    want = a(rows * 4) * 2 + a(rows * d * 4) + a(S * hkv * 8) + a(S * hkv * NP * 4)
    assert lib.pa_decode_workspace_size(S, hq, hkv, d, 16, maxlen, P, 1) == want
    assert lib.pa_decode_workspace_size(S, hq, 2, d, 16, maxlen, -1, 1) == 0


# ------------------------------------------------------------- allocator
def replay(alloc, steps):
    for st in steps:
        ev = st["event"]
        if ev[0] == "add":
            alloc.add(ev[1])
            alloc.append(ev[1], ev[2])
        elif ev[0] == "append":
            alloc.append(ev[1], ev[2])
        elif ev[0] == "free":
            alloc.release(ev[1])
        yield st


def test_native_allocator_hand_worked_table(lib, golden_dir):
    g = read_json(os.path.join(golden_dir, "p2_hand_worked_table.json"))
    ids = {"A": 1, "B": 2, "C": 3}
    alloc = api.BlockAllocator(g["num_blocks"], g["block_size"])
    for st in g["steps"]:
        ev = list(st["event"])
        if len(ev) > 1:
            ev[1] = ids[ev[1]]
        for _ in replay(alloc, [{"event": ev}]):
            pass
        for name, table in st["tables"].items():
            assert alloc.table(ids[name]) == table, st
            assert alloc.length(ids[name]) == st["tokens"][name]
        assert alloc.free_list() == st["free"], st


def test_native_allocator_prefix_sharing(lib, golden_dir):
    g = read_json(os.path.join(golden_dir, "p2_prefix_sharing.json"))
    ids = {"S1": 1, "S2": 2}
    alloc = api.BlockAllocator(g["num_blocks"], g["block_size"])
    for st in g["steps"]:
        ev = st["event"]
        copies = []
        if ev[0] == "prompt":
            alloc.add(ids[ev[1]])
            _, copies = alloc.append(ids[ev[1]], g["prompt_tokens"])
        elif ev[0] == "fork":
            alloc.fork(ids[ev[1]], ids[ev[2]])
        else:
            _, copies = alloc.append(ids[ev[1]], ev[2])
        for name, t in st["tables"].items():
            assert alloc.table(ids[name]) == t
        assert [alloc.refcount(b) for b in (0, 1, 2)] == st["refs_0_1_2"]
        assert alloc.free_list() == st["free"]
        assert [list(c) for c in copies] == st["copies"]


def test_native_allocator_errors_leave_state(lib):
    alloc = api.BlockAllocator(3, 4)
    alloc.add(1)
    alloc.append(1, 6)
    alloc.fork(1, 2)
    alloc.add(3)
    alloc.append(3, 3)
    before = (alloc.table(1), alloc.table(2), alloc.table(3), alloc.free_list(),
              [alloc.refcount(b) for b in range(3)])
    with pytest.raises(_lib.OutOfBlocks):
        alloc.append(2, 1)
    with pytest.raises(_lib.OutOfBlocks):
        alloc.append(3, 2)
    with pytest.raises(_lib.PagedAttentionError):
        alloc.add(1)            # duplicate id
    with pytest.raises(_lib.PagedAttentionError):
        alloc.fork(9, 10)       # unknown parent
    with pytest.raises(_lib.PagedAttentionError):
        alloc.release(42)
    assert before == (alloc.table(1), alloc.table(2), alloc.table(3), alloc.free_list(),
                      [alloc.refcount(b) for b in range(3)])
    assert alloc.refcount(-1) == -1 and alloc.refcount(3) == -1
    with pytest.raises(_lib.PagedAttentionError):
        api.BlockAllocator(4, 2, free_order=[0, 1, 1, 2])


@pytest.mark.parametrize("seed", range(5))
def test_native_allocator_matches_model_random(lib, seed):
    """400 mixed operations on both allocators: identical slots, copies,
    tables, free lists and refcounts after every operation."""
    rng = np.random.default_rng(100 + seed)
    nb, B = 24, 4
    order = rng.permutation(nb)
    native = api.BlockAllocator(nb, B, free_order=order)
    model = BlockAllocatorModel(nb, B, free_order=order)
    next_id = 0
    for _ in range(400):
        op = rng.choice(["add", "append", "fork", "free"], p=[0.2, 0.5, 0.15, 0.15])
        live = sorted(model.tables)
        if op == "add" or not live:
            native.add(next_id)
            model.add(next_id)
            next_id += 1
        elif op == "append":
            s = live[rng.integers(len(live))]
            n = int(rng.integers(0, 7))
            try:
                want = model.append(s, n)
            except ModelOutOfBlocks:
                with pytest.raises(_lib.OutOfBlocks):
                    native.append(s, n)
                continue
            assert native.append(s, n) == want
        elif op == "fork":
            s = live[rng.integers(len(live))]
            native.fork(s, next_id)
            model.fork(s, next_id)
            next_id += 1
        else:
            s = live[rng.integers(len(live))]
            native.release(s)
            model.release(s)
        assert native.free_list() == model.free_list()
        assert [native.refcount(b) for b in range(nb)] == model.refs
        for s in model.tables:
            assert native.table(s) == model.table(s)
            assert native.length(s) == model.length(s)


@pytest.mark.parametrize("name,cow", [("tiny", False), ("qwen", False), ("prefix", False),
                                      ("prefix", True), ("long", False), ("llama", False)])
def test_workload_layouts_agree(lib, name, cow):
    """The native allocator and the model lay every workload out identically
    (tables, lengths, new-token slots, copy-on-write pairs)."""
    kw = {"num_seqs": 32} if name == "llama" else {}
    plan = workloads.make_plan(name, cow=cow, **kw)
    a = workloads.layout(plan, api.BlockAllocator)
    b = workloads.layout(plan, BlockAllocatorModel)
    for f in ("block_tables", "seq_lens", "slot_mapping", "pre_copies", "pre_slots",
              "step_copies"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    if name == "prefix" and cow:
        assert len(a.pre_copies) == 63  # the 64th writer owns the shared block alone
    if name == "prefix" and not cow:
        assert len(a.pre_copies) == 0   # full shared blocks are never written


@pytest.mark.parametrize("shape", [(7, 28, 4, 128, 16, "f16", (0, 1500)),
                                   (7, 6, 2, 64, 32, "f16", (0, 1500)),
                                   (3000, 4, 1, 64, 16, "f16", (0, 24))])
def test_shape_plan_layouts_agree(lib, shape):
    """Shape-sweep batches: native allocator and model agree, every table
    entry a sequence uses is a distinct block of the pool, and each new
    token's slot is the one its table gives for position L - 1."""
    plan = workloads.make_shape_plan(*shape, seed=5)
    a = workloads.layout(plan, api.BlockAllocator)
    b = workloads.layout(plan, BlockAllocatorModel)
    for f in ("block_tables", "seq_lens", "slot_mapping", "pre_copies", "step_copies"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    B = plan.spec.block_size
    assert np.array_equal(a.seq_lens, plan.cached_lens + 1)
    used = [a.block_tables[s, :-(-int(L) // B)] for s, L in enumerate(a.seq_lens)]
    flat = np.concatenate(used)
    assert len(np.unique(flat)) == len(flat) and flat.min() >= 0 and flat.max() < plan.num_blocks
    last = a.seq_lens.astype(np.int64) - 1
    want = a.block_tables[np.arange(len(last)), last // B].astype(np.int64) * B + last % B
    assert np.array_equal(a.slot_mapping, want)


def test_shared_prefix_len():
    """Whole blocks that every sequence reaches through the same entries,
    capped by the shortest sequence."""
    t = np.array([[4, 7, 9, 1], [4, 7, 9, 2], [4, 7, 3, 5]], dtype=np.int32)
    assert api.shared_prefix_len(t, [64, 64, 64], 16) == 32
    assert api.shared_prefix_len(t[:2], [64, 64], 16) == 48
    assert api.shared_prefix_len(t[:2], [64, 40], 16) == 32      # shortest: 2 whole blocks
    assert api.shared_prefix_len(t[:1], [50], 16) == 48          # one sequence: its whole blocks
    assert api.shared_prefix_len(t[[0, 2]][:, ::-1], [64, 64], 16) == 0
    assert api.shared_prefix_len(np.zeros((0, 4), np.int32), [], 16) == 0
    for cow in (False, True):
        plan = workloads.make_plan("prefix", cow=cow)
        lay = workloads.layout(plan, BlockAllocatorModel)
        assert api.shared_prefix_len(lay.block_tables, lay.seq_lens, 32) == 4096


def test_shared_prefix_len_brute_force_and_errors():
    """pa_shared_prefix_len against a direct count on random tables; bad
    arguments are refused."""
    rng = np.random.default_rng(3)
    for _ in range(300):
        S, nb, B = int(rng.integers(1, 6)), int(rng.integers(0, 9)), int(rng.choice([1, 4, 16]))
        t = rng.integers(0, 4, (S, nb)).astype(np.int32)
        share = int(rng.integers(0, nb + 1))
        t[:, :share] = t[0, :share]
        lens = rng.integers(0, nb * B + 3, S)
        want = 0
        while (want < min(int(lens.min()) // B, nb)
               and all(t[i, want] == t[0, want] for i in range(S))):
            want += 1
        assert api.shared_prefix_len(t, lens, B) == want * B
    t = np.zeros((2, 3), np.int32)
    for lens, B in (([5, -1], 16), ([5, 5], 0)):
        with pytest.raises(_lib.PagedAttentionError) as e:
            api.shared_prefix_len(t, lens, B)
        assert e.value.code == 1


def test_prefix_caching_layout_agrees(lib):
    """The prefix workload as 64 separate requests laid out by the
    prefix-caching pool: native pool and model agree, and the prompt's 128
    blocks are shared by every request."""
    from oracle.prefix_cache import PrefixCachePoolModel
    plan = workloads.make_plan("prefix", apc=True)
    a = workloads.layout(plan, api.PrefixCachePool)
    b = workloads.layout(plan, PrefixCachePoolModel)
    for f in ("block_tables", "seq_lens", "slot_mapping", "pre_copies", "pre_slots",
              "step_copies"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    assert api.shared_prefix_len(a.block_tables, a.seq_lens, 32) == 4096
    assert len(a.pre_copies) == 0
    tails = plan.cached_lens - 4096
    # written before the step: the first prompt in full, then only each tail
    assert len(a.pre_slots) == 4096 + int(tails.sum())
