"""Seeded synthetic workloads for the paged decode step.

This module holds none of the method's arithmetic.  It draws sequence lengths,
the initial free-list order of the pool (a seeded permutation, so physical
blocks are scattered) and random K/V/q values, and it lists the allocator
operations that lay the cache out.  The allocator passed to `layout` (the
library's BlockAllocator, or the oracle's model in tests) decides every block,
slot and copy-on-write pair.

Workloads (sizes from the pages' own examples):
  tiny    4 sequences, 5/17/33/64 cached tokens, 4 q / 2 KV heads, d 64, fp16,
          B 16, 32-block pool.
  qwen    Qwen2.5-0.5B shape: 14 q / 2 KV heads, d 64, fp16, B 16, 128
          sequences with lognormal lengths (median 200, sigma 0.858, clipped
          to 1..2048), 65,536-block pool, 24 layers run back to back.
  llama   Llama-3-8B shape: 32 q / 8 KV heads, d 128, bf16, B 16, 256
          sequences, lengths uniform in 512..8192, pool 1.2x the blocks used.
  prefix  64 sequences forked from one 4,096-token prompt (or 4,112 for the
          copy-on-write case) plus tails uniform in 1..256 tokens, 32 q / 8 KV
          heads, d 128, bf16, B 32, pool 1.2x the distinct blocks.
  long    16 sequences, lengths uniform in 16,384..32,768, 64 q / 8 KV heads,
          d 128, bf16, B 16, split-KV partitions of 512 positions.
Every workload then runs one decode step: each sequence appends one new token
(its K/V written by the cache write) and attends over all its tokens.
K, V, q and the new tokens are drawn N(0, 1).
"""
import math
from dataclasses import dataclass, field

import numpy as np

DTYPE_BYTES = {"f16": 2, "bf16": 2}


@dataclass(frozen=True)
class Spec:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str
    num_layers: int
    seed: int
    partition_tokens: int  # 0 = automatic
    describe: str


SPECS = {
    "tiny": Spec("tiny", 4, 4, 2, 64, 16, "f16", 1, 1, 0,
                 "4 seqs, cached lengths 5/17/33/64, 4q/2kv heads, d64, fp16, B16, 32-block pool"),
    "qwen": Spec("qwen", 128, 14, 2, 64, 16, "f16", 24, 2, 0,
                 "Qwen2.5-0.5B shape, 128 seqs, lognormal lengths (median 200), 24 layers"),
    "llama": Spec("llama", 256, 32, 8, 128, 16, "bf16", 1, 3, 0,
                  "Llama-3-8B shape, 256 seqs, lengths U[512, 8192], one layer"),
    "prefix": Spec("prefix", 64, 32, 8, 128, 32, "bf16", 1, 4, 0,
                   "64 seqs sharing a 4096(+16)-token prefix, tails U[1, 256], B32"),
    "long": Spec("long", 16, 64, 8, 128, 16, "bf16", 1, 5, 512,
                 "16 seqs, lengths U[16384, 32768], 64q/8kv heads, split-KV P=512"),
}

LOGNORMAL_SIGMA = math.sqrt(2.0 * math.log(260.0 / 180.0))  # ~0.858


@dataclass
class Plan:
    spec: Spec
    cached_lens: np.ndarray          # tokens already cached per sequence
    num_blocks: int
    free_order: np.ndarray           # int32 permutation of the pool's block ids
    ops: list                        # allocator operations before the step
    pre_write_seqs: list = field(default_factory=list)  # (seq, n) whose tokens get written
    cow_case: bool = False
    # automatic prefix caching: separate requests with their prompts' token
    # ids, laid out by a prefix-caching pool; step_tokens are the ids the
    # decode step appends
    apc: bool = False
    step_tokens: np.ndarray = None

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.spec.head_dim)


def _blocks(n, B):
    return -(-int(n) // B)


def make_plan(name, num_seqs=None, len_range=None, cow=False, seed=None, apc=False):
    """Draw the plan of a workload.  num_seqs / len_range shrink a workload for
    tests (same structure, fewer or shorter sequences)."""
    base = SPECS[name]
    S = int(num_seqs or base.num_seqs)
    spec = Spec(base.name, S, base.num_q_heads, base.num_kv_heads, base.head_dim,
                base.block_size, base.dtype, base.num_layers,
                base.seed if seed is None else seed, base.partition_tokens, base.describe)
    rng = np.random.default_rng(spec.seed)
    B = spec.block_size
    ops, pre = [], []
    if name == "tiny":
        lens = np.array([5, 17, 33, 64][:S], dtype=np.int64)
        nb = 32
    elif name == "qwen":
        lo, hi = len_range or (1, 2048)
        lens = np.clip(np.rint(rng.lognormal(math.log(200.0), LOGNORMAL_SIGMA, S)), lo, hi)
        lens = lens.astype(np.int64)
        nb = 65536
    elif name in ("llama", "long"):
        lo, hi = len_range or ((512, 8192) if name == "llama" else (16384, 32768))
        lens = rng.integers(lo, hi, S, endpoint=True).astype(np.int64)
        nb = int(math.ceil(1.2 * sum(_blocks(L + 1, B) for L in lens)))
    elif name == "prefix" and apc:
        # the same 4,096-token prompt in 64 separate requests, each with its
        # own tail: the pool's prefix cache, not a fork, shares the prompt
        lo, hi = len_range or (1, 256)
        prefix = 4096
        tails = rng.integers(lo, hi, S, endpoint=True).astype(np.int64)
        lens = prefix + tails
        prompt = rng.integers(0, 32000, prefix).astype(np.int32)
        uniq = _blocks(prefix, B) + sum(_blocks(prefix + t + 1, B) - prefix // B for t in tails)
        nb = int(math.ceil(1.2 * uniq))
        for s in range(S):
            tail = rng.integers(0, 32000, int(tails[s])).astype(np.int32)
            ops.append(("request", s, np.concatenate([prompt, tail])))
        step_tokens = rng.integers(0, 32000, S).astype(np.int32)
        free_order = rng.permutation(nb).astype(np.int32)
        return Plan(spec, lens, nb, free_order, ops, pre, False, True, step_tokens)
    elif name == "prefix":
        lo, hi = len_range or (1, 256)
        prefix = 4096 + (16 if cow else 0)
        tails = rng.integers(lo, hi, S, endpoint=True).astype(np.int64)
        lens = prefix + tails
        uniq = _blocks(prefix, B) + sum(_blocks(prefix + t + 1, B) - prefix // B for t in tails)
        nb = int(math.ceil(1.2 * uniq))
        ops.append(("add", 0))
        ops.append(("append", 0, prefix))
        for s in range(1, S):
            ops.append(("fork", 0, s))
        for s in range(S):
            # the tail tokens' K/V are written by the cache write before the step
            ops.append(("append", s, int(tails[s]), "write"))
            pre.append((s, int(tails[s])))
    else:
        raise KeyError(name)
    if name != "prefix":
        for s in range(S):
            ops.append(("add", s))
            ops.append(("append", s, int(lens[s])))
    free_order = rng.permutation(nb).astype(np.int32)
    return Plan(spec, lens, nb, free_order, ops, pre, cow)


def make_shape_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                    len_range, seed):
    """A plain decode batch of any supported head shape, for tests that sweep
    shapes: num_seqs sequences with cached lengths uniform in len_range (both
    ends included), each added and appended on its own, in a pool of 1.2x the
    blocks the step needs (at least 8), block ids handed out in a seeded
    permutation."""
    spec = Spec("shape", int(num_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim),
                int(block_size), dtype, 1, int(seed), 0,
                f"{num_seqs} seqs, {num_q_heads}q/{num_kv_heads}kv, d{head_dim}, {dtype}, "
                f"B{block_size}, lengths U[{len_range[0]}, {len_range[1]}]")
    rng = np.random.default_rng(spec.seed)
    lo, hi = len_range
    lens = rng.integers(lo, hi, spec.num_seqs, endpoint=True).astype(np.int64)
    nb = max(8, int(math.ceil(1.2 * sum(_blocks(L + 1, spec.block_size) for L in lens))))
    ops = []
    for s in range(spec.num_seqs):
        ops.append(("add", s))
        if lens[s]:
            ops.append(("append", s, int(lens[s])))
    free_order = rng.permutation(nb).astype(np.int32)
    return Plan(spec, lens, nb, free_order, ops)


@dataclass
class Layout:
    block_tables: np.ndarray   # int32 [S, max_blocks_per_seq] after the step
    seq_lens: np.ndarray       # int32 [S] after the step (cached + 1)
    slot_mapping: np.ndarray   # int64 [S]: slot of each sequence's new token
    pre_copies: np.ndarray     # int64 [n, 2] copy-on-write pairs before the step
    pre_slots: np.ndarray      # int64 [m]: slots of tokens written before the step
    step_copies: np.ndarray    # int64 [k, 2] copy-on-write pairs of the step itself
    max_seq_len: int


def layout(plan, allocator_factory):
    """Run the plan's operations and the decode step's appends on an allocator
    made by allocator_factory(num_blocks, block_size, free_order): a block
    allocator (add / append / fork), or for a plan with apc a prefix-caching
    pool (add_request / append)."""
    spec = plan.spec
    alloc = allocator_factory(plan.num_blocks, spec.block_size, plan.free_order)
    pre_copies, pre_slots = [], []
    for op in plan.ops:
        if op[0] == "add":
            alloc.add(op[1])
        elif op[0] == "fork":
            alloc.fork(op[1], op[2])
        elif op[0] == "append":
            slots, copies = alloc.append(op[1], op[2])
            pre_copies.extend(copies)
            if len(op) > 3 and op[3] == "write":
                pre_slots.extend(slots)
        elif op[0] == "request":
            # prompt positions the cache already holds are not written again
            cached, slots = alloc.add_request(op[1], op[2])
            pre_slots.extend(slots[cached:])
    step_slots, step_copies = [], []
    for s in range(spec.num_seqs):
        if plan.apc:
            step_slots.append(alloc.append(s, int(plan.step_tokens[s])))
            continue
        slots, copies = alloc.append(s, 1)
        step_slots.extend(slots)
        step_copies.extend(copies)
    seqs = list(range(spec.num_seqs))
    lens = [alloc.length(s) for s in seqs]
    maxb = max(1, max(_blocks(L, spec.block_size) for L in lens))
    tables = np.zeros((spec.num_seqs, maxb), dtype=np.int32)
    for s in seqs:
        t = alloc.table(s)
        tables[s, :len(t)] = t
    return Layout(tables, np.asarray(lens, dtype=np.int32),
                  np.asarray(step_slots, dtype=np.int64),
                  np.asarray(pre_copies, dtype=np.int64).reshape(-1, 2),
                  np.asarray(pre_slots, dtype=np.int64),
                  np.asarray(step_copies, dtype=np.int64).reshape(-1, 2),
                  int(max(lens)) if lens else 0)


def native_allocator(plan):
    """The library's allocator class that lays the plan out."""
    from . import api
    return api.PrefixCachePool if plan.apc else api.BlockAllocator


def torch_dtype(name):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16}[name]


def normal(shape, dtype, device, seed):
    """N(0, 1) values of a 16-bit type, from a seeded torch generator on the
    given device."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(shape, generator=g, dtype=dtype, device=device)


@dataclass
class Values:
    q: object
    k_pools: list
    v_pools: list
    k_new: list
    v_new: list
    k_pre: list
    v_pre: list


def make_values(plan, lay, device, layers=None):
    """Random tensors for the plan on `device` (pools, q, new tokens, and the
    tokens written before the step).  `layers` limits how many layers are
    made (default: all of the workload's)."""
    spec = plan.spec
    dt = torch_dtype(spec.dtype)
    L = spec.num_layers if layers is None else layers
    S, hq, hkv, d, B = (spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                        spec.block_size)
    base = spec.seed * 100003
    q = normal((S, hq, d), dt, device, base + 1)
    kp, vp, kn, vn, kpre, vpre = [], [], [], [], [], []
    npre = int(lay.pre_slots.size)
    for layer in range(L):
        s0 = base + 1000 * (layer + 1)
        kp.append(normal((plan.num_blocks, hkv, B, d), dt, device, s0 + 1))
        vp.append(normal((plan.num_blocks, hkv, B, d), dt, device, s0 + 2))
        kn.append(normal((S, hkv, d), dt, device, s0 + 3))
        vn.append(normal((S, hkv, d), dt, device, s0 + 4))
        if npre:
            kpre.append(normal((npre, hkv, d), dt, device, s0 + 5))
            vpre.append(normal((npre, hkv, d), dt, device, s0 + 6))
    return Values(q, kp, vp, kn, vn, kpre, vpre)


def algorithmic_bytes(spec, seq_lens, kv_bytes=None):
    """Bytes the decode must move for one layer (K and V of every cached
    token, the block-table entries used, q in, out, the length word).
    kv_bytes: bytes per K/V element when the pools differ from q (1 for
    E4M3 pools)."""
    b = DTYPE_BYTES[spec.dtype]
    L = np.asarray(seq_lens, dtype=np.int64)
    kv = 2 * L.sum() * spec.num_kv_heads * spec.head_dim * (kv_bytes or b)
    table = 4 * sum(_blocks(x, spec.block_size) for x in L)
    qo = 2 * len(L) * spec.num_q_heads * spec.head_dim * b
    return int(kv + table + qo + 4 * len(L))


def cache_write_bytes(spec, num_tokens, kv_bytes=None):
    """Bytes of one layer's cache write: read K and V of each token (16-bit)
    and write them into the pools (kv_bytes per element, default 16-bit)."""
    b = DTYPE_BYTES[spec.dtype]
    per = b + (kv_bytes or b)
    return int(2 * per * num_tokens * spec.num_kv_heads * spec.head_dim + 8 * num_tokens)


def cascade_bytes(spec, seq_lens, prefix_len):
    """Bytes a shared-prefix (cascade) decode must move for one layer: the
    prefix's K and V once per KV head, each sequence's tail, the block-table
    entries read (the prefix's once), q in and out, the length words."""
    b = DTYPE_BYTES[spec.dtype]
    L = np.asarray(seq_lens, dtype=np.int64)
    per_token = 2 * spec.num_kv_heads * spec.head_dim * b
    kv = per_token * (prefix_len + (L - prefix_len).sum())
    B = spec.block_size
    table = 4 * (prefix_len // B + sum(_blocks(x, B) - prefix_len // B for x in L))
    qo = 2 * len(L) * spec.num_q_heads * spec.head_dim * b
    return int(kv + table + qo + 4 * len(L))
