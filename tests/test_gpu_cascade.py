"""GPU parity of the shared-prefix (cascade) decode against the fp64 oracle.

The oracle knows nothing of the cascade: it attends each sequence over all
of its positions through its block table.  The library computes the shared
prefix once per KV head for every sequence's queries (tensor-core prefix
pass), each tail separately, and merges the two; both must agree within the
output tolerance, and the fused cache write must be bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.allocator import BlockAllocatorModel
from paged_kv_cache_64_gb300 import _lib, api, workloads

from _parity import Case, assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_errors():
    assert torch.cuda.is_available()
    prev = api.get_decode_impl()
    yield
    api.set_decode_impl(prev)
    api.check_error()


# ------------------------------------------------------------ the prefix workload
def cascade_step(case, prefix_len):
    """Copies and earlier writes, then the cascade with the fused write."""
    case.gpu_pre_writes(0)
    out = torch.empty_like(case.vals.q)
    api.decode_cascade(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                       case.lens, case.max_seq_len, case.plan.scale, prefix_len,
                       k_new=case.vals.k_new[0], v_new=case.vals.v_new[0], slot_mapping=case.slots)
    return out


@pytest.mark.parametrize("cow", [False, True])
def test_prefix_workload_small(cow):
    case = Case(workloads.make_plan("prefix", num_seqs=6, cow=cow))
    hk, hv = case.snapshot(0)
    out = cascade_step(case, 4096)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    assert_close(out, ref, f"cascade prefix cow={cow}")
    # the fused write left the pools exactly as the oracle's writes did
    assert np.array_equal(bits(case.vals.k_pools[0]), hk)
    assert np.array_equal(bits(case.vals.v_pools[0]), hv)


@pytest.mark.parametrize("cow", [False, True])
def test_prefix_workload_full_size_sampled(cow):
    case = Case(workloads.make_plan("prefix", cow=cow))
    lens = case.lay.seq_lens
    rng = np.random.default_rng(21)
    seqs = {int(np.argmax(lens)), int(np.argmin(lens)), 0, len(lens) - 1, 31, 32}
    seqs.update(rng.choice(len(lens), 8, replace=False).tolist())
    seqs = sorted(seqs)
    # whole pools: the copy-on-write sources need not be in the sampled tables
    hk, hv = case.snapshot(0)
    out = cascade_step(case, 4096)
    ref = case.oracle_step(0, hk, hv, seqs)
    api.check_error()
    assert_close(out, ref, f"cascade full prefix cow={cow}", mask_rows=np.asarray(seqs))


def test_cascade_matches_plain_decode():
    """Same inputs through pa_decode and pa_decode_cascade: both match the
    oracle, and each other, within the output tolerance."""
    case = Case(workloads.make_plan("prefix", num_seqs=20, cow=True))
    hk, hv = case.snapshot(0)
    case.gpu_writes(0)
    ref = case.oracle_step(0, hk, hv)
    plain = case.gpu_decode(0)
    out = torch.empty_like(plain)
    api.decode_cascade(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                       case.lens, case.max_seq_len, case.plan.scale, 4096)
    api.check_error()
    assert_close(plain, ref, "plain vs oracle")
    assert_close(out, ref, "cascade vs oracle")
    assert_close(out, plain.double().cpu().numpy(), "cascade vs plain")


# ------------------------------------------------------------ other shapes
class SharedPrefix:
    """S sequences forked from one prompt of prefix_len tokens, each then
    holding tails[s] more cached tokens (+1 new token when step)."""

    def __init__(self, S, hq, hkv, d, B, dtype, prefix_len, tails, seed, step):
        rng = np.random.default_rng(seed)
        tails = np.asarray(tails, dtype=np.int64)
        nb = prefix_len // B + int(sum(-(-(t + 1) // B) + 1 for t in tails)) + 8
        alloc = BlockAllocatorModel(nb, B, free_order=rng.permutation(nb))
        alloc.add(0)
        alloc.append(0, prefix_len)
        for s in range(1, S):
            alloc.fork(0, s)
        copies = []
        for s in range(S):
            copies += alloc.append(s, int(tails[s]))[1]
        assert not copies  # prefix_len is whole blocks: nothing shared is written
        slots = []
        if step:
            for s in range(S):
                sl, cp = alloc.append(s, 1)
                assert not cp
                slots += sl
        lens = np.array([alloc.length(s) for s in range(S)], dtype=np.int32)
        maxb = max(-(-int(L) // B) for L in lens)
        tables = np.zeros((S, maxb), dtype=np.int32)
        for s in range(S):
            t = alloc.table(s)
            tables[s, :len(t)] = t
        self.S, self.hq, self.hkv, self.d, self.B = S, hq, hkv, d, B
        self.dtype, self.prefix_len, self.step = dtype, prefix_len, step
        self.tables_np, self.lens_np = tables, lens
        self.max_seq_len = int(lens.max())
        self.scale = 1.0 / np.sqrt(d)
        dt = workloads.torch_dtype(dtype)
        base = seed * 7919
        self.q = workloads.normal((S, hq, d), dt, "cuda", base + 1)
        self.kp = workloads.normal((nb, hkv, B, d), dt, "cuda", base + 2)
        self.vp = workloads.normal((nb, hkv, B, d), dt, "cuda", base + 3)
        self.k_new = workloads.normal((S, hkv, d), dt, "cuda", base + 4)
        self.v_new = workloads.normal((S, hkv, d), dt, "cuda", base + 5)
        self.slots_np = np.asarray(slots, dtype=np.int64)
        self.tables = torch.as_tensor(tables, device="cuda")
        self.lens = torch.as_tensor(lens, device="cuda")
        self.slots = torch.as_tensor(self.slots_np, device="cuda")

    def run(self, prefix_len=None):
        out = torch.full_like(self.q, float("nan"))
        kw = {}
        if self.step:
            kw = dict(k_new=self.k_new, v_new=self.v_new, slot_mapping=self.slots)
        api.decode_cascade(out, self.q, self.kp, self.vp, self.tables, self.lens,
                           self.max_seq_len, self.scale,
                           self.prefix_len if prefix_len is None else prefix_len, **kw)
        return out

    def oracle(self, hk, hv):
        if self.step:
            oracle.cache_write(hk, hv, bits(self.k_new), bits(self.v_new), self.slots_np)
        return oracle.decode(bits(self.q), hk, hv, self.tables_np, self.lens_np, self.scale,
                             self.dtype)


SHAPES = {
    # name: (S, hq, hkv, d, B, dtype, prefix_len, tail range, step)
    # 1,008 = 7 full tiles of 128 and one of 112; 280 query rows = 3 row tiles, the last ragged;
    # tails from 0 (the sequence is all prefix) upwards
    "qwen_g7_partial_tile": (40, 14, 2, 64, 16, "f16", 1008, (0, 300), False),
    # long tails: the tail pass splits into partitions (ready flags)
    "g8_long_tails": (5, 64, 8, 128, 16, "bf16", 2048, (1000, 3000), True),
    # one query head per KV head; 130 rows = 2 row tiles
    "mha_b32": (130, 4, 4, 128, 32, "bf16", 512, (1, 64), True),
    # a one-block prefix and a single sequence
    "single_seq_one_block": (1, 8, 2, 64, 32, "f16", 32, (5, 5), True),
}


@pytest.mark.parametrize("impl", ["auto", "cuda_cores"])
@pytest.mark.parametrize("name", sorted(SHAPES))
def test_shapes(name, impl):
    S, hq, hkv, d, B, dtype, P, (lo, hi), step = SHAPES[name]
    rng = np.random.default_rng(len(name))
    tails = rng.integers(lo, hi, S, endpoint=True)
    if lo == 0:
        tails[:3] = 0  # empty tails
    c = SharedPrefix(S, hq, hkv, d, B, dtype, P, tails, seed=len(name) + 3, step=step)
    hk, hv = bits(c.kp), bits(c.vp)
    api.set_decode_impl(impl)
    out = c.run()
    api.check_error()
    ref = c.oracle(hk, hv)
    assert_close(out, ref, f"cascade {name} {impl}")
    if step:
        assert np.array_equal(bits(c.kp), hk) and np.array_equal(bits(c.vp), hv)


def test_prefix_len_zero_is_plain_decode():
    c = SharedPrefix(6, 8, 2, 128, 16, "bf16", 256, np.full(6, 40), seed=5, step=False)
    hk, hv = bits(c.kp), bits(c.vp)
    out = c.run(prefix_len=0)
    api.check_error()
    assert_close(out, c.oracle(hk, hv), "cascade P=0")


def test_shorter_prefix_than_shared():
    """Any whole-block prefix of the shared one gives the same result."""
    c = SharedPrefix(9, 32, 8, 128, 32, "bf16", 1024, np.arange(9) * 13, seed=6, step=False)
    hk, hv = bits(c.kp), bits(c.vp)
    ref = c.oracle(hk, hv)
    for P in (32, 512, 1024):
        out = c.run(prefix_len=P)
        api.check_error()
        assert_close(out, ref, f"cascade P={P}")


def test_unshared_prefix_is_reported():
    c = SharedPrefix(4, 8, 2, 64, 16, "f16", 256, np.full(4, 20), seed=8, step=False)
    t = c.tables.clone()
    t[2, 3] = t[2, -1] if t[2, -1] != t[0, 3] else t[1, -1]  # a valid block, not the shared one
    out = torch.empty_like(c.q)
    api.decode_cascade(out, c.q, c.kp, c.vp, t, c.lens, c.max_seq_len, c.scale, 256)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6  # PA_ERR_BAD_INDEX


def test_short_sequence_is_reported():
    c = SharedPrefix(4, 8, 2, 64, 16, "f16", 256, np.full(4, 20), seed=9, step=False)
    lens = c.lens.clone()
    lens[1] = 100  # shorter than the prefix
    out = torch.empty_like(c.q)
    api.decode_cascade(out, c.q, c.kp, c.vp, c.tables, lens, c.max_seq_len, c.scale, 256)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6


def test_invalid_prefix_len_rejected_on_host():
    c = SharedPrefix(2, 8, 2, 64, 16, "f16", 64, np.full(2, 3), seed=10, step=False)
    out = torch.empty_like(c.q)
    for P in (24, c.max_seq_len + 16, -16):
        with pytest.raises(_lib.PagedAttentionError) as e:
            api.decode_cascade(out, c.q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.scale, P)
        assert e.value.code == 1


def test_graph_replay():
    """Captured once, replayed: the same output each time (the workspace is
    scratch and its ready flags carry over between replays)."""
    c = SharedPrefix(5, 64, 8, 128, 16, "bf16", 2048, np.array([1200, 2900, 5, 2000, 1700]),
                     seed=11, step=False)
    hk, hv = bits(c.kp), bits(c.vp)
    ref = c.oracle(hk, hv)
    out = torch.empty_like(c.q)
    ws = api.alloc_workspace(api.cascade_workspace_size(c.S, c.hq, c.hkv, c.d, c.B,
                                                        c.max_seq_len, 2048, c.q.dtype), "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.decode_cascade(out, c.q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.scale, 2048,
                           workspace=ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.decode_cascade(out, c.q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.scale, 2048,
                           workspace=ws, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, "cascade graph replay")


@pytest.mark.parametrize("name", ["mha_b32", "g8_long_tails"])
def test_back_to_back_calls_chain_outputs(name):
    """Layers run back to back on one stream, each call's q the previous
    call's output, one workspace for all: the tail pass may start while the
    prefix pass runs, and must still see every earlier write (the previous
    layer's output) and leave the next prefix pass its workspace.  Every
    output equals the same call made alone between device-wide synchronizes,
    bit for bit; the first also matches the oracle."""
    S, hq, hkv, d, B, dtype, P, (lo, hi), step = SHAPES[name]
    tails = np.random.default_rng(5).integers(lo, hi, S, endpoint=True)
    c = SharedPrefix(S, hq, hkv, d, B, dtype, P, tails, seed=17, step=step)
    hk, hv = bits(c.kp), bits(c.vp)
    kw = dict(k_new=c.k_new, v_new=c.v_new, slot_mapping=c.slots) if step else {}
    ws = api.alloc_workspace(api.cascade_workspace_size(c.S, c.hq, c.hkv, c.d, c.B,
                                                        c.max_seq_len, P, c.q.dtype), "cuda")
    layers = 4
    outs = [torch.full_like(c.q, float("nan")) for _ in range(layers)]
    q = c.q
    for layer in range(layers):
        api.decode_cascade(outs[layer], q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.scale,
                           P, workspace=ws, **kw)
        q = outs[layer]
    torch.cuda.synchronize()
    api.check_error()
    assert_close(outs[0], c.oracle(hk, hv), f"cascade {name} first layer")
    q = c.q
    for layer in range(layers):
        alone = torch.full_like(c.q, float("nan"))
        torch.cuda.synchronize()
        api.decode_cascade(alone, q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.scale, P,
                           workspace=ws, **kw)
        torch.cuda.synchronize()
        assert np.array_equal(bits(alone), bits(outs[layer])), f"layer {layer}"
        q = outs[layer]


# ------------------------------------------------------------ prefix caching layout
@pytest.mark.parametrize("cascade", [False, True])
def test_prefix_caching_layout_small(cascade):
    """Separate requests with one prompt, laid out by the prefix-caching pool:
    plain decode and the cascade both match the oracle."""
    case = Case(workloads.make_plan("prefix", num_seqs=6, apc=True))
    hk, hv = case.snapshot(0)
    if cascade:
        out = cascade_step(case, 4096)
    else:
        out = case.gpu_step_fused(0)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    assert_close(out, ref, f"prefix caching layout, cascade={cascade}")
    assert np.array_equal(bits(case.vals.k_pools[0]), hk)


def test_prefix_caching_layout_full_size_sampled():
    case = Case(workloads.make_plan("prefix", apc=True))
    lens = case.lay.seq_lens
    seqs = sorted({0, 1, 31, 32, 63, int(np.argmax(lens)), int(np.argmin(lens))})
    hk, hv = case.snapshot(0)
    out = cascade_step(case, 4096)
    ref = case.oracle_step(0, hk, hv, seqs)
    api.check_error()
    assert_close(out, ref, "prefix caching layout full size", mask_rows=np.asarray(seqs))
