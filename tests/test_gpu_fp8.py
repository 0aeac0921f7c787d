"""GPU parity of the FP8 (E4M3) KV-cache variant against the fp64 oracle:
the quantising cache write bit-exact, the decode within the output
tolerance, over the shapes of the workloads."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_64_gb300 import api, workloads

from _parity import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_errors():
    assert torch.cuda.is_available()
    yield
    api.check_error()


def codes_like(shape, seed):
    """Random finite E4M3 codes with magnitudes 2^-3 .. 15 (exponent fields
    4 .. 10) and random signs."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    mag = torch.randint(0x20, 0x58, shape, generator=g, device="cuda", dtype=torch.int32)
    sign = torch.randint(0, 2, shape, generator=g, device="cuda", dtype=torch.int32) << 7
    return (mag | sign).to(torch.uint8)


def np_codes(t):
    return t.cpu().numpy().astype(np.uint8)


# Every finite E4M3 code: 0x00..0x7E and 0x80..0xFE (0x7F and 0xFF are NaN):
# zeros, the subnormals 0x01..0x07 (2^-9 .. 7 * 2^-9), normals up to 0x7E = 448.
FINITE_CODES = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def full_range_codes(shape, seed):
    """Codes drawn uniformly from every finite E4M3 code."""
    rng = np.random.default_rng(seed)
    return torch.as_tensor(rng.choice(FINITE_CODES, shape), device="cuda")


class Fp8Case:
    """A workload's layout with E4M3 pools of random codes.  `codes(shape,
    seed)` draws the pools' codes; `scales` are (k_scale, v_scale)."""

    def __init__(self, name, seed=0, plan=None, codes=codes_like, scales=(1.0 / 16, 0.37), **kw):
        self.plan = plan if plan is not None else workloads.make_plan(name, **kw)
        self.spec = spec = self.plan.spec
        self.lay = workloads.layout(self.plan, workloads.native_allocator(self.plan))
        shape = (self.plan.num_blocks, spec.num_kv_heads, spec.block_size, spec.head_dim)
        self.kp = codes(shape, 100 + seed)
        self.vp = codes(shape, 200 + seed)
        dt = workloads.torch_dtype(spec.dtype)
        self.q = workloads.normal((spec.num_seqs, spec.num_q_heads, spec.head_dim), dt, "cuda", 300 + seed)
        self.k_new = workloads.normal((spec.num_seqs, spec.num_kv_heads, spec.head_dim), dt, "cuda", 400 + seed)
        self.v_new = workloads.normal((spec.num_seqs, spec.num_kv_heads, spec.head_dim), dt, "cuda", 500 + seed)
        self.tables = torch.as_tensor(self.lay.block_tables, device="cuda")
        self.lens = torch.as_tensor(self.lay.seq_lens, device="cuda")
        self.slots = torch.as_tensor(self.lay.slot_mapping, device="cuda")
        self.max_seq_len = int(self.lay.max_seq_len)
        self.k_scale, self.v_scale = scales

    def gpu(self, partition=0, step=False, workspace=None):
        out = torch.full_like(self.q, float("nan"))
        kw = dict(k_new=self.k_new, v_new=self.v_new, slot_mapping=self.slots) if step else {}
        api.decode_fp8(out, self.q, self.kp, self.vp, self.tables, self.lens, self.max_seq_len,
                       self.plan.scale, self.k_scale, self.v_scale, partition_tokens=partition,
                       workspace=workspace, **kw)
        return out

    def oracle(self, kc, vc, step=False, seqs=None):
        if step:
            oracle.cache_write_fp8(kc, vc, bits(self.k_new), bits(self.v_new), self.lay.slot_mapping,
                                   self.spec.dtype, self.k_scale, self.v_scale)
        return oracle.decode_fp8(bits(self.q), kc, vc, self.lay.block_tables, self.lay.seq_lens,
                                 self.plan.scale, self.spec.dtype, self.k_scale, self.v_scale,
                                 seqs=seqs)


# ------------------------------------------------------------------ cache write
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
def test_cache_write_fp8_bit_exact(dtype, d):
    rng = np.random.default_rng(d + (dtype == "bf16"))
    T, hkv, B, nb = 300, 2, 16, 64
    tdt = workloads.torch_dtype(dtype)
    x = rng.standard_normal((T, hkv, d)) * rng.choice([1e-3, 0.1, 1.0, 30.0, 1e4], (T, 1, 1))
    x[0, 0, :8] = [1.0625, 1.1875, -0.0, 0.0, 464.0, -500.0, 2.0**-10, 3 * 2.0**-11]  # ties, saturation, underflow
    k_new = torch.tensor(x, dtype=tdt, device="cuda")
    v_new = torch.tensor(-x * 0.5, dtype=tdt, device="cuda")
    slots = rng.permutation(nb * B)[:T].astype(np.int64)
    slots[5] = -1                                          # skipped
    kp = torch.zeros((nb, hkv, B, d), dtype=torch.uint8, device="cuda")
    vp = torch.zeros_like(kp)
    for ks, vs in ((1.0, 1.0), (0.037, 3.3)):
        kp.zero_()
        vp.zero_()
        api.cache_write_fp8(k_new, v_new, torch.as_tensor(slots, device="cuda"), kp, vp, ks, vs)
        api.check_error()
        rk = np.zeros(tuple(kp.shape), np.uint8)
        rv = np.zeros(tuple(vp.shape), np.uint8)
        oracle.cache_write_fp8(rk, rv, bits(k_new), bits(v_new), slots, dtype, ks, vs)
        assert np.array_equal(np_codes(kp), rk), f"K codes differ (scales {ks})"
        assert np.array_equal(np_codes(vp), rv), f"V codes differ (scales {vs})"


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("name,kw,partition", [
    ("tiny", {}, -1),
    ("tiny", {}, 16),
    ("qwen", {"num_seqs": 24}, 0),
    ("qwen", {"num_seqs": 24}, -1),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 0),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 256),
    ("prefix", {"num_seqs": 6}, 0),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512),  # > 8 partitions: reduce kernel
])
def test_decode_fp8_every_output(name, kw, partition):
    c = Fp8Case(name, **kw)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, c.oracle(kc, vc), f"fp8 {name} P={partition}")


@pytest.mark.parametrize("name,kw,partition", [
    ("tiny", {}, -1),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 512),
    ("qwen", {"num_seqs": 24}, 0),
])
def test_decode_fp8_fused_step(name, kw, partition):
    c = Fp8Case(name, seed=3, **kw)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition, step=True)
    api.check_error()
    ref = c.oracle(kc, vc, step=True)
    assert_close(out, ref, f"fp8 fused step {name}")
    assert np.array_equal(np_codes(c.kp), kc) and np.array_equal(np_codes(c.vp), vc)


def test_decode_fp8_full_size_llama_sampled():
    c = Fp8Case("llama", seed=5)
    lens = c.lay.seq_lens
    rng = np.random.default_rng(7)
    seqs = sorted({int(np.argmax(lens)), int(np.argmin(lens))} | set(rng.choice(len(lens), 6, replace=False).tolist()))
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(0, step=True)
    api.check_error()
    ref = c.oracle(kc, vc, step=True, seqs=seqs)
    assert_close(out, ref, "fp8 llama full size", mask_rows=np.asarray(seqs))


def test_decode_fp8_stale_slots_poisoned_with_nan():
    c = Fp8Case("long", seed=7, num_seqs=2, len_range=(1000, 1500))
    B = c.spec.block_size
    used = np.zeros(c.plan.num_blocks, dtype=bool)
    for s, L in enumerate(c.lay.seq_lens):
        nb = -(-int(L) // B)
        used[c.lay.block_tables[s, :nb]] = True
        last = c.lay.block_tables[s, nb - 1]
        for p in range(int(L), nb * B):
            c.kp[last, :, p % B, :] = 0x7F  # NaN code
            c.vp[last, :, p % B, :] = 0xFF
    unused = torch.as_tensor(np.flatnonzero(~used), device="cuda")
    c.kp[unused] = 0x7F
    c.vp[unused] = 0x7F
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    for P in (-1, 512, 160):
        out = c.gpu(P)
        assert torch.isfinite(out).all()
        assert_close(out, c.oracle(kc, vc), f"fp8 poison P={P}")


def test_decode_fp8_zero_and_one_token():
    c = Fp8Case("tiny", seed=9)
    lens = c.lay.seq_lens.copy()
    lens[0], lens[1] = 0, 1
    c.lay.seq_lens = lens
    c.lens = torch.as_tensor(lens, device="cuda")
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    for P in (-1, 16):
        out = c.gpu(P)
        assert torch.all(out[0] == 0)
        assert_close(out, c.oracle(kc, vc), f"fp8 edge P={P}")


def test_fp8_rejects_bad_scale():
    from paged_kv_cache_64_gb300 import _lib
    c = Fp8Case("tiny")
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.decode_fp8(torch.empty_like(c.q), c.q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len,
                       c.plan.scale, 0.0, 1.0)
    assert e.value.code == 1


# ------------------------------------------- several partitions per CTA
@pytest.fixture
def span():
    prev = []

    def set_span(n):
        prev.append(api.set_decode_span(n))

    yield set_span
    if prev:
        api.set_decode_span(prev[0])


@pytest.mark.parametrize("name,kw,partition,R", [
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512, 2),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512, 3),   # ragged last span
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 256, 4),   # 2 tiles a partition
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 512, 4),
    ("llama", {"num_seqs": 6, "len_range": (100, 900)}, 256, 8),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 128, 3),   # one tile a partition
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 128, 5),
])
def test_decode_fp8_partitions_per_cta_every_output(span, name, kw, partition, R):
    span(R)
    c = Fp8Case(name, **kw)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, c.oracle(kc, vc), f"fp8 span {name} P={partition} R={R}")


@pytest.mark.parametrize("R", [2, 4])
def test_decode_fp8_fused_step_partitions_per_cta(span, R):
    span(R)
    c = Fp8Case("long", seed=11, num_seqs=2, len_range=(1000, 1900))
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(256, step=True)
    api.check_error()
    ref = c.oracle(kc, vc, step=True)
    assert_close(out, ref, "fp8 fused step, span")
    assert np.array_equal(np_codes(c.kp), kc) and np.array_equal(np_codes(c.vp), vc)


def test_decode_fp8_partitions_per_cta_stale_slots_poisoned(span):
    span(4)
    c = Fp8Case("long", seed=13, num_seqs=2, len_range=(1000, 1500))
    B = c.spec.block_size
    for s, L in enumerate(c.lay.seq_lens):
        nb = -(-int(L) // B)
        last = c.lay.block_tables[s, nb - 1]
        for p in range(int(L), nb * B):
            c.kp[last, :, p % B, :] = 0x7F
            c.vp[last, :, p % B, :] = 0xFF
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(256)
    assert torch.isfinite(out).all()
    assert_close(out, c.oracle(kc, vc), "fp8 span poison")


# ------------------------------------------- the whole E4M3 format
# Pools of codes drawn from every finite E4M3 code (subnormals, zeros, +-448)
# with the scales a cache of values up to about 7 in magnitude would use
# (amax / 448 = 1/64), through single pass, the fused combine, the combine
# kernel, several partitions a CTA and the fused cache write; head dims 64 and
# 128, groups padded to 4 and to 8 query heads.
FULL_SCALES = (1.0 / 64, 1.0 / 64)
# (q heads, KV heads, head_dim, block_size, dtype): G = 4 and 8 at d = 64 and 128
FULL_SHAPES = {
    "g4_d64": (16, 4, 64, 16, "f16"),
    "g8_d64": (16, 2, 64, 32, "bf16"),
    "g4_d128": (8, 2, 128, 16, "bf16"),
    "g8_d128": (16, 2, 128, 16, "f16"),
}


def full_plan(name, seed=0, lens=(0, 1500), num_seqs=5):
    hq, hkv, d, B, dt = FULL_SHAPES[name]
    return workloads.make_shape_plan(num_seqs, hq, hkv, d, B, dt, lens, seed=41 + seed)


def used_codes(c):
    """The set of codes the sequences' valid positions hold (K and V)."""
    B = c.spec.block_size
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    seen = set()
    for s, L in enumerate(c.lay.seq_lens):
        for p in range(int(L)):
            blk = c.lay.block_tables[s, p // B]
            seen.update(np.unique(kc[blk, :, p % B]).tolist())
            seen.update(np.unique(vc[blk, :, p % B]).tolist())
    return seen


@pytest.mark.parametrize("name", sorted(FULL_SHAPES))
@pytest.mark.parametrize("partition,fused,R", [
    (-1, False, 1),    # single pass
    (512, True, 1),    # fused cache write, partials combined inside the launch
    (128, False, 1),   # > 8 partitions: the combine kernel
    (256, False, 2),   # two partitions a CTA
])
def test_decode_fp8_every_finite_code(span, name, partition, fused, R):
    span(R)
    c = Fp8Case("shape", seed=1, plan=full_plan(name), codes=full_range_codes, scales=FULL_SCALES)
    assert used_codes(c) >= set(FINITE_CODES.tolist())  # every finite code is read
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition, step=fused)
    api.check_error()
    assert_close(out, c.oracle(kc, vc, step=fused), f"fp8 all codes {name} P={partition} R={R}")


def log_uniform_q(shape, dtype, seed, span_log2=25):
    """Random signs, magnitudes 2^U(-22, 3): a row spans about 2^25."""
    rng = np.random.default_rng(seed)
    x = rng.choice([-1.0, 1.0], shape) * 2.0 ** rng.uniform(-22, 3, shape)
    return torch.as_tensor(x, dtype=workloads.torch_dtype(dtype), device="cuda")


@pytest.mark.parametrize("name", sorted(FULL_SHAPES))
@pytest.mark.parametrize("partition", [-1, 256])
def test_decode_fp8_q_rows_spanning_2_25(name, partition):
    """q elements from 2^-22 to 2^3 in one row: the small ones sit far below
    the row's largest, where a split of q into terms with one scale a head
    loses them unless its floor is low enough."""
    c = Fp8Case("shape", seed=2, plan=full_plan(name, seed=2), codes=full_range_codes,
                scales=FULL_SCALES)
    c.q = log_uniform_q(tuple(c.q.shape), c.spec.dtype, 5)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, c.oracle(kc, vc), f"fp8 q spanning 2^25 {name} P={partition}")


def fill_pools(c, k, v):
    """Overwrite the pools with host code arrays of the pools' shape."""
    c.kp.copy_(torch.as_tensor(k, device="cuda"))
    c.vp.copy_(torch.as_tensor(v, device="cuda"))


@pytest.mark.parametrize("name", sorted(FULL_SHAPES))
@pytest.mark.parametrize("partition", [-1, 512])
def test_decode_fp8_small_q_elements_against_large_keys(name, partition):
    """Each head: one q element of about 1000 whose key column holds
    subnormal codes, every other element about 2^-17.6 of it, their key
    columns all +448 or all -448 (by position).  The scores' differences then
    come entirely from the small elements (about +-0.4 after scaling)."""
    c = Fp8Case("shape", seed=3, plan=full_plan(name, seed=3), codes=full_range_codes,
                scales=FULL_SCALES)
    rng = np.random.default_rng(11)
    shape = tuple(c.kp.shape)
    k = np.empty(shape, np.uint8)
    k[..., 0] = rng.integers(1, 8, shape[:-1]) | (rng.integers(0, 2, shape[:-1]) << 7)
    k[..., 1:] = np.where(rng.random(shape[:-1] + (1,)) < 0.5, 0x7E, 0xFE)
    fill_pools(c, k, np_codes(c.vp))
    S, Hq, d = c.q.shape
    big = 1000.0 * rng.uniform(0.7, 1.4, (S, Hq))
    q = np.empty((S, Hq, d))
    q[..., 0] = big
    q[..., 1:] = (big * 2.0 ** -17.6)[..., None] * rng.uniform(0.8, 1.2, (S, Hq, d - 1))
    c.q = torch.as_tensor(q, dtype=workloads.torch_dtype(c.spec.dtype), device="cuda")
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, c.oracle(kc, vc), f"fp8 small q elements {name} P={partition}")


@pytest.mark.parametrize("name", sorted(FULL_SHAPES))
@pytest.mark.parametrize("partition", [-1, 256])
def test_decode_fp8_output_from_weights_near_2_minus_17(name, partition):
    """The first position of every 128-position tile has a score about 17.5
    (log2 units) above the rest and a value row of zeros; the other
    positions' values are +448 codes (56 with the V scale 1/8).  The output
    is then made only of weights 2^-16.5 .. 2^-18.5 of the largest, the range
    where a split of P into terms meets its floor."""
    c = Fp8Case("shape", seed=4, plan=full_plan(name, seed=4), codes=full_range_codes,
                scales=(FULL_SCALES[0], 1.0 / 8))
    rng = np.random.default_rng(13)
    shape = tuple(c.kp.shape)
    d, B = shape[-1], c.spec.block_size
    top = np.zeros(shape[:-1], bool)
    for s, L in enumerate(c.lay.seq_lens):
        for p in range(0, int(L), 128):
            top[c.lay.block_tables[s, p // B], :, p % B] = True
    k = np.zeros(shape, np.uint8)
    # 448 at the top positions, 160 / 176 / 192 at the others (score gaps of
    # 18.5 / 17.5 / 16.5 in log2 units with q0 below)
    low = oracle.e4m3_encode(rng.choice([160.0, 176.0, 192.0], shape[:-1]))
    k[..., 0] = np.where(top, 0x7E, low)
    v = np.where(top[..., None], 0x00, 0x7E).astype(np.uint8) * np.ones((1, 1, 1, d), np.uint8)
    fill_pools(c, k, v)
    S, Hq, _ = c.q.shape
    q0 = 17.5 * np.log(2) / (c.plan.scale * FULL_SCALES[0] * (448 - 176))
    q = np.zeros((S, Hq, d))
    q[..., 0] = q0
    c.q = torch.as_tensor(q, dtype=workloads.torch_dtype(c.spec.dtype), device="cuda")
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    ref = c.oracle(kc, vc)
    # the outputs (about 0.045) come from the tiny weights only
    assert 0.02 < np.abs(ref).max() < 0.1
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, ref, f"fp8 tiny weights {name} P={partition}")


# ------------------------------------------- group sizes and compact grids
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7])
@pytest.mark.parametrize("partition", [-1, 256])
def test_decode_fp8_group_sizes(G, d, partition):
    """Groups of 1..7 query heads a KV head (8 and 4 are covered above): the
    q and P terms of the absent heads of an 8-head operand must not reach
    the present heads' outputs.  Every finite code, every output."""
    plan = workloads.make_shape_plan(4, 2 * G, 2, d, 16, "bf16" if G % 2 else "f16", (1, 700),
                                     seed=90 + G + d)
    c = Fp8Case("shape", seed=G, plan=plan, codes=full_range_codes, scales=FULL_SCALES)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition)
    api.check_error()
    assert_close(out, c.oracle(kc, vc), f"fp8 G={G} d={d} P={partition}")


@pytest.mark.parametrize("hq,hkv,d,dtype,num_seqs,lens,partition,fused", [
    (14, 2, 64, "f16", 100, (2000, 3000), 512, False),   # ~1,000 items over the resident slots
    (14, 2, 64, "f16", 100, (2000, 3000), 512, True),    # the same, fused cache write
    (32, 8, 128, "bf16", 40, (1100, 1500), 512, True),   # d = 128: 960 items
])
def test_decode_fp8_compact_several_items_per_cta(span, hq, hkv, d, dtype, num_seqs, lens,
                                                   partition, fused):
    """A compact launch over E4M3 pools with more items than resident CTA
    slots but within four waves: each CTA computes several items in turn.
    Every output."""
    span(1)
    plan = workloads.make_shape_plan(num_seqs, hq, hkv, d, 16, dtype, lens, seed=81 + d)
    c = Fp8Case("shape", seed=9, plan=plan, codes=full_range_codes, scales=FULL_SCALES)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition, step=fused)
    api.check_error()
    assert_close(out, c.oracle(kc, vc, step=fused), f"fp8 several items a CTA d={d} fused={fused}")


# ------------------------------------------- garbage workspace, graph replay
@pytest.mark.parametrize("name,kw,partition", [
    ("llama", {"num_seqs": 6, "len_range": (900, 2100)}, 512),   # ready flags (one wave)
    ("qwen", {"num_seqs": 100}, 0),                             # compact grid, flags or counters
])
def test_decode_fp8_garbage_workspace_and_graph_replay(name, kw, partition):
    """Over E4M3 pools: the fused combine needs no initialised workspace, and
    a CUDA graph of the decode replays correctly (each replay reuses the
    captured epoch; the combining CTA clears the flags it read)."""
    c = Fp8Case(name, seed=21, codes=full_range_codes, scales=FULL_SCALES, **kw)
    spec = c.spec
    size = api.fp8_workspace_size(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads,
                                  spec.head_dim, spec.block_size, c.max_seq_len, partition,
                                  c.q.dtype)
    ws = api.alloc_workspace(size, "cuda")
    ws.fill_(0xFF)
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    ref = c.oracle(kc, vc)
    out = torch.empty_like(c.q)

    def run():
        api.decode_fp8(out, c.q, c.kp, c.vp, c.tables, c.lens, c.max_seq_len, c.plan.scale,
                       c.k_scale, c.v_scale, partition_tokens=partition, workspace=ws)

    run()
    api.check_error()
    assert_close(out, ref, f"fp8 garbage workspace {name}")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            run()
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, f"fp8 graph replay {name}")
    api.check_error()
