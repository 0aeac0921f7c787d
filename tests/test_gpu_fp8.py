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


class Fp8Case:
    """A workload's layout with E4M3 pools of random codes."""

    def __init__(self, name, seed=0, plan=None, **kw):
        self.plan = plan if plan is not None else workloads.make_plan(name, **kw)
        self.spec = spec = self.plan.spec
        self.lay = workloads.layout(self.plan, workloads.native_allocator(self.plan))
        shape = (self.plan.num_blocks, spec.num_kv_heads, spec.block_size, spec.head_dim)
        self.kp = codes_like(shape, 100 + seed)
        self.vp = codes_like(shape, 200 + seed)
        dt = workloads.torch_dtype(spec.dtype)
        self.q = workloads.normal((spec.num_seqs, spec.num_q_heads, spec.head_dim), dt, "cuda", 300 + seed)
        self.k_new = workloads.normal((spec.num_seqs, spec.num_kv_heads, spec.head_dim), dt, "cuda", 400 + seed)
        self.v_new = workloads.normal((spec.num_seqs, spec.num_kv_heads, spec.head_dim), dt, "cuda", 500 + seed)
        self.tables = torch.as_tensor(self.lay.block_tables, device="cuda")
        self.lens = torch.as_tensor(self.lay.seq_lens, device="cuda")
        self.slots = torch.as_tensor(self.lay.slot_mapping, device="cuda")
        self.max_seq_len = int(self.lay.max_seq_len)
        self.k_scale, self.v_scale = 1.0 / 16, 0.37

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
