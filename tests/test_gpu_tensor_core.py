"""GPU parity of the tensor-core decode kernel (tcgen05 MMAs with TMEM
accumulators, K/V tiles by TMA tensor copies) against the fp64 oracle.

The kernel is forced for these tests (pa_set_decode_impl(2)), whatever the
automatic choice would be, so every group size and head dim it serves is
checked; the CUDA-core kernel is checked by test_gpu_parity.py and both are
compared with each other here.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_64_gb300 import api, workloads

from _parity import Case, assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tensor_cores():
    assert torch.cuda.is_available()
    prev = api.set_decode_impl("tensor_cores")
    yield
    api.set_decode_impl(prev)
    api.check_error()


def step_parity(case, partition=None, seqs=None):
    blocks = None if seqs is None else case.blocks_of(seqs)
    if case.lay.pre_copies.size:
        blocks = None
    hk, hv = case.snapshot(0, blocks)
    case.gpu_writes(0)
    out = case.gpu_decode(0, partition)
    ref = case.oracle_step(0, hk, hv, seqs)
    api.check_error()
    return assert_close(out, ref, "tensor cores " + case.spec.name,
                        mask_rows=None if seqs is None else np.asarray(seqs))


@pytest.mark.parametrize("partition", [-1, 16, 128, 0])
def test_tc_tiny(partition):
    step_parity(Case(workloads.make_plan("tiny")), partition=partition)


@pytest.mark.parametrize("name,kw,partition", [
    ("qwen", {"num_seqs": 24}, None),
    ("qwen", {"num_seqs": 24}, -1),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, None),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, -1),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 256),
    ("prefix", {"num_seqs": 6}, None),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, None),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, -1),
])
def test_tc_small_every_output(name, kw, partition):
    step_parity(Case(workloads.make_plan(name, **kw)), partition=partition)


def test_tc_prefix_cow_small():
    step_parity(Case(workloads.make_plan("prefix", num_seqs=6, cow=True)))


@pytest.mark.parametrize("name,cow,nsample", [("long", False, 3), ("qwen", False, 16),
                                             ("llama", False, 8), ("prefix", True, 6)])
def test_tc_full_size_sampled(name, cow, nsample):
    case = Case(workloads.make_plan(name, cow=cow))
    lens = case.lay.seq_lens
    rng = np.random.default_rng(12)
    seqs = {int(np.argmax(lens)), int(np.argmin(lens))}
    seqs.update(rng.choice(len(lens), nsample, replace=False).tolist())
    step_parity(case, seqs=sorted(seqs))


def test_tc_zero_and_one_token():
    case = Case(workloads.make_plan("tiny"))
    case.gpu_writes(0)
    lens = case.lay.seq_lens.copy()
    lens[0], lens[1] = 0, 1
    lens_t = torch.as_tensor(lens, device="cuda")
    for P in (-1, 16):
        out = torch.full_like(case.vals.q, float("nan"))
        api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                   lens_t, case.max_seq_len, case.plan.scale, partition_tokens=P)
        ref = oracle.decode(bits(case.vals.q), bits(case.vals.k_pools[0]),
                            bits(case.vals.v_pools[0]), case.ref_lay.block_tables, lens,
                            case.plan.scale, "f16")
        assert torch.all(out[0] == 0)
        assert_close(out, ref, f"tc edge P={P}")


def test_tc_stale_slots_poisoned_with_nan():
    case = Case(workloads.make_plan("long", num_seqs=2, len_range=(1000, 1500)))
    case.gpu_writes(0)
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    B = case.spec.block_size
    used = np.zeros(case.plan.num_blocks, dtype=bool)
    for s, L in enumerate(case.lay.seq_lens):
        nb = -(-int(L) // B)
        used[case.lay.block_tables[s, :nb]] = True
        last = case.lay.block_tables[s, nb - 1]
        for p in range(int(L), nb * B):
            kp[last, :, p % B, :] = float("nan")
            vp[last, :, p % B, :] = float("nan")
    unused = torch.as_tensor(np.flatnonzero(~used), device="cuda")
    kp[unused] = float("nan")
    vp[unused] = float("nan")
    for P in (-1, 512, 160):
        out = case.gpu_decode(0, partition=P)
        assert torch.isfinite(out).all()
        ref = oracle.decode(bits(case.vals.q), bits(kp), bits(vp), case.ref_lay.block_tables,
                            case.ref_lay.seq_lens, case.plan.scale, case.spec.dtype)
        assert_close(out, ref, f"tc poison P={P}")


def test_tc_partitions_match_oracle():
    case = Case(workloads.make_plan("long", num_seqs=2, len_range=(1500, 2600)))
    case.gpu_writes(0)
    spec, P = case.spec, 512
    ws = api.alloc_workspace(api.workspace_size(spec.num_seqs, spec.num_q_heads,
                                                spec.num_kv_heads, spec.head_dim,
                                                spec.block_size, case.max_seq_len, P,
                                                case.dtype), "cuda")
    api.decode_partitions(case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                          case.lens, case.max_seq_len, case.plan.scale, P, ws)
    m, l, o = api.partials_view(ws, spec.num_seqs, spec.num_q_heads, spec.head_dim,
                                case.max_seq_len, P)
    NP = api.partition_count(case.max_seq_len, P)
    rm, rl, ro = oracle.partitions(bits(case.vals.q), bits(case.vals.k_pools[0]),
                                   bits(case.vals.v_pools[0]), case.ref_lay.block_tables,
                                   case.ref_lay.seq_lens, case.plan.scale, spec.dtype, P, NP)
    gm = m.double().cpu().numpy() * np.log(2.0)
    gl, go = l.double().cpu().numpy(), o.double().cpu().numpy()
    empty = np.isinf(rm)
    assert np.array_equal(np.isinf(gm), empty)
    ok = ~empty
    assert np.max(np.abs(gm[ok] - rm[ok])) <= 1e-2 * (1 + np.max(np.abs(rm[ok])))
    # P rounded to bf16 before P.V: l and O carry that rounding (relative 2^-9)
    assert np.max(np.abs(gl[ok] - rl[ok]) / rl[ok]) <= 1e-4
    err = np.abs(go[ok] - ro[ok])
    assert (err <= 2e-3 + 1e-2 * np.abs(ro[ok])).all(), float(err.max())


@pytest.mark.parametrize("name,kw,partition", [
    ("qwen", {"num_seqs": 24}, None),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 512),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, None),
    ("tiny", {}, 16),
])
def test_tc_decode_step_fused(name, kw, partition):
    case = Case(workloads.make_plan(name, **kw))
    hk, hv = case.snapshot(0)
    out = case.gpu_step_fused(0, partition)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    assert_close(out, ref, f"tc fused step {name}")
    assert np.array_equal(bits(case.vals.k_pools[0]), hk)


def test_tc_matches_cuda_core_kernel():
    """Both kernels on the same inputs match the oracle, and each other,
    within the output tolerance."""
    case = Case(workloads.make_plan("long", num_seqs=4, len_range=(2000, 9000)))
    hk, hv = case.snapshot(0)
    case.gpu_writes(0)
    ref = case.oracle_step(0, hk, hv)
    a = case.gpu_decode(0)
    api.set_decode_impl("cuda_cores")
    try:
        b = case.gpu_decode(0)
    finally:
        api.set_decode_impl("tensor_cores")
    assert_close(a, ref, "tensor cores vs oracle")
    assert_close(b, ref, "CUDA cores vs oracle")
    assert_close(a, b.double().cpu().numpy(), "tensor vs CUDA cores")
