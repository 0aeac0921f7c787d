"""GPU parity over the head shapes and batch sizes the library accepts.

Every group size G = H_q / H_kv from 1 to 8 (the CUDA-core kernel pads a
group to 1, 2, 4 or 8 heads, the E4M3 kernel to 4 or 8, the tensor-core
kernels pad the MMA N), with each head dim, block size and 16-bit type
appearing, through the tensor-core, CUDA-core and E4M3 kernels, single pass
and split-KV (combined inside the launch up to 8 partitions, by the separate
combine kernel beyond); and the largest batch one launch takes, 65,535
sequences.  Every output is compared with the fp64 oracle:
|gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""
import pytest
import torch

from paged_kv_cache_64_gb300 import _lib, api, workloads

from _parity import Case, assert_close
from test_gpu_fp8 import Fp8Case, np_codes

pytestmark = pytest.mark.gpu

# (q heads, KV heads, head_dim, block_size, dtype)
SHAPES = {
    "g1_d128_b16": (8, 8, 128, 16, "bf16"),
    "g2_d64_b16": (16, 8, 64, 16, "f16"),
    "g3_d64_b32": (6, 2, 64, 32, "f16"),
    "g4_one_kv_head_d128_b32": (4, 1, 128, 32, "f16"),
    "g5_d128_b32": (10, 2, 128, 32, "bf16"),
    "g6_d64_b16": (12, 2, 64, 16, "bf16"),
    "g7_d128_b16": (28, 4, 128, 16, "f16"),
    "g8_d64_b32": (16, 2, 64, 32, "bf16"),
}
# cached lengths 0..1,500 over 7 sequences: empty ones (one token after the
# step), ragged last blocks, up to 12 partitions of 128 positions
LENS = (0, 1500)


def plan_of(name, seed=0):
    hq, hkv, d, B, dt = SHAPES[name]
    return workloads.make_shape_plan(7, hq, hkv, d, B, dt, LENS, seed=17 + len(name) + seed)


@pytest.fixture
def impl():
    prev = api.get_decode_impl()
    yield api.set_decode_impl
    api.set_decode_impl(prev)
    api.check_error()


def step_parity(case, partition, fused):
    hk, hv = case.snapshot(0)
    if fused:
        out = case.gpu_step_fused(0, partition)
    else:
        case.gpu_writes(0)
        out = case.gpu_decode(0, partition)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    return out, ref


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("kernel,partition,fused", [
    ("tensor_cores", -1, False),
    ("tensor_cores", 256, True),    # fused write + combine inside the launch
    ("tensor_cores", 128, False),   # > 8 partitions: the combine kernel
    ("tensor_cores", 0, True),
    ("cuda_cores", -1, True),
    ("cuda_cores", 256, False),
])
def test_shape_every_output(impl, name, kernel, partition, fused):
    impl(kernel)
    case = Case(plan_of(name))
    out, ref = step_parity(case, partition, fused)
    assert_close(out, ref, f"{name} {kernel} P={partition} fused={fused}")


@pytest.mark.parametrize("name", sorted(SHAPES))
@pytest.mark.parametrize("partition,fused", [(-1, True), (256, False), (0, True)])
def test_shape_fp8_every_output(name, partition, fused):
    c = Fp8Case("shape", seed=len(name), plan=plan_of(name, seed=1))
    kc, vc = np_codes(c.kp), np_codes(c.vp)
    out = c.gpu(partition, step=fused)
    api.check_error()
    assert_close(out, c.oracle(kc, vc, step=fused), f"fp8 {name} P={partition}")


@pytest.mark.parametrize("partition", [-1, 16])
def test_largest_batch(impl, partition):
    """65,535 sequences of 1 to 25 tokens after the step (the grid's limit on
    sequences), every output checked; 16-position partitions split the
    longer ones in two."""
    impl("auto")
    case = Case(workloads.make_shape_plan(65535, 4, 1, 64, 16, "f16", (0, 24), seed=29))
    out, ref = step_parity(case, partition, fused=True)
    assert_close(out, ref, f"65,535 sequences P={partition}")


def test_batch_past_the_limit_is_rejected_before_launch():
    S, hq, hkv, d, B = 65536, 4, 1, 64, 16
    q = torch.zeros((S, hq, d), dtype=torch.float16, device="cuda")
    pool = torch.zeros((4, hkv, B, d), dtype=torch.float16, device="cuda")
    tables = torch.zeros((S, 1), dtype=torch.int32, device="cuda")
    lens = torch.ones(S, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    with pytest.raises(_lib.PagedAttentionError):
        api.decode(out, q, pool, pool, tables, lens, 1, 0.125, partition_tokens=-1)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "a rejected call must not launch"
    api.check_error()
