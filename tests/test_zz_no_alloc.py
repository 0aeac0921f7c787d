"""pa_decode_static_scratch: decode for callers that cannot allocate.

Some users of the library cannot give it a workspace: a serving engine that
has already handed nearly all device memory to its KV-cache pool, a decode
loop that must never call cudaMalloc (it can synchronise the device or fail
under memory pressure), or a host that reaches the library only through the
C ABI.  For them the split-KV partials live in one fixed device array inside
the library.  These tests call that entry point through the C ABI and check
every output against the fp64 oracle at the tolerance the other decode tests
use, |gpu - ref| <= 2e-3 + 1e-2 |ref|, and against pa_decode with a caller
workspace, on two calls in a row (the array keeps whatever the previous call
left in it).  The Python wrapper is checked the same way with automatic
partitions (a split chosen by the library) and single pass.

This file is named so that pytest collects it last.
"""
import ctypes
import re
from pathlib import Path

import pytest
import torch

from paged_kv_cache_64_gb300 import _lib, api, workloads

from _parity import Case, assert_close


def static_call(case, out, partition, max_seq_len=None):
    spec = case.spec
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    return _lib.load().pa_decode_static_scratch(
        vp(out), vp(case.vals.q), vp(case.vals.k_pools[0]), vp(case.vals.v_pools[0]),
        case.plan.num_blocks, vp(case.tables), case.tables.shape[1], vp(case.lens),
        case.max_seq_len if max_seq_len is None else max_seq_len, spec.num_seqs,
        spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size,
        float(case.plan.scale), int(partition),
        _lib.PA_BF16 if spec.dtype == "bf16" else _lib.PA_F16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def oracle_output(case):
    """Write the step's tokens on the GPU and return the oracle's output on
    the pools as they were before (the oracle applies the same writes)."""
    hk, hv = case.snapshot(0)
    case.gpu_writes(0)
    return case.oracle_step(0, hk, hv)


def test_static_scratch_size_matches_header():
    """The binding's constant is the header's PA_STATIC_SCRATCH_BYTES."""
    text = (Path(__file__).resolve().parents[1] / "include" / "pa.h").read_text()
    m = re.search(r"#define\s+PA_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "PA_STATIC_SCRATCH_BYTES not found in pa.h"
    assert _lib.STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw,partition", [
    ("tiny", {}, 16),
    ("llama", {"num_seqs": 8, "len_range": (600, 3000)}, 256),
    ("qwen", {"num_seqs": 32}, 64),
    ("long", {"num_seqs": 2, "len_range": (3000, 6000)}, 512),
])
def test_static_scratch_matches_oracle_and_workspace_decode(name, kw, partition):
    assert torch.cuda.is_available()
    case = Case(workloads.make_plan(name, **kw))
    ref = oracle_output(case)
    spec = case.spec
    need = api.workspace_size(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads,
                              spec.head_dim, spec.block_size, case.max_seq_len, partition,
                              case.dtype)
    assert 0 < need <= _lib.STATIC_SCRATCH_BYTES  # the split-KV path is the one exercised
    with_workspace = case.gpu_decode(0, partition=partition)  # pa_decode, caller workspace
    assert_close(with_workspace, ref, f"workspace decode {name}")
    for _ in range(2):  # two calls in a row on the same fixed array
        out = torch.full_like(case.vals.q, float("nan"))
        assert static_call(case, out, partition) == 0
        api.check_error()
        assert_close(out, ref, f"static scratch {name} vs oracle")
        assert_close(out, with_workspace.double().cpu().numpy(), f"static scratch {name} vs pa_decode")


@pytest.mark.gpu
@pytest.mark.parametrize("partition", [0, -1])
def test_static_scratch_python_wrapper(partition):
    """api.decode_static_scratch with automatic partitions (the library picks
    a split for this batch) and single pass (no scratch used)."""
    case = Case(workloads.make_plan("qwen", num_seqs=16))
    spec = case.spec
    if partition == 0:
        auto = api.auto_partition(spec.num_seqs, spec.num_kv_heads, case.max_seq_len,
                                  spec.head_dim, spec.block_size,
                                  spec.num_q_heads // spec.num_kv_heads, case.dtype)
        assert auto > 0, "the automatic choice should split this batch"
    ref = oracle_output(case)
    for _ in range(2):
        out = torch.full_like(case.vals.q, float("nan"))
        api.decode_static_scratch(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0],
                                  case.tables, case.lens, case.max_seq_len, case.plan.scale,
                                  partition_tokens=partition)
        api.check_error()
        assert_close(out, ref, f"static scratch wrapper P={partition}")


@pytest.mark.gpu
def test_static_scratch_rejects_oversized_requests():
    """Partials larger than the fixed array are refused before any launch."""
    case = Case(workloads.make_plan("tiny"))
    out = torch.full_like(case.vals.q, float("nan"))
    rc = static_call(case, out, 16, max_seq_len=1 << 20)  # 65,536 partitions of 16
    assert rc == 8  # PA_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert torch.isnan(out).all()  # nothing ran
    api.check_error()
