"""The Python API has no CPU path: every device entry point refuses host
tensors before anything is launched or computed, and a missing library build
is an error, not a fallback.  Runs without a GPU.
"""
import pytest
import torch

from paged_kv_cache_64_gb300 import _lib, api

S, HQ, HKV, D, B, NB = 2, 4, 2, 64, 16, 8


def host_case(dtype=torch.float16):
    g = torch.Generator().manual_seed(3)
    q = torch.randn(S, HQ, D, generator=g).to(dtype)
    pools = [torch.randn(NB, HKV, B, D, generator=g).to(dtype) for _ in range(2)]
    tables = torch.arange(S * 2, dtype=torch.int32).reshape(S, 2)
    lens = torch.tensor([5, 20], dtype=torch.int32)
    k_new = torch.randn(S, HKV, D, generator=g).to(dtype)
    v_new = torch.randn(S, HKV, D, generator=g).to(dtype)
    slots = torch.tensor([4, 2 * B + 19], dtype=torch.int64)
    return q, pools, tables, lens, k_new, v_new, slots


def entry_points():
    q, (kp, vp), tables, lens, k_new, v_new, slots = host_case()
    codes = [torch.zeros(NB, HKV, B, D, dtype=torch.uint8) for _ in range(2)]
    out = torch.full_like(q, float("nan"))
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64)
    return out, {
        "cache_write": lambda: api.cache_write(k_new, v_new, slots, kp, vp),
        "copy_blocks": lambda: api.copy_blocks([kp], [vp], pairs),
        "decode": lambda: api.decode(out, q, kp, vp, tables, lens, 20, 0.125,
                                     partition_tokens=-1),
        "decode split": lambda: api.decode(out, q, kp, vp, tables, lens, 20, 0.125,
                                           partition_tokens=16, workspace=ws),
        "decode_step": lambda: api.decode_step(out, q, k_new, v_new, slots, kp, vp, tables,
                                               lens, 20, 0.125, partition_tokens=-1),
        "decode_cascade": lambda: api.decode_cascade(out, q, kp, vp, tables, lens, 20, 0.125,
                                                     0, workspace=ws),
        "cache_write_fp8": lambda: api.cache_write_fp8(k_new, v_new, slots, codes[0], codes[1],
                                                       1.0, 1.0),
        "decode_fp8": lambda: api.decode_fp8(out, q, codes[0], codes[1], tables, lens, 20,
                                             0.125, 1.0, 1.0, partition_tokens=-1),
        "decode_static_scratch": lambda: api.decode_static_scratch(out, q, kp, vp, tables, lens,
                                                                   20, 0.125,
                                                                   partition_tokens=-1),
        "decode_partitions": lambda: api.decode_partitions(q, kp, vp, tables, lens, 20, 0.125,
                                                           16, workspace=ws),
        "split_kv_reduce": lambda: api.split_kv_reduce(out, ws, lens, 20, 16),
    }


@pytest.mark.parametrize("name", sorted(entry_points()[1]))
def test_device_entry_points_refuse_host_tensors(name):
    out, calls = entry_points()
    with pytest.raises((ValueError, TypeError)) as e:
        calls[name]()
    assert "CUDA" in str(e.value) or "cuda" in str(e.value), str(e.value)
    assert torch.isnan(out).all()  # nothing was written on the host either


def test_missing_build_is_an_error(monkeypatch, tmp_path):
    """With the shared library absent the first call raises LibraryMissing;
    nothing is computed some other way."""
    monkeypatch.setattr(_lib._build, "LIB", str(tmp_path / "libpa.so"))
    monkeypatch.setattr(_lib, "_lib", None)  # the loaded handle, if any
    with pytest.raises(_lib.LibraryMissing):
        _lib.load()
