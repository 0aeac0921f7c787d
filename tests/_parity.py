"""Helpers for the GPU parity tests: run one decode step of a workload through
the C ABI and through the CPU oracle, on the same seeded inputs.

The GPU side uses the library's allocator layout; the oracle side uses the
allocator model's layout (the two are asserted identical).  Oracle inputs are
copies of the pools taken BEFORE the GPU kernels write them; the oracle then
applies its own block copies and cache writes.
"""
import numpy as np
import torch

import oracle
from oracle.allocator import BlockAllocatorModel
from oracle.prefix_cache import PrefixCachePoolModel
from paged_kv_cache_64_gb300 import api, workloads

# Tolerance for fp16/bf16 outputs: |gpu - ref| <= TOL_ABS + TOL_REL * |ref|.
TOL_ABS, TOL_REL = 2e-3, 1e-2


def bits(t):
    """16-bit tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu, ref, what="", mask_rows=None):
    g = gpu.detach().double().cpu().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    if mask_rows is not None:
        g, ref = g[mask_rows], ref[mask_rows]
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.isfinite(ref).all(), f"{what}: oracle produced non-finite values"
    err = np.abs(g - ref)
    bad = ~(err <= TOL_ABS + TOL_REL * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; max abs err "
            f"{float(np.nanmax(err)):.3g}; first {idx}: gpu {g[bad][:5]} ref {ref[bad][:5]}")
    return float(err.max()) if err.size else 0.0


class Case:
    """One workload instance on the GPU plus the matching oracle inputs."""

    def __init__(self, plan, device="cuda", layers=1):
        self.plan = plan
        self.spec = spec = plan.spec
        self.lay = workloads.layout(plan, workloads.native_allocator(plan))
        self.ref_lay = workloads.layout(plan, PrefixCachePoolModel if plan.apc
                                        else BlockAllocatorModel)
        for f in ("block_tables", "seq_lens", "slot_mapping", "pre_copies", "pre_slots",
                  "step_copies"):
            assert np.array_equal(getattr(self.lay, f), getattr(self.ref_lay, f)), f
        self.vals = workloads.make_values(plan, self.lay, device, layers)
        dev = torch.device(device)
        self.tables = torch.as_tensor(self.lay.block_tables, device=dev)
        self.lens = torch.as_tensor(self.lay.seq_lens, device=dev)
        self.slots = torch.as_tensor(self.lay.slot_mapping, device=dev)
        self.pre_copies = torch.as_tensor(self.lay.pre_copies, device=dev)
        self.pre_slots = torch.as_tensor(self.lay.pre_slots, device=dev)
        self.max_seq_len = int(self.lay.max_seq_len)
        self.dtype = workloads.torch_dtype(spec.dtype)

    # ---------------------------------------------------------------- oracle
    def blocks_of(self, seqs):
        t = self.ref_lay.block_tables
        n = -(-self.ref_lay.seq_lens.astype(np.int64) // self.spec.block_size)
        used = set()
        for s in seqs:
            used.update(t[s, :n[s]].tolist())
        return sorted(used)

    def snapshot(self, layer, blocks=None):
        """Host copies of the layer's K/V pools (only `blocks` filled when
        given; the rest stays zero and is never read)."""
        out = []
        for pool in (self.vals.k_pools[layer], self.vals.v_pools[layer]):
            if blocks is None:
                out.append(bits(pool))
            else:
                host = np.zeros(tuple(pool.shape), dtype=np.uint16)
                idx = torch.as_tensor(blocks, dtype=torch.long, device=pool.device)
                host[np.asarray(blocks)] = bits(pool.index_select(0, idx))
                out.append(host)
        return out

    def oracle_step(self, layer, host_k, host_v, seqs=None):
        lay = self.ref_lay
        oracle.copy_blocks([host_k, host_v], lay.pre_copies)
        if lay.pre_slots.size:
            oracle.cache_write(host_k, host_v, bits(self.vals.k_pre[layer]),
                               bits(self.vals.v_pre[layer]), lay.pre_slots)
        oracle.cache_write(host_k, host_v, bits(self.vals.k_new[layer]),
                           bits(self.vals.v_new[layer]), lay.slot_mapping)
        return oracle.decode(bits(self.vals.q), host_k, host_v, lay.block_tables, lay.seq_lens,
                             self.plan.scale, self.spec.dtype, seqs=seqs)

    # ------------------------------------------------------------------- GPU
    def gpu_writes(self, layer):
        kp, vp = self.vals.k_pools[layer], self.vals.v_pools[layer]
        if self.pre_copies.numel():
            api.copy_blocks([kp], [vp], self.pre_copies)
        if self.pre_slots.numel():
            api.cache_write(self.vals.k_pre[layer], self.vals.v_pre[layer], self.pre_slots, kp, vp)
        api.cache_write(self.vals.k_new[layer], self.vals.v_new[layer], self.slots, kp, vp)

    def gpu_pre_writes(self, layer):
        kp, vp = self.vals.k_pools[layer], self.vals.v_pools[layer]
        if self.pre_copies.numel():
            api.copy_blocks([kp], [vp], self.pre_copies)
        if self.pre_slots.numel():
            api.cache_write(self.vals.k_pre[layer], self.vals.v_pre[layer], self.pre_slots, kp, vp)

    def gpu_step_fused(self, layer, partition=None, workspace=None):
        """Copies and earlier writes, then the fused write + decode launch."""
        P = self.spec.partition_tokens if partition is None else partition
        self.gpu_pre_writes(layer)
        out = torch.empty_like(self.vals.q)
        api.decode_step(out, self.vals.q, self.vals.k_new[layer], self.vals.v_new[layer],
                        self.slots, self.vals.k_pools[layer], self.vals.v_pools[layer],
                        self.tables, self.lens, self.max_seq_len, self.plan.scale,
                        partition_tokens=P, workspace=workspace)
        return out

    def gpu_decode(self, layer, partition=None, workspace=None):
        P = self.spec.partition_tokens if partition is None else partition
        out = torch.empty_like(self.vals.q)
        api.decode(out, self.vals.q, self.vals.k_pools[layer], self.vals.v_pools[layer],
                   self.tables, self.lens, self.max_seq_len, self.plan.scale,
                   partition_tokens=P, workspace=workspace)
        return out
