"""Benchmark of the paged decode step on GB300.

One step = the whole hot path over one batch: (copy-on-write block copies,)
the cache write of every sequence's new token, and paged decode attention
(split-KV partition kernel + reduce) -- for every layer of the workload.

Default workload: the Llama-3-8B-shaped decode batch (256 sequences, lengths
U[512, 8192], 32 q / 8 KV heads, d 128, bf16, B 16), whose K/V (~4.6 GB per
step) is far larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Prints one JSON line (rank 0).  Multi-GPU: one process per GPU under
torch.distributed.run; every rank decodes its own batch (weak scaling, no
collective on the data path); value = bytes of all ranks / max time.
"""
import argparse
import dataclasses
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention achieved HBM GB/s (% of GB300 peak); decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def reduce_over_ranks(seconds, units, device=None):
    """(max seconds, summed units) over all ranks; identity when not
    distributed.  Works with gloo (CPU tensors) and nccl (CUDA tensors)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return seconds, units
    dev = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest():
    """Hash of the decode kernel source, to tell whether a stored ncu traffic
    figure still describes the kernel being timed."""
    h = hashlib.sha256()
    for f in ("pa_decode.cu", "pa_decode_tc.cu", "pa_decode_tc.cuh", "pa_decode_tc_fp8.cu",
              "pa_decode_tc_fp8_g4.cu", "pa_decode.cuh", "pa_common.cuh", "pa_fp8.cuh",
              "pa_tcgen05.cuh", "pa_cascade.cu"):
        with open(os.path.join(ROOT, "paged_kv_cache_64_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary of this
    workload, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"pa_decode_{workload}.md")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        text = fh.read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_digest():
        return None
    return float(m.group(1))


# ----------------------------------------------------------------- oracle arm
def _bits16(x, dtype):
    """float32 array -> uint16 bit patterns of f16 or bf16 (round to nearest
    even), the host inputs' storage format."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    b = x.view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def oracle_inputs(plan, seed=0):
    """Host inputs of the oracle arm: the plan's layout (the allocator
    model's), q drawn N(0, 1), and K/V pools filled in every block a sequence
    uses with N(0, 1) draws, taken as seeded slices of one seeded table of
    2^24 draws (the oracle's time does not depend on the values; drawing
    every element afresh would take the host longer than the oracle does).
    Returns (layout, q, k, v)."""
    from oracle.allocator import BlockAllocatorModel
    from oracle.prefix_cache import PrefixCachePoolModel
    from paged_kv_cache_64_gb300 import workloads

    spec = plan.spec
    lay = workloads.layout(plan, PrefixCachePoolModel if plan.apc else BlockAllocatorModel)
    rng = np.random.default_rng(spec.seed * 7919 + seed)
    B = spec.block_size
    shape = (plan.num_blocks, spec.num_kv_heads, B, spec.head_dim)
    per_block = spec.num_kv_heads * B * spec.head_dim
    k = np.zeros(shape, dtype=np.uint16)  # pages are only touched where filled
    v = np.zeros(shape, dtype=np.uint16)
    q = _bits16(rng.standard_normal((spec.num_seqs, spec.num_q_heads, spec.head_dim),
                                    dtype=np.float32), spec.dtype)
    T = 1 << 24
    table = _bits16(rng.standard_normal(T, dtype=np.float32), spec.dtype)
    chunk = (T // 2) // per_block  # blocks per slice
    for s in range(spec.num_seqs):
        ids = lay.block_tables[s, :-(-int(lay.seq_lens[s]) // B)]
        for pool in (k, v):
            for c in range(0, len(ids), chunk):
                part = ids[c:c + chunk]
                n = len(part) * per_block
                off = int(rng.integers(0, T - n))
                pool[part] = table[off:off + n].reshape((len(part),) + shape[1:])
    return lay, q, k, v


def oracle_sample(plan, inputs, budget_s, first=0):
    """Time the fp64 oracle on as many of the workload's sequences as fit in
    about budget_s seconds of host time, starting at sequence `first` and
    going round the batch.  Returns (seconds, algorithmic bytes, tokens,
    number of sequences, threads)."""
    import oracle
    from paged_kv_cache_64_gb300 import workloads

    spec = plan.spec
    lay, q, k, v = inputs
    S = spec.num_seqs
    order = [(first + i) % S for i in range(S)]
    done, seconds, nbytes, tokens = 0, 0.0, 0, 0
    batch = 1
    while order and seconds < budget_s:
        take, order = order[:batch], order[batch:]
        if not order and seconds < 0.6 * budget_s:
            order = list(range(S))  # go round the batch again
        t0 = time.perf_counter()
        oracle.decode(q, k, v, lay.block_tables, lay.seq_lens, plan.scale, spec.dtype, seqs=take)
        dt_s = time.perf_counter() - t0
        seconds += dt_s
        done += len(take)
        nbytes += workloads.algorithmic_bytes(spec, lay.seq_lens[take])
        tokens += len(take)
        per_seq = dt_s / len(take)
        batch = max(1, min(len(order), int((budget_s - seconds) / max(per_seq, 1e-6) / 2) or 1))
    return seconds, nbytes, tokens, done, oracle.num_threads()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def single_thread_gbs(plan, inputs, budget_s):
    """The oracle on one host thread: GB/s equivalent on a sample of about
    budget_s seconds (the thread count is restored afterwards)."""
    import oracle
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        secs, nbytes, _, _, _ = oracle_sample(plan, inputs, budget_s)
    finally:
        oracle.set_num_threads(n)
    return nbytes / secs / 1e9


def sample_text(nseq, total):
    if nseq <= total:
        return f"{nseq} of {total} sequences"
    return f"all {total} sequences, {nseq / total:.1f} passes"



def run_reference(args, rank, world):
    from paged_kv_cache_64_gb300 import workloads
    if rank != 0:
        return
    plan = workloads.make_plan(args.workload, num_seqs=args.num_seqs)
    inputs = oracle_inputs(plan)
    per_step = []
    info = None
    # each step a bounded sample: the whole run's oracle time stays near
    # --ref-total-seconds whatever --steps and --warmup are
    budget = min(args.ref_step_seconds,
                 max(0.25, args.ref_total_seconds / (args.warmup + args.steps)))
    first = 0
    for i in range(args.warmup + args.steps):
        secs, nbytes, toks, nseq, threads = oracle_sample(plan, inputs, budget, first)
        first = (first + nseq) % plan.spec.num_seqs
        if i >= args.warmup:
            per_step.append((secs, nbytes, toks, nseq))
        info = threads
    secs = sum(s for s, _, _, _ in per_step)
    nbytes = sum(b for _, b, _, _ in per_step)
    toks = sum(t for _, _, t, _ in per_step)
    gbs = nbytes / secs / 1e9
    layers = plan.spec.num_layers
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / len(per_step), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": plan.spec.dtype, "data": "synthetic",
        "config": {"workload": plan.spec.name + ": " + plan.spec.describe,
                   "layers_in_step": layers,
                   "sample": "each step decodes as many of the batch's sequences as fit in "
                             f"~{budget:.2g} s (all heads of each), the next step going on "
                             "from there"},
        "tokens_per_s": toks / secs / layers,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": info, "kind": "oracle",
                         "sample": sample_text(per_step[0][3], plan.spec.num_seqs) + " per step",
                         "cpu_model": cpu_model()},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def host_pool_timing(plan, reps=5):
    """Host time of the prefix-caching pool on the plan's requests, through
    the Python binding: every request's add (prefix lookup, touch, new
    blocks, hashing), one decode-step append per request, then the frees.
    Median of `reps` fresh pools, microseconds per call."""
    from paged_kv_cache_64_gb300 import api
    S = plan.spec.num_seqs
    add, app, free = [], [], []
    for _ in range(reps):
        pool = api.PrefixCachePool(plan.num_blocks, plan.spec.block_size, plan.free_order)
        t0 = time.perf_counter()
        for op in plan.ops:
            pool.add_request(op[1], op[2])
        t1 = time.perf_counter()
        for s in range(S):
            pool.append(s, int(plan.step_tokens[s]))
        t2 = time.perf_counter()
        for s in range(S):
            pool.release(s)
        t3 = time.perf_counter()
        add.append((t1 - t0) / len(plan.ops))
        app.append((t2 - t1) / S)
        free.append((t3 - t2) / S)
    return {"add_request_us": 1e6 * statistics.median(add),
            "append_us": 1e6 * statistics.median(app),
            "free_us": 1e6 * statistics.median(free),
            "prompt_tokens": int(len(plan.ops[0][2])), "requests": len(plan.ops),
            "via": "Python binding (ctypes) on the host cores"}


# -------------------------------------------------------------------- GPU arm
class GpuStep:
    """Device state of one workload and the calls of one decode step."""

    FP8_SCALE = 1.0 / 64  # E4M3 pools of N(0, 1) values: +-448 codes cover +-7 sigma

    def __init__(self, plan, device, partition_tokens=None, cascade=False, kv="16bit"):
        import torch
        from paged_kv_cache_64_gb300 import api, workloads

        self.api, self.torch = api, torch
        self.plan, self.spec = plan, plan.spec
        self.device = device
        self.lay = workloads.layout(plan, workloads.native_allocator(plan))
        self.vals = workloads.make_values(plan, self.lay, device)
        self.fp8 = kv == "fp8"
        if self.fp8:
            # the same N(0, 1) values, quantised into E4M3 pools (setup, untimed)
            self.vals.k_pools = [self._quantize(p) for p in self.vals.k_pools]
            self.vals.v_pools = [self._quantize(p) for p in self.vals.v_pools]
            torch.cuda.empty_cache()
        t = lambda a: torch.as_tensor(a, device=device)
        self.tables, self.lens = t(self.lay.block_tables), t(self.lay.seq_lens)
        self.slots, self.copies = t(self.lay.slot_mapping), t(self.lay.pre_copies)
        self.max_seq_len = int(self.lay.max_seq_len)
        spec = self.spec
        self.P = spec.partition_tokens if partition_tokens is None else partition_tokens
        self.resolved_P = self.P if self.P else api.auto_partition(
            spec.num_seqs, spec.num_kv_heads, self.max_seq_len, spec.head_dim, spec.block_size,
            spec.num_q_heads // spec.num_kv_heads, self.vals.q.dtype, fp8=self.fp8)
        wsize = api.fp8_workspace_size if self.fp8 else api.workspace_size
        size = wsize(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                     spec.block_size, self.max_seq_len, self.P, self.vals.q.dtype)
        # shared-prefix (cascade) path: the prefix every sequence reaches
        # through the same block-table entries, attended once per KV head
        self.prefix_len = (api.shared_prefix_len(self.lay.block_tables, self.lay.seq_lens,
                                                 spec.block_size) if cascade else 0)
        if self.prefix_len:
            size = api.cascade_workspace_size(spec.num_seqs, spec.num_q_heads,
                                              spec.num_kv_heads, spec.head_dim, spec.block_size,
                                              self.max_seq_len, self.prefix_len,
                                              self.vals.q.dtype)
        self.ws = api.alloc_workspace(size, device) if size else None
        self.out = [torch.empty_like(self.vals.q) for _ in range(spec.num_layers)]
        kvb = 1 if self.fp8 else None
        self.logical_bytes = workloads.algorithmic_bytes(spec, self.lay.seq_lens, kvb)
        self.decode_bytes = (workloads.cascade_bytes(spec, self.lay.seq_lens, self.prefix_len)
                             if self.prefix_len else self.logical_bytes)
        self.write_bytes = workloads.cache_write_bytes(spec, spec.num_seqs, kvb)
        self.copy_bytes = 2 * 2 * len(self.lay.pre_copies) * spec.num_kv_heads * \
            spec.block_size * spec.head_dim * (kvb or workloads.DTYPE_BYTES[spec.dtype])
        # positions a partial covers (the partition times the partitions a
        # CTA merges), hence the partials per row and the launches
        self.partial_tokens = api.partial_tokens(
            spec.num_seqs, spec.num_kv_heads, self.max_seq_len, spec.head_dim, spec.block_size,
            spec.num_q_heads // spec.num_kv_heads, self.vals.q.dtype, self.P, fp8=self.fp8)
        NP = -(-self.max_seq_len // self.partial_tokens) if self.partial_tokens > 0 else 1
        # fused write + decode (+ combine) launch, a separate combine above 8
        # partitions, and the copy-on-write copies when there are any
        per_layer = 1 + (1 if NP > 8 else 0) + (1 if len(self.lay.pre_copies) else 0)
        if self.prefix_len:  # prefix pass + tail pass (write, decode and merge)
            per_layer = 2 + (1 if len(self.lay.pre_copies) else 0)
        self.launches_per_step = per_layer * spec.num_layers

    def _quantize(self, pool16):
        """E4M3 copy of a 16-bit pool, by the library's quantising cache
        write over every slot, in chunks."""
        torch, api = self.torch, self.api
        nb, hkv, B, d = pool16.shape
        out = torch.empty((nb, hkv, B, d), dtype=torch.uint8, device=pool16.device)
        step = 4096
        for b0 in range(0, nb, step):
            b1 = min(nb, b0 + step)
            tok = pool16[b0:b1].permute(0, 2, 1, 3).reshape(-1, hkv, d).contiguous()
            slots = torch.arange(b0 * B, b1 * B, dtype=torch.int64, device=pool16.device)
            api.cache_write_fp8(tok, tok, slots, out, out, self.FP8_SCALE, self.FP8_SCALE)
        return out

    def step_bytes(self):
        return self.spec.num_layers * (self.decode_bytes + self.write_bytes + self.copy_bytes)

    def run(self, ev=None, q=None, k_new=None, v_new=None, stream=None, tables=None, lens=None,
            slots=None, out=None, cev=None):
        """One step.  ev / cev: optional lists collecting (start, end) events
        around each decode call / each block-copy call.  q .. out: other
        input and output tensors of the same shapes (the end-to-end run's
        second buffer set)."""
        api, v = self.api, self.vals
        q = v.q if q is None else q
        tables = self.tables if tables is None else tables
        lens = self.lens if lens is None else lens
        slots = self.slots if slots is None else slots
        outs = self.out if out is None else out
        for layer in range(self.spec.num_layers):
            kp, vp = v.k_pools[layer], v.v_pools[layer]
            if self.copies.numel():
                if cev is not None:
                    c0 = self.torch.cuda.Event(enable_timing=True)
                    c1 = self.torch.cuda.Event(enable_timing=True)
                    c0.record(stream)
                api.copy_blocks([kp], [vp], self.copies, stream=stream)
                if cev is not None:
                    c1.record(stream)
                    cev.append((c0, c1))
            if ev is not None:
                a = self.torch.cuda.Event(enable_timing=True)
                b = self.torch.cuda.Event(enable_timing=True)
                a.record(stream)
            if self.fp8:
                # E4M3 pools: quantised write of the new token and the decode, one launch
                api.decode_fp8(outs[layer], q, kp, vp, tables, lens,
                               self.max_seq_len, self.plan.scale, self.FP8_SCALE, self.FP8_SCALE,
                               partition_tokens=self.P,
                               k_new=v.k_new[layer] if k_new is None else k_new[layer],
                               v_new=v.v_new[layer] if v_new is None else v_new[layer],
                               slot_mapping=slots, workspace=self.ws, stream=stream)
            elif self.prefix_len:
                # prefix pass, then the tails with the new token's write and the merge
                api.decode_cascade(outs[layer], q, kp, vp, tables, lens,
                                   self.max_seq_len, self.plan.scale, self.prefix_len,
                                   k_new=v.k_new[layer] if k_new is None else k_new[layer],
                                   v_new=v.v_new[layer] if v_new is None else v_new[layer],
                                   slot_mapping=slots, workspace=self.ws, stream=stream)
            else:
                # the new token's cache write and the decode, one launch
                api.decode_step(outs[layer], q,
                                v.k_new[layer] if k_new is None else k_new[layer],
                                v.v_new[layer] if v_new is None else v_new[layer], slots,
                                kp, vp, tables, lens, self.max_seq_len,
                                self.plan.scale, partition_tokens=self.P, workspace=self.ws,
                                stream=stream)
            if ev is not None:
                b.record(stream)
                ev.append((a, b))


def run_gpu(args, rank, world, local_rank):
    import torch
    from paged_kv_cache_64_gb300 import api, workloads

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    api.set_decode_impl(args.decode_impl)
    base = workloads.SPECS[args.workload]
    plan = workloads.make_plan(args.workload, num_seqs=args.num_seqs,
                               len_range=tuple(args.len_range) if args.len_range else None,
                               seed=base.seed + 1000 * rank if rank else None, apc=args.apc,
                               cow=args.cow)
    if args.layers:
        plan.spec = dataclasses.replace(plan.spec, num_layers=int(args.layers))
    st = GpuStep(plan, device, args.partition_tokens, cascade=args.cascade, kv=args.kv)
    stream = torch.cuda.current_stream()
    spec = st.spec
    flush = None
    if st.step_bytes() < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)

    for _ in range(args.warmup):
        st.run()
    api.check_error()
    use_graph = args.graph == "on" or (args.graph == "auto" and spec.num_layers > 1)
    graph = None
    if use_graph:
        # The step's library calls, captured once and replayed (launch-bound
        # multi-layer steps); the captured kernels are the same launches.
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            st.run()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            st.run()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        api.check_error()

    def one_step(ev=None, cev=None):
        if graph is not None:
            graph.replay()
        else:
            st.run(ev, cev=cev)

    # The timed region runs the K steps `repeats` times, enough for at least
    # --min-timed-seconds (so the clock sampler sees the GPU under load for a
    # while); the count comes from one untimed pass of K steps, the largest
    # over the ranks so that every rank times the same steps.
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(args.steps):
        if flush is not None:
            flush.fill_(1)
        one_step()
    c1.record()
    torch.cuda.synchronize()
    repeats = max(1, int(np.ceil(args.min_timed_seconds * 1e3 / max(c0.elapsed_time(c1), 1e-3))))
    repeats = int(reduce_over_ranks(float(repeats), 0.0, device)[0])
    n_timed = repeats * args.steps

    # ------------------------------------------------ timed region (device)
    ev = []
    cev = []  # block-copy launches (copy-on-write workloads)
    step_ev = []
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        if flush is None and graph is None:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            for _ in range(n_timed):
                one_step(ev, cev)
            t1.record()
            torch.cuda.synchronize()
            total_ms = t0.elapsed_time(t1)
        else:
            for _ in range(n_timed):
                if flush is not None:
                    flush.fill_(1)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                one_step(ev, cev)
                b.record()
                step_ev.append((a, b))
            torch.cuda.synchronize()
            total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    barrier()
    api.check_error()
    secs, all_bytes = reduce_over_ranks(total_ms / 1e3, st.step_bytes() * n_timed, device)
    value = all_bytes / secs / 1e9
    if ev:
        dec_avg_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        kernel_note = ("pa_decode_step launch (new-token cache write + split-KV decode + combine), "
                       "CUDA events")
        if st.fp8:
            kernel_note = ("pa_decode_fp8 launch (quantised new-token write + decode over E4M3 "
                           "pools + combine), CUDA events")
        if st.prefix_len:
            kernel_note = ("pa_decode_cascade call (tensor-core prefix pass + tail pass with the "
                           "new-token write and the merge), CUDA events")
    else:
        # graph replay: a step's time spread over its layers (cache write included)
        dec_avg_ms = statistics.mean(a.elapsed_time(b) for a, b in step_ev) / spec.num_layers
        kernel_note = ("pa_decode_step per layer: graph-replayed step time / layers "
                       "(CUDA events around each replay)")
    peak, peak_kind = measured_peaks()
    launch_bytes = st.decode_bytes + st.write_bytes  # what one decode_step launch must move
    achieved = launch_bytes / (dec_avg_ms / 1e3) / 1e9
    traffic = stored_traffic(args.workload + ("_cow" if args.cow else "") +
                             ("_cascade" if st.prefix_len else "") + ("_fp8" if st.fp8 else ""))

    # ------------------------------------------------ end to end (host buffers)
    # Every step copies its inputs from pinned host memory into device input
    # tensors, runs the step, and reads every layer's output back.  Steps
    # alternate between two device buffer sets, with the
    # host-to-device copies on one side stream and the device-to-host copies
    # on another: step i+1's inputs arrive while step i runs, and step i's
    # output leaves while step i+1 runs.  A graph-replayed step gets a second
    # graph, captured on the second buffer set.
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(st.vals.q)] + [pin(t) for t in st.vals.k_new + st.vals.v_new] + \
        [pin(st.tables), pin(st.lens), pin(st.slots)]
    h_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in st.out]
    h2d = sum(t.nbytes for t in h_in)
    d2h = sum(t.nbytes for t in h_out)
    nl = spec.num_layers
    d_in = [[st.vals.q] + list(st.vals.k_new) + list(st.vals.v_new) + [st.tables, st.lens, st.slots]]
    d_out = [st.out]
    d_in.append([t.clone() for t in d_in[0]])
    d_out.append([o.clone() for o in st.out])

    def run_set(b, stream=None):
        ins = d_in[b]
        st.run(q=ins[0], k_new=ins[1:1 + nl], v_new=ins[1 + nl:1 + 2 * nl], tables=ins[-3],
               lens=ins[-2], slots=ins[-1], out=d_out[b], stream=stream)

    graphs = None
    if graph is not None:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run_set(1)
        torch.cuda.current_stream().wait_stream(side)
        graph1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph1):
            run_set(1)
        torch.cuda.synchronize()
        graphs = [graph, graph1]
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    read = [torch.cuda.Event(), torch.cuda.Event()]
    k = [0]  # steps issued

    def e2e_step():
        b = k[0] % 2
        with torch.cuda.stream(up):
            if k[0] >= 2:
                up.wait_event(done[b])  # step k-2 has read this set's inputs
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
            ready[b].record(up)
        main.wait_event(ready[b])
        if k[0] >= 2:
            main.wait_event(read[b])  # step k-2's output has left
        if graphs is not None:
            graphs[b].replay()
        else:
            run_set(b, stream=main)
        done[b].record(main)
        with torch.cuda.stream(down):
            down.wait_event(done[b])
            for h, o in zip(h_out, d_out[b]):
                h.copy_(o, non_blocking=True)
            read[b].record(down)
        k[0] += 1

    def e2e_drain():
        main.wait_stream(up)
        main.wait_stream(down)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_drain()
    torch.cuda.synchronize()
    e2e_steps = max(3, args.steps // 2)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(main)
    up.wait_stream(main)    # no copy of the timed steps starts before t0
    down.wait_stream(main)
    for _ in range(e2e_steps):
        e2e_step()
    e2e_drain()
    t1.record(main)
    torch.cuda.synchronize()
    e2e_s, e2e_bytes = reduce_over_ranks(t0.elapsed_time(t1) / 1e3,
                                         st.step_bytes() * e2e_steps, device)
    api.check_error()

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / n_timed,
        "repeats": repeats, "timed_steps": n_timed, "timed_seconds": total_ms / 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (f"e4m3 K/V ({spec.dtype} q/out, E4M3 x E5M2 products, fp32 accumulate)"
                  if st.fp8
                  else spec.dtype), "data": "synthetic",
        "config": {
            "workload": f"{spec.name}: {spec.describe}",
            "num_seqs": spec.num_seqs, "q_heads": spec.num_q_heads,
            "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "block_size": spec.block_size, "layers": spec.num_layers,
            "mean_seq_len": float(np.mean(st.lay.seq_lens)),
            "partition_tokens": st.resolved_P,
            "partial_tokens": st.partial_tokens,
            "decode_ctas_per_sm": api.ctas_per_sm(spec.head_dim,
                                                  spec.num_q_heads // spec.num_kv_heads,
                                                  st.vals.q.dtype),
            "step": ("copy_blocks (if any) + pa_decode_cascade (prefix pass; tails with the "
                     "cache write and the merge), every layer" if st.prefix_len else
                     "copy_blocks (if any) + pa_decode_step (cache write + decode), every layer"),
            "decode_path": (f"cascade, shared prefix {st.prefix_len} positions"
                            if st.prefix_len else "paged"),
            "launch": "CUDA graph replay" if graph is not None else "eager",
            "kv_format": ("E4M3 codes, scale 1/64 per pool, quantised from the same N(0,1) "
                          "values" if st.fp8 else spec.dtype),
            "decode_kernel": ("tensor cores (tcgen05 kind::f8f6f4 on the E4M3 codes, q and P as "
                              "E5M2 terms)") if st.fp8 else
                             ("CUDA cores" if args.decode_impl == "cuda_cores"
                              else "tensor cores (tcgen05)"),
            "l2": ("inputs larger than L2 (%.2f GB per step)" % (st.step_bytes() / 1e9))
            if flush is None else "L2 flushed (256 MiB write) before every step",
        },
        "pct_of_peak": 100.0 * value / peak,
        # bytes plain paged decode would read for the same attention, per second
        "logical_gbs": value * (st.logical_bytes + st.write_bytes + st.copy_bytes) /
        (st.decode_bytes + st.write_bytes + st.copy_bytes),
        "tokens_per_s": spec.num_seqs * world / (secs / n_timed),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": kernel_note,
                     "bytes_per_launch": launch_bytes, "avg_launch_ms": dec_avg_ms,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "e2e": {"value": e2e_bytes / e2e_s / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": 1e3 * e2e_s / e2e_steps,
                "copies": ("pinned host buffers; two device buffer sets (a graph each when "
                           "replayed), copies on side streams overlapping the neighbouring "
                           "steps")},
        "gpu_launches": st.launches_per_step * n_timed,
        "clocks": clocks.summary(),
    }
    if cev:
        copy_s = statistics.mean(a.elapsed_time(b) for a, b in cev) / 1e3
        per_launch = st.copy_bytes  # K and V blocks read and written, one layer
        line["copy_blocks"] = {
            "pairs": int(len(st.lay.pre_copies)), "launches": len(cev),
            "bytes_per_launch": int(per_launch), "avg_us": 1e6 * copy_s,
            "achieved_gbs": per_launch / copy_s / 1e9,
            "note": ("pa_copy_blocks of the layout's copy-on-write pairs (K and V), re-run "
                     "every step as its timing stand-in, CUDA events")}
    if args.cow:
        line["config"]["copy_on_write"] = (
            "shared prompt of 4,112 positions: its last block half full and shared, so the "
            "first tail token of 63 of the 64 sequences copies it")
    if plan.apc:
        line["config"]["layout"] = ("separate requests with one prompt, shared by the "
                                    "prefix-caching pool (pa_pcache)")
        line["host_allocator"] = host_pool_timing(plan)
    if world == 1 and not args.no_cpu_baseline:
        inputs = oracle_inputs(plan)
        secs_c, nbytes_c, toks_c, nseq_c, threads = oracle_sample(plan, inputs, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": nbytes_c / secs_c / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 oracle decode of {sample_text(nseq_c, spec.num_seqs)} (all "
                      f"heads), {secs_c:.1f} s on host cores",
            "cpu_model": cpu_model(),
            "single_thread_value": single_thread_gbs(plan, inputs, 3.0)}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama",
                    choices=["tiny", "qwen", "llama", "prefix", "long"])
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the batch (profiling of small cases only)")
    ap.add_argument("--len-range", type=int, nargs=2, default=None, metavar=("LO", "HI"),
                    help="cached lengths uniform in [LO, HI] (profiling of small cases only)")
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (profiling of small cases only)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--graph", default="auto", choices=["auto", "on", "off"],
                    help="replay the step as a CUDA graph (auto: when the step has >1 layer)")
    ap.add_argument("--partition-tokens", type=int, default=None,
                    help="override the workload's split-KV partition size (0 auto, -1 single pass)")
    ap.add_argument("--decode-impl", default="auto",
                    choices=["auto", "cuda_cores", "tensor_cores"],
                    help="decode kernel (default: the library's automatic choice)")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix decode: attend the prefix every sequence shares "
                         "through its block table once per KV head (prefix workload)")
    ap.add_argument("--kv", default="16bit", choices=["16bit", "fp8"],
                    help="K/V pool format: the workload's 16-bit type, or E4M3 codes with one "
                         "scale per pool (q and out stay 16-bit)")
    ap.add_argument("--cow", action="store_true",
                    help="prefix workload, copy-on-write reading: a 4,112-position shared "
                         "prompt whose half-full last block is copied 63 times, every step")
    ap.add_argument("--apc", action="store_true",
                    help="prefix workload as separate requests laid out by the prefix-caching "
                         "pool (automatic prefix caching) instead of forks")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=8.0,
                    help="reference arm: at most this much oracle time a step")
    ap.add_argument("--ref-total-seconds", type=float, default=120.0,
                    help="reference arm: about this much oracle time over all steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-timed-seconds", type=float, default=2.0,
                    help="repeat the K timed steps until the timed region lasts at least this "
                         "long (the count is reported as `repeats`)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    rank, world, local_rank = dist_env()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} needs {args.gpus} ranks, one per GPU: launch with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py "
                 f"--gpus {args.gpus} (this process sees WORLD_SIZE={world})")
    if args.apc and args.workload != "prefix":
        ap.error("--apc applies to the prefix workload")
    if args.cow and (args.workload != "prefix" or args.apc):
        ap.error("--cow applies to the prefix workload laid out by forks")
    if args.kv == "fp8" and args.cascade:
        ap.error("--cascade reads 16-bit pools")
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
