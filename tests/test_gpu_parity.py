"""GPU parity: the CUDA kernels, called through the C ABI, against the fp64
CPU oracle on the same seeded inputs.

Decode outputs must satisfy |gpu - ref| <= 2e-3 + 1e-2 |ref| element by
element; cache writes and block copies must be bit-exact over the whole pool.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_64_gb300 import _lib, api, workloads

from _parity import Case, assert_close, bits

pytestmark = pytest.mark.gpu

LOG2E = 1.0 / math.log(2.0)


@pytest.fixture(scope="module", autouse=True)
def cuda_ready():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    _lib.load()  # fails loudly when the library was not built
    yield
    api.check_error()


def full_step_parity(case, layer=0, partition=None, seqs=None):
    blocks = None if seqs is None else case.blocks_of(seqs)
    if case.lay.pre_copies.size:
        blocks = None  # copies read blocks outside the sample: take whole pools
    hk, hv = case.snapshot(layer, blocks)
    case.gpu_writes(layer)
    out = case.gpu_decode(layer, partition)
    ref = case.oracle_step(layer, hk, hv, seqs)
    api.check_error()
    rows = None if seqs is None else np.asarray(seqs)
    return assert_close(out, ref, case.spec.name, mask_rows=rows)


# -------------------------------------------------------------- cache write
@pytest.mark.parametrize("name", ["tiny", "qwen", "llama", "long"])
def test_cache_write_bit_exact(name):
    kw = {"tiny": {}, "qwen": {"num_seqs": 64}, "llama": {"num_seqs": 16, "len_range": (512, 1024)},
          "long": {"num_seqs": 2, "len_range": (2000, 3000)}}[name]
    case = Case(workloads.make_plan(name, **kw))
    hk, hv = case.snapshot(0)
    slots = case.slots.clone()
    slots[::3] = -1  # negative slot: skip
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    api.cache_write(case.vals.k_new[0], case.vals.v_new[0], slots, kp, vp)
    oracle.cache_write(hk, hv, bits(case.vals.k_new[0]), bits(case.vals.v_new[0]),
                       slots.cpu().numpy())
    api.check_error()
    assert np.array_equal(bits(kp), hk)
    assert np.array_equal(bits(vp), hv)


def test_cache_write_many_tokens_bit_exact():
    """The prefix workload writes ~9k tail tokens in one call."""
    case = Case(workloads.make_plan("prefix", cow=True))
    hk, hv = case.snapshot(0)
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    api.copy_blocks([kp], [vp], case.pre_copies)
    api.cache_write(case.vals.k_pre[0], case.vals.v_pre[0], case.pre_slots, kp, vp)
    oracle.copy_blocks([hk, hv], case.ref_lay.pre_copies)
    oracle.cache_write(hk, hv, bits(case.vals.k_pre[0]), bits(case.vals.v_pre[0]),
                       case.ref_lay.pre_slots)
    api.check_error()
    assert np.array_equal(bits(kp), hk) and np.array_equal(bits(vp), hv)


# -------------------------------------------------------------- copy blocks
def test_copy_blocks_cow_pairs_bit_exact():
    case = Case(workloads.make_plan("prefix", cow=True))
    assert case.pre_copies.shape == (63, 2)
    hk, hv = case.snapshot(0)
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    api.copy_blocks([kp], [vp], case.pre_copies)
    oracle.copy_blocks([hk, hv], case.ref_lay.pre_copies)
    api.check_error()
    assert np.array_equal(bits(kp), hk) and np.array_equal(bits(vp), hv)


def test_copy_blocks_multi_layer_bit_exact():
    """Three layers of the Qwen-shaped pool, 40 random disjoint pairs."""
    plan = workloads.make_plan("qwen", num_seqs=8)
    case = Case(plan, layers=3)
    rng = np.random.default_rng(7)
    ids = rng.choice(plan.num_blocks, 80, replace=False)
    pairs = np.stack([ids[:40], ids[40:]], axis=1).astype(np.int64)
    hosts = [case.snapshot(l) for l in range(3)]
    api.copy_blocks(case.vals.k_pools, case.vals.v_pools, torch.as_tensor(pairs, device="cuda"))
    for hk, hv in hosts:
        oracle.copy_blocks([hk, hv], pairs)
    api.check_error()
    for l, (hk, hv) in enumerate(hosts):
        assert np.array_equal(bits(case.vals.k_pools[l]), hk)
        assert np.array_equal(bits(case.vals.v_pools[l]), hv)


def test_copy_blocks_empty_is_noop():
    case = Case(workloads.make_plan("prefix"))
    assert case.pre_copies.numel() == 0  # full shared blocks are never copied
    before = bits(case.vals.k_pools[0])
    api.copy_blocks([case.vals.k_pools[0]], [case.vals.v_pools[0]], case.pre_copies)
    api.check_error()
    assert np.array_equal(bits(case.vals.k_pools[0]), before)


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("partition", [None, -1, 16, 32])
def test_decode_tiny_full(partition):
    """Tiny workload: every output compared; single pass and split-KV with
    partitions of one and two blocks."""
    full_step_parity(Case(workloads.make_plan("tiny")), partition=partition)


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
def test_decode_small_every_output(name, kw, partition):
    """Reduced workloads (same heads, d, B, dtype) where the oracle checks
    every output: many tiles, ragged last blocks, several partitions."""
    full_step_parity(Case(workloads.make_plan(name, **kw)), partition=partition)


def test_decode_prefix_cow_small():
    full_step_parity(Case(workloads.make_plan("prefix", num_seqs=6, cow=True)))


@pytest.mark.parametrize("name,cow,nsample", [("llama", False, 12), ("long", False, 3),
                                             ("prefix", True, 8), ("qwen", False, 16)])
def test_decode_full_size_sampled(name, cow, nsample):
    """Full-size workloads in the launch configuration the benchmark times;
    the oracle checks every head of a sample of sequences (always including
    the longest and the shortest)."""
    case = Case(workloads.make_plan(name, cow=cow))
    lens = case.lay.seq_lens
    rng = np.random.default_rng(11)
    seqs = {int(np.argmax(lens)), int(np.argmin(lens))}
    seqs.update(rng.choice(len(lens), nsample, replace=False).tolist())
    full_step_parity(case, seqs=sorted(seqs)[:nsample + 2])


def test_decode_qwen_layers_sampled():
    """Several layers of the 24-layer Qwen-shaped step, each with its own pools."""
    case = Case(workloads.make_plan("qwen"), layers=3)
    seqs = [0, 5, int(np.argmax(case.lay.seq_lens))]
    for layer in range(3):
        full_step_parity(case, layer=layer, seqs=seqs)


# ------------------------------------------------------------- edge cases
def test_zero_and_one_token_sequences():
    case = Case(workloads.make_plan("tiny"))
    case.gpu_writes(0)
    lens = case.lay.seq_lens.copy()
    lens[0], lens[1] = 0, 1
    lens_t = torch.as_tensor(lens, device="cuda")
    for P in (-1, 16, 0):
        out = torch.full_like(case.vals.q, float("nan"))
        api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                   lens_t, case.max_seq_len, case.plan.scale, partition_tokens=P)
        hk, hv = bits(case.vals.k_pools[0]), bits(case.vals.v_pools[0])
        ref = oracle.decode(bits(case.vals.q), hk, hv, case.ref_lay.block_tables, lens,
                            case.plan.scale, "f16")
        assert torch.all(out[0] == 0)
        # one token: the output is that token's value vector (rounded once)
        v0 = oracle.widen(hv[case.ref_lay.block_tables[1, 0], :, 0, :], "f16")
        assert np.allclose(ref[1], np.repeat(v0, 2, axis=0), atol=0)
        assert_close(out, ref, f"edge P={P}")
    api.check_error()


def test_all_zero_lengths():
    case = Case(workloads.make_plan("tiny"))
    lens_t = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.full_like(case.vals.q, float("nan"))
    api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
               lens_t, 0, case.plan.scale, partition_tokens=0)
    api.check_error()
    assert torch.all(out == 0)


@pytest.mark.parametrize("name,kw", [("llama", {"num_seqs": 4, "len_range": (600, 1500)}),
                                     ("qwen", {"num_seqs": 16})])
def test_stale_slots_poisoned_with_nan(name, kw):
    """NaN in every unreferenced block and in every slot past a sequence's
    length: the output stays finite and equal to the oracle's (which ignores
    those slots by definition)."""
    case = Case(workloads.make_plan(name, **kw))
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
    out = case.gpu_decode(0)
    assert torch.isfinite(out).all()
    hk, hv = bits(kp), bits(vp)
    ref = oracle.decode(bits(case.vals.q), hk, hv, case.ref_lay.block_tables,
                        case.ref_lay.seq_lens, case.plan.scale, case.spec.dtype)
    assert_close(out, ref, "poison")
    api.check_error()


def test_paging_invariance_bitwise():
    """The same logical cache under a different physical permutation of the
    blocks gives bitwise the same output (only the addressing changes)."""
    case = Case(workloads.make_plan("llama", num_seqs=5, len_range=(700, 1800)))
    case.gpu_writes(0)
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    nb = case.plan.num_blocks
    perm = torch.as_tensor(np.random.default_rng(3).permutation(nb), device="cuda")
    kp2 = torch.empty_like(kp)
    vp2 = torch.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    tables2 = perm.to(torch.int32)[case.tables.long()]
    for P in (-1, 0, 512):
        a = torch.empty_like(case.vals.q)
        b = torch.empty_like(case.vals.q)
        api.decode(a, case.vals.q, kp, vp, case.tables, case.lens, case.max_seq_len,
                   case.plan.scale, partition_tokens=P)
        api.decode(b, case.vals.q, kp2, vp2, tables2, case.lens, case.max_seq_len,
                   case.plan.scale, partition_tokens=P)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), P
    api.check_error()


def test_uniform_keys_give_mean_values_on_gpu():
    """All keys of a sequence equal -> output = mean of its values."""
    case = Case(workloads.make_plan("llama", num_seqs=3, len_range=(513, 900)))
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    kp.copy_(kp[0:1, :, 0:1, :].expand_as(kp))
    out = case.gpu_decode(0, partition=256)
    hk, hv = bits(kp), bits(vp)
    ref = oracle.decode(bits(case.vals.q), hk, hv, case.ref_lay.block_tables,
                        case.ref_lay.seq_lens, case.plan.scale, "bf16")
    assert_close(out, ref, "uniform keys")
    api.check_error()


def test_decode_on_side_stream_and_repeat_deterministic():
    case = Case(workloads.make_plan("llama", num_seqs=8, len_range=(512, 3000)))
    case.gpu_writes(0)
    a = case.gpu_decode(0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = case.gpu_decode(0)
    s.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    api.check_error()


# ------------------------------------------------ fused write + decode
@pytest.mark.parametrize("name,kw,partition", [
    ("tiny", {}, None), ("tiny", {}, 16),
    ("qwen", {"num_seqs": 24}, None),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 512),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 128),
    ("prefix", {"num_seqs": 6, "cow": True}, None),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, None),
])
def test_decode_step_fused_matches_oracle(name, kw, partition):
    """pa_decode_step (new token written inside the decode launch, and the
    split-KV combine inside it when a sequence has <= 8 partitions) against
    the oracle's cache write + decode; the pools afterwards are bit-exact."""
    case = Case(workloads.make_plan(name, **kw))
    hk, hv = case.snapshot(0)
    out = case.gpu_step_fused(0, partition)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    assert_close(out, ref, f"fused step {name}")
    assert np.array_equal(bits(case.vals.k_pools[0]), hk)
    assert np.array_equal(bits(case.vals.v_pools[0]), hv)


def test_fused_combine_garbage_workspace_and_graph_replay():
    """The fused combine's ready flags need no initialisation (garbage
    workspace), and a CUDA graph of the step replays correctly (each replay
    reuses the captured epoch; the combining CTA clears the flags it read)."""
    case = Case(workloads.make_plan("llama", num_seqs=6, len_range=(900, 2100)))
    spec, P = case.spec, 512
    size = api.workspace_size(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                              spec.block_size, case.max_seq_len, P, case.dtype)
    ws = api.alloc_workspace(size, "cuda")
    ws.fill_(0xFF)
    hk, hv = case.snapshot(0)
    case.gpu_writes(0)
    ref = case.oracle_step(0, hk, hv)
    out = torch.empty_like(case.vals.q)
    api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
               case.lens, case.max_seq_len, case.plan.scale, partition_tokens=P, workspace=ws)
    api.check_error()
    assert_close(out, ref, "garbage workspace")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0],
                       case.tables, case.lens, case.max_seq_len, case.plan.scale,
                       partition_tokens=P, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert_close(out, ref, "graph replay")
    api.check_error()


def test_decode_step_rejects_a_slot_off_the_table():
    case = Case(workloads.make_plan("tiny"))
    bad = case.slots.clone()
    bad[2] += 1  # not the slot of position L-1
    out = torch.empty_like(case.vals.q)
    api.decode_step(out, case.vals.q, case.vals.k_new[0], case.vals.v_new[0], bad,
                    case.vals.k_pools[0], case.vals.v_pools[0], case.tables, case.lens,
                    case.max_seq_len, case.plan.scale)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6


# -------------------------------------------------------- split-KV steps
@pytest.mark.parametrize("name,kw,P,R", [
    ("long", {"num_seqs": 2, "len_range": (1500, 2600)}, 512, 0),
    ("tiny", {}, 16, 0),
    ("qwen", {"num_seqs": 8}, 64, 0),
    ("long", {"num_seqs": 2, "len_range": (1500, 2600)}, 512, 2),   # two partitions a CTA
    ("long", {"num_seqs": 2, "len_range": (1500, 2600)}, 512, 4),   # ragged last span
    ("llama", {"num_seqs": 4, "len_range": (300, 1200)}, 256, 4),
])
def test_partitions_match_oracle(span, name, kw, P, R):
    """Split-KV step 2 on its own: (m, l, O) per partition against the
    oracle's partials; empty partitions hold (-inf, 0, 0).  With R > 0 a CTA
    computes R consecutive partitions and still writes each one's partial."""
    if R:
        span(R)
    case = Case(workloads.make_plan(name, **kw))
    case.gpu_writes(0)
    spec = case.spec
    size = api.workspace_size(spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                              spec.block_size, case.max_seq_len, P, case.dtype)
    ws = api.alloc_workspace(size, "cuda")
    ws.fill_(0xAB)
    api.decode_partitions(case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
                          case.lens, case.max_seq_len, case.plan.scale, P, ws)
    m, l, o = api.partials_view(ws, spec.num_seqs, spec.num_q_heads, spec.head_dim,
                                case.max_seq_len, P)
    hk, hv = bits(case.vals.k_pools[0]), bits(case.vals.v_pools[0])
    NP = api.partition_count(case.max_seq_len, P)
    rm, rl, ro = oracle.partitions(bits(case.vals.q), hk, hv, case.ref_lay.block_tables,
                                   case.ref_lay.seq_lens, case.plan.scale, spec.dtype, P, NP)
    gm = m.double().cpu().numpy() / LOG2E   # base-2 units -> natural
    gl = l.double().cpu().numpy()
    go = o.double().cpu().numpy()
    empty = np.isinf(rm)
    assert np.array_equal(np.isinf(gm), empty)
    assert (gl[empty] == 0).all() and (go[empty] == 0).all()
    ok = ~empty
    # fp32 intermediates: m to 1e-4 absolute, l to 1e-4 relative, O within
    # the output tolerance (it is rounded once more before use)
    assert np.max(np.abs(gm[ok] - rm[ok])) <= 1e-4 * (1 + np.max(np.abs(rm[ok])))
    assert np.max(np.abs(gl[ok] - rl[ok]) / rl[ok]) <= 1e-4
    err = np.abs(go[ok] - ro[ok])
    assert (err <= 2e-3 + 1e-2 * np.abs(ro[ok])).all(), float(err.max())
    api.check_error()


@pytest.mark.parametrize("dtype,d,P,lens", [
    ("f16", 128, 64, [0, 1, 64, 65, 200, 448, 129]),
    ("bf16", 128, 64, [0, 1, 64, 65, 200, 448, 129]),
    # hundreds of partials a row (313, 1 and 2): the four-at-a-time walk,
    # its tail, and empty partials inside a row
    ("bf16", 64, 16, [5000, 16, 17]),
    ("f16", 128, 32, [2049, 4000, 33, 95]),
])
def test_split_reduce_matches_oracle(dtype, d, P, lens):
    """Split-KV step 3 on its own: oracle partials (converted to the
    workspace's fp32 base-2 layout) combined by the kernel against the
    oracle's combine."""
    rng = np.random.default_rng(5 + len(lens))
    lens = np.array(lens, dtype=np.int32)
    S, Hq = len(lens), 6
    max_len = int(lens.max())
    NP = api.partition_count(max_len, P)
    m = rng.normal(0, 3, (S, Hq, NP))
    l = rng.uniform(0.5, 40, (S, Hq, NP))
    o = rng.normal(0, 1, (S, Hq, NP, d))
    for i, L in enumerate(lens):
        k = -(-int(L) // P)
        m[i, :, k:], l[i, :, k:], o[i, :, k:] = -np.inf, 0, 0
        if k > 8:  # a few empty partials inside the row (all positions masked)
            hole = rng.choice(k - 1, 3, replace=False)
            m[i, :, hole], l[i, :, hole], o[i, :, hole] = -np.inf, 0, 0
    tdt = workloads.torch_dtype(dtype)
    size = api.workspace_size(S, Hq, 1, d, 16, max_len, P, tdt)
    ws = api.alloc_workspace(size, "cuda")
    gm, gl, go = api.partials_view(ws, S, Hq, d, max_len, P)
    gm.copy_(torch.as_tensor(m * LOG2E, dtype=torch.float32))
    gl.copy_(torch.as_tensor(l, dtype=torch.float32))
    go.copy_(torch.as_tensor(o, dtype=torch.float32))
    out = torch.full((S, Hq, d), float("nan"), dtype=tdt, device="cuda")
    api.split_kv_reduce(out, ws, torch.as_tensor(lens, device="cuda"), max_len, P)
    # oracle on the fp32-rounded partials the kernel actually read
    ref = oracle.reduce(gm.double().cpu().numpy() / LOG2E, gl.double().cpu().numpy(),
                        go.double().cpu().numpy())
    for i, L in enumerate(lens):
        if L == 0:
            assert torch.all(out[i] == 0)
    assert_close(out, ref, f"reduce d={d} P={P}")
    api.check_error()


# ------------------------------------------------------------- error word
def test_bad_indices_are_reported_not_dereferenced():
    case = Case(workloads.make_plan("tiny"))
    api.check_error()
    kp, vp = case.vals.k_pools[0], case.vals.v_pools[0]
    nb = case.plan.num_blocks
    # cache write: one slot past the pool
    bad = case.slots.clone()
    bad[1] = nb * case.spec.block_size + 5
    before = bits(kp)
    api.cache_write(case.vals.k_new[0], case.vals.v_new[0], bad, kp, vp)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6
    after = bits(kp)
    hk = before.copy()
    hv = bits(vp)  # only K compared below
    good = bad.cpu().numpy().copy()
    good[1] = -1
    oracle.cache_write(hk, hv.copy(), bits(case.vals.k_new[0]), bits(case.vals.v_new[0]), good)
    assert np.array_equal(after, hk)
    # decode: a block-table entry past the pool and a negative one
    tables = case.tables.clone()
    tables[0, 0] = nb + 100
    tables[2, 1] = -7
    out = torch.empty_like(case.vals.q)
    api.decode(out, case.vals.q, kp, vp, tables, case.lens, case.max_seq_len, case.plan.scale)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6
    # a length beyond max_seq_len
    lens = case.lens.clone()
    lens[3] = case.max_seq_len + 50
    api.decode(out, case.vals.q, kp, vp, case.tables, lens, case.max_seq_len, case.plan.scale)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6
    # copy pair with a bad block id
    pairs = torch.tensor([[0, nb + 3]], dtype=torch.int64, device="cuda")
    api.copy_blocks([kp], [vp], pairs)
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 6
    api.check_error()  # cleared


def test_bounded_wait_times_out_and_context_survives():
    api.selftest_wait_timeout()
    with pytest.raises(_lib.PagedAttentionError) as e:
        api.check_error()
    assert e.value.code == 5
    # the context is still usable
    full_step_parity(Case(workloads.make_plan("tiny")))


# ------------------------------------- several partitions per CTA (span)
@pytest.fixture
def span():
    """Force the number of consecutive split-KV partitions a tensor-core CTA
    computes; restored afterwards."""
    prev = []

    def set_span(n):
        prev.append(api.set_decode_span(n))

    yield set_span
    if prev:
        api.set_decode_span(prev[0])


@pytest.mark.parametrize("name,kw,partition,R", [
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512, 2),
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512, 3),   # ragged last span
    ("long", {"num_seqs": 2, "len_range": (3000, 5000)}, 512, 4),
    ("llama", {"num_seqs": 6, "len_range": (512, 2100)}, 256, 4),  # 2 tiles a partition
    ("llama", {"num_seqs": 6, "len_range": (100, 700)}, 128, 8),   # 1 tile a partition
    ("qwen", {"num_seqs": 24}, 128, 3),
])
def test_decode_partitions_per_cta_every_output(span, name, kw, partition, R):
    """A CTA computing R consecutive partitions writes each partition's own
    partial: every output matches the oracle, with the fused combine (<= 8
    partitions) or the separate reduce (more)."""
    span(R)
    full_step_parity(Case(workloads.make_plan(name, **kw)), partition=partition)


@pytest.mark.parametrize("R", [2, 4])
def test_decode_step_fused_partitions_per_cta(span, R):
    """The fused cache write runs in the CTA whose span holds the last
    partition."""
    span(R)
    case = Case(workloads.make_plan("long", num_seqs=2, len_range=(1000, 1900)))
    hk, hv = case.snapshot(0)
    out = case.gpu_step_fused(0, 256)
    ref = case.oracle_step(0, hk, hv)
    api.check_error()
    assert_close(out, ref, "fused step, span")
    assert np.array_equal(bits(case.vals.k_pools[0]), hk)
    assert np.array_equal(bits(case.vals.v_pools[0]), hv)


def test_decode_partitions_per_cta_zero_and_one_token(span):
    span(4)
    case = Case(workloads.make_plan("llama", num_seqs=6, len_range=(100, 700)))
    case.gpu_writes(0)
    lens = case.lay.seq_lens.copy()
    lens[0], lens[1] = 0, 1
    lens_t = torch.as_tensor(lens, device="cuda")
    hk, hv = case.snapshot(0)
    out = torch.full_like(case.vals.q, float("nan"))
    api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
               lens_t, case.max_seq_len, case.plan.scale, partition_tokens=128)
    api.check_error()
    ref = oracle.decode(bits(case.vals.q), hk, hv, case.lay.block_tables, lens, case.plan.scale,
                        case.spec.dtype)
    assert torch.all(out[0] == 0)
    assert_close(out, ref, "span, zero and one token")


# ------------------------------------------------ compact grid (<= 128 seqs)
@pytest.mark.parametrize("num_seqs", [127, 128, 129])       # 129: the 3-D grid
@pytest.mark.parametrize("partition,R", [(128, 1), (256, 2), (0, 0)])
def test_decode_compact_grid_mixed_lengths(span, num_seqs, partition, R):
    """Batches around the compact-grid limit with zero-length, one-token and
    long sequences in the middle of the batch: every output."""
    if R:
        span(R)
    case = Case(workloads.make_plan("qwen", num_seqs=num_seqs))
    case.gpu_writes(0)
    lens = case.lay.seq_lens.copy()
    rng = np.random.default_rng(num_seqs)
    pick = rng.choice(num_seqs, 12, replace=False)
    lens[pick[:6]] = 0
    lens[pick[6:9]] = 1
    lens_t = torch.as_tensor(lens, device="cuda")
    hk, hv = case.snapshot(0)
    out = torch.full_like(case.vals.q, float("nan"))
    api.decode(out, case.vals.q, case.vals.k_pools[0], case.vals.v_pools[0], case.tables,
               lens_t, case.max_seq_len, case.plan.scale, partition_tokens=partition)
    api.check_error()
    ref = oracle.decode(bits(case.vals.q), hk, hv, case.lay.block_tables, lens, case.plan.scale,
                        case.spec.dtype)
    assert torch.all(out[torch.as_tensor(pick[:6], device="cuda")] == 0)
    assert_close(out, ref, f"compact S={num_seqs} P={partition} R={R}")


# ------------------------- compact grid capped at the resident slots
@pytest.mark.parametrize("hq,hkv,d,dtype,num_seqs,lens,partition,R,fused", [
    (14, 2, 64, "f16", 100, (2000, 3000), 512, 1, False),   # ~1,000 items, 304 CTAs
    (14, 2, 64, "f16", 100, (2000, 3000), 512, 1, True),    # the same, fused cache write
    (32, 8, 128, "bf16", 40, (1100, 1500), 512, 1, True),   # d = 128: 960 items
])
def test_decode_compact_several_items_per_cta(span, hq, hkv, d, dtype, num_seqs, lens, partition,
                                              R, fused):
    """A compact launch (one partition a CTA) whose upper bound (every
    sequence at the longest length) is within four waves runs one CTA a
    resident slot; when the batch has more items than that, each CTA
    computes several in turn and the arrival counters pick the combining
    CTA.  Every output."""
    span(R)
    case = Case(workloads.make_shape_plan(num_seqs, hq, hkv, d, 16, dtype, lens, seed=71 + d))
    hk, hv = case.snapshot(0)
    if fused:
        out = case.gpu_step_fused(0, partition)
    else:
        case.gpu_writes(0)
        out = case.gpu_decode(0, partition)
    api.check_error()
    ref = case.oracle_step(0, hk, hv)
    assert_close(out, ref, f"several items a CTA S={num_seqs} d={d} P={partition} R={R}")
