"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its source), closed forms,
special cases that reduce to a library routine (numpy / scipy softmax on a
contiguous array), invariants, and brute force on tiny inputs.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from conftest import read_json

RNG = np.random.default_rng(20261202)


def f16_bits(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def bf16_bits_truncate(x):
    # Only used to make inputs: exact bf16 values (x already representable)
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_values(shape, rng):
    # Random values that are exactly representable in bf16 (8 significant bits)
    raw = rng.standard_normal(shape).astype(np.float32)
    return (raw.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


def widen_lib(bits, dtype):
    """Library widening used as the independent side of the checks."""
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):  # NaN patterns stay NaN
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def scatter_into_pool(logical, table, num_blocks, block_size, fill):
    """Test-side layout: put logical[p] (shape [L, Hkv, d]) at slot p % B of
    physical block table[p // B] of a pool [NB, Hkv, B, d] filled with
    `fill` elsewhere.  Written independently of the oracle."""
    L, hkv, d = logical.shape
    pool = np.full((num_blocks, hkv, block_size, d), fill, dtype=np.uint16)
    for p in range(L):
        pool[table[p // block_size], :, p % block_size, :] = logical[p]
    return pool


def contiguous_attention(q, K, V, scale):
    """softmax(scale * q K^T) V per query head on contiguous fp64 arrays."""
    hq = q.shape[0]
    hkv = K.shape[1]
    g = hq // hkv
    out = np.zeros((hq, q.shape[1]))
    for h in range(hq):
        if K.shape[0] == 0:
            continue
        s = scale * (K[:, h // g, :] @ q[h])
        out[h] = softmax(s) @ V[:, h // g, :]
    return out


def build_case(lengths, hq, hkv, d, block_size, dtype, rng, fill_bits=None):
    """Random paged inputs: per sequence logical K/V, scattered into a pool
    through a random permutation of physical blocks."""
    nblk = [math.ceil(L / block_size) for L in lengths]
    num_blocks = sum(nblk) + 3
    perm = rng.permutation(num_blocks)
    maxb = max(max(nblk), 1)
    tables = np.zeros((len(lengths), maxb), dtype=np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = perm[pos:pos + n]
        pos += n
    if dtype == "f16":
        mk = lambda shape: f16_bits(rng.standard_normal(shape))
    else:
        mk = lambda shape: bf16_bits_truncate(bf16_values(shape, rng))
    fill = np.uint16(0x7E00) if fill_bits is None else np.uint16(fill_bits)  # NaN for f16
    if dtype == "bf16" and fill_bits is None:
        fill = np.uint16(0x7FC0)  # bf16 NaN
    k_pool = np.full((num_blocks, hkv, block_size, d), fill, dtype=np.uint16)
    v_pool = k_pool.copy()
    logical = []
    for i, L in enumerate(lengths):
        K = mk((L, hkv, d))
        V = mk((L, hkv, d))
        logical.append((K, V))
        for p in range(L):
            k_pool[tables[i, p // block_size], :, p % block_size, :] = K[p]
            v_pool[tables[i, p // block_size], :, p % block_size, :] = V[p]
    q = mk((len(lengths), hq, d))
    return q, k_pool, v_pool, tables, np.asarray(lengths, dtype=np.int32), logical


# ---------------------------------------------------------------- widening
def test_widen_f16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "f16")
    ref = widen_lib(bits, "f16")
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_widen_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits, "bf16")
    ref = widen_lib(bits, "bf16")
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


# ------------------------------------------------------------- decode math
@pytest.mark.parametrize("block_size", [1, 4, 16, 32])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_paged_equals_contiguous(block_size, dtype):
    """Reading through the table equals reading one flat array (the pages'
    central claim: only the addressing changes)."""
    rng = np.random.default_rng(block_size * 7 + (dtype == "bf16"))
    lengths = [1, 5, 17, 33, 64, 13]
    hq, hkv, d = 6, 2, 16
    q, kp, vp, tables, sl, logical = build_case(lengths, hq, hkv, d, block_size, dtype, rng)
    scale = 1.0 / math.sqrt(d)
    got = oracle.decode(q, kp, vp, tables, sl, scale, dtype)
    for i, (K, V) in enumerate(logical):
        ref = contiguous_attention(widen_lib(q[i], dtype), widen_lib(K, dtype),
                                   widen_lib(V, dtype), scale)
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-13)


def test_brute_force_tiny_pure_python():
    """Tiny case recomputed with plain Python floats and math.exp."""
    rng = np.random.default_rng(3)
    lengths = [3, 6]
    q, kp, vp, tables, sl, logical = build_case(lengths, 2, 1, 4, 4, "f16", rng)
    scale = 0.5
    got = oracle.decode(q, kp, vp, tables, sl, scale, "f16")
    for i, (K, V) in enumerate(logical):
        Kf = K.view(np.float16).astype(float).tolist()
        Vf = V.view(np.float16).astype(float).tolist()
        for h in range(2):
            qf = q[i, h].view(np.float16).astype(float).tolist()
            s = [scale * sum(a * b for a, b in zip(qf, Kf[p][0])) for p in range(lengths[i])]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            z = sum(e)
            o = [sum(e[p] / z * Vf[p][0][x] for p in range(lengths[i])) for x in range(4)]
            np.testing.assert_allclose(got[i, h], o, rtol=1e-13, atol=1e-15)


def test_uniform_keys_give_mean_of_values():
    """All keys equal -> every weight is 1/L -> output is the mean of V."""
    rng = np.random.default_rng(11)
    lengths = [7, 16, 40]
    hq, hkv, d, B = 4, 2, 8, 16
    q, kp, vp, tables, sl, logical = build_case(lengths, hq, hkv, d, B, "f16", rng)
    key = f16_bits(rng.standard_normal(d))
    for i, L in enumerate(lengths):
        for p in range(L):
            kp[tables[i, p // B], :, p % B, :] = key
    got = oracle.decode(q, kp, vp, tables, sl, 0.3, "f16")
    for i, (_, V) in enumerate(logical):
        mean = widen_lib(V, "f16").mean(axis=0)  # [Hkv, d]
        for h in range(hq):
            np.testing.assert_allclose(got[i, h], mean[h // 2], rtol=1e-13, atol=1e-15)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(5)
    q, kp, vp, tables, sl, logical = build_case([1, 1], 4, 4, 8, 16, "bf16", rng)
    got = oracle.decode(q, kp, vp, tables, sl, 1.0, "bf16")
    for i, (_, V) in enumerate(logical):
        assert np.array_equal(got[i], widen_lib(V[0], "bf16"))


def test_two_tokens_closed_form():
    """Two tokens: w_0 = 1 / (1 + exp(s_1 - s_0))."""
    d, B = 4, 16
    q = f16_bits(np.array([[[1.5, 0.0, 0.0, 0.0]]]))
    K = f16_bits(np.array([[[1.0, 0, 0, 0]], [[0.0, 0, 0, 0]]]))
    V = f16_bits(np.array([[[2.0, -1.0, 0.5, 4.0]], [[-6.0, 3.0, 1.0, 0.0]]]))
    tables = np.array([[1]], dtype=np.int32)
    kp = scatter_into_pool(K, [1], 2, B, 0x7E00)
    vp = scatter_into_pool(V, [1], 2, B, 0x7E00)
    scale = 0.75
    got = oracle.decode(q, kp, vp, tables, np.array([2], np.int32), scale, "f16")
    s0, s1 = scale * 1.5, 0.0
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    ref = w0 * np.array([2.0, -1.0, 0.5, 4.0]) + (1 - w0) * np.array([-6.0, 3.0, 1.0, 0.0])
    np.testing.assert_allclose(got[0, 0], ref, rtol=1e-14)


def test_gqa_head_map_is_consecutive_groups():
    """Query head h reads KV head h // G: give each KV head a constant value
    vector, so out[h] must equal the constant of KV head h // G."""
    rng = np.random.default_rng(8)
    hq, hkv, d, B = 12, 3, 8, 16
    q, kp, vp, tables, sl, logical = build_case([20], hq, hkv, d, B, "f16", rng)
    consts = [f16_bits(np.full(d, c)) for c in (1.25, -3.5, 7.0)]
    for p in range(20):
        for kv in range(hkv):
            vp[tables[0, p // B], kv, p % B, :] = consts[kv]
    got = oracle.decode(q, kp, vp, tables, sl, 0.2, "f16")
    for h in range(hq):
        np.testing.assert_allclose(got[0, h], widen_lib(consts[h // 4], "f16"), rtol=1e-14)


def test_stale_slots_never_read():
    """NaN in every slot past L (last block tail, unreferenced blocks) leaves
    the result finite and equal to the contiguous one."""
    rng = np.random.default_rng(9)
    lengths = [3, 18, 31]
    q, kp, vp, tables, sl, logical = build_case(lengths, 4, 2, 16, 16, "bf16", rng)
    got = oracle.decode(q, kp, vp, tables, sl, 0.25, "bf16")
    assert np.isfinite(got).all()
    for i, (K, V) in enumerate(logical):
        ref = contiguous_attention(widen_lib(q[i], "bf16"), widen_lib(K, "bf16"),
                                   widen_lib(V, "bf16"), 0.25)
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-13)


def test_zero_length_gives_zeros():
    rng = np.random.default_rng(1)
    q, kp, vp, tables, sl, _ = build_case([0, 4], 2, 1, 8, 4, "f16", rng)
    got = oracle.decode(q, kp, vp, tables, sl, 1.0, "f16")
    assert np.array_equal(got[0], np.zeros((2, 8)))


def test_subset_leaves_other_rows_nan():
    rng = np.random.default_rng(2)
    q, kp, vp, tables, sl, _ = build_case([5, 6, 7], 2, 1, 8, 4, "f16", rng)
    full = oracle.decode(q, kp, vp, tables, sl, 1.0, "f16")
    sub = oracle.decode(q, kp, vp, tables, sl, 1.0, "f16", seqs=[2])
    assert np.isnan(sub[:2]).all()
    assert np.array_equal(sub[2], full[2])


# ----------------------------------------------------------------- split-KV
@pytest.mark.parametrize("partition", [4, 16, 32, 512])
def test_partitions_then_reduce_equals_single_pass(partition):
    rng = np.random.default_rng(partition)
    lengths = [1, 16, 47, 100, 0]
    hq, hkv, d, B = 4, 2, 16, 4
    q, kp, vp, tables, sl, _ = build_case(lengths, hq, hkv, d, B, "f16", rng)
    npart = max(1, -(-max(lengths) // partition))
    m, l, o = oracle.partitions(q, kp, vp, tables, sl, 0.25, "f16", partition, npart)
    got = oracle.reduce(m, l, o)
    ref = oracle.decode(q, kp, vp, tables, sl, 0.25, "f16")
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    # partitions past the end are empty
    for i, L in enumerate(lengths):
        for k in range(npart):
            if k * partition >= L:
                assert m[i, :, k].tolist() == [-math.inf] * hq and (l[i, :, k] == 0).all()


def test_partition_values_uniform_keys():
    """Identical keys: every partition has m_k = s, l_k = (tokens in it)."""
    B, d, P = 4, 8, 8
    rng = np.random.default_rng(4)
    q, kp, vp, tables, sl, logical = build_case([21], 1, 1, d, B, "f16", rng)
    key = f16_bits(rng.standard_normal(d))
    for p in range(21):
        kp[tables[0, p // B], 0, p % B, :] = key
    m, l, o = oracle.partitions(q, kp, vp, tables, sl, 0.5, "f16", P, 3)
    s = 0.5 * float(widen_lib(q[0, 0], "f16") @ widen_lib(key, "f16"))
    np.testing.assert_allclose(m[0, 0], [s, s, s], rtol=1e-15)
    np.testing.assert_allclose(l[0, 0], [8, 8, 5], rtol=1e-15)
    V = widen_lib(logical[0][1], "f16")[:, 0, :]
    np.testing.assert_allclose(o[0, 0, 2], V[16:21].mean(axis=0), rtol=1e-13)


def test_reduce_closed_form():
    """Two partials with m = (0, ln 2), l = (1, 1):
    weights l_k exp(m_k - m) = (1/2, 1), l = 3/2."""
    m = np.array([[0.0, math.log(2.0)]])
    l = np.array([[1.0, 1.0]])
    a = np.array([1.0, -2.0, 3.0])
    b = np.array([4.0, 0.5, -1.0])
    o = np.stack([a, b])[None]
    got = oracle.reduce(m, l, o)
    np.testing.assert_allclose(got[0], (0.5 * a + b) / 1.5, rtol=1e-15)
    # an empty partial (m = -inf) is skipped
    m2 = np.array([[0.0, -math.inf]])
    o2 = np.stack([a, np.full(3, np.nan)])[None]
    np.testing.assert_allclose(oracle.reduce(m2, np.array([[2.0, 0.0]]), o2)[0], a)


# ---------------------------------------------------------- cache writes
def test_cache_write_and_copy_blocks_readback():
    B, hkv, d = 4, 2, 8
    rng = np.random.default_rng(6)
    kp = rng.integers(0, 65535, (6, hkv, B, d), dtype=np.uint16)
    vp = rng.integers(0, 65535, (6, hkv, B, d), dtype=np.uint16)
    before_k, before_v = kp.copy(), vp.copy()
    kn = rng.integers(0, 65535, (3, hkv, d), dtype=np.uint16)
    vn = rng.integers(0, 65535, (3, hkv, d), dtype=np.uint16)
    slots = np.array([9, -1, 22])
    oracle.cache_write(kp, vp, kn, vn, slots)
    assert np.array_equal(kp[2, :, 1, :], kn[0]) and np.array_equal(vp[5, :, 2, :], vn[2])
    changed = np.argwhere((kp != before_k).any(axis=(1, 3)))
    assert {tuple(x) for x in changed.tolist()} <= {(2, 1), (5, 2)}
    oracle.copy_blocks([kp, vp], [(2, 0), (0, 3)])
    assert np.array_equal(kp[0], kp[2]) and np.array_equal(kp[3], kp[2])
    assert np.array_equal(vp[3], vp[2])
    assert np.array_equal(kp[1], before_k[1]) and np.array_equal(kp[4], before_k[4])


# ------------------------------------------------------------- closed forms
def test_kv_bytes_closed_forms(golden_dir):
    g = read_json(os.path.join(golden_dir, "kv_sizes.json"))
    for c in g["per_token"]:
        assert oracle.kv_bytes_per_token(c["n_layers"], c["n_kv_heads"], c["head_dim"],
                                         c["bytes_per_elem"]) == c["bytes"], c["source"]
    for c in g["per_request"]:
        per = oracle.kv_bytes_per_token(c["n_layers"], c["n_kv_heads"], c["head_dim"],
                                        c["bytes_per_elem"])
        assert per * c["tokens"] == c["bytes"], c["source"]
    for c in g["per_block_per_layer"]:
        assert oracle.kv_bytes_per_token(1, c["n_kv_heads"], c["head_dim"],
                                         c["bytes_per_elem"]) * c["block_size"] == c["bytes"]


def test_address_translation(golden_dir):
    g = read_json(os.path.join(golden_dir, "address_translation.json"))
    for c in g["cases"]:
        j, o, phys = oracle.translate(c["table"], c["t"], c["block_size"])
        assert (j, o, phys) == (c["j"], c["o"], c["phys"]), c["source"]
        assert oracle.slot_of(c["table"], c["t"], c["block_size"]) == phys * c["block_size"] + o
    for c in g["blocks_needed"]:
        model = oracle.allocator.BlockAllocatorModel(c["blocks"] + 2, c["block_size"])
        model.add("r")
        model.append("r", c["tokens"])
        assert len(model.table("r")) == c["blocks"], c["source"]
        assert c["tokens"] - (c["blocks"] - 1) * c["block_size"] == c["last_block_fill"]
