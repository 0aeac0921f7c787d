"""Pins of the oracle's FP8 (OCP E4M3) KV-cache variant, no GPU: the format's
fixed points, brute-force nearest-code rounding, and the FP8 decode reduced to
the already-pinned 16-bit decode on values both formats hold exactly."""
import numpy as np
import pytest

import oracle


def test_e4m3_fixed_points():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x7E] == 448.0                      # largest finite
    assert v[0x08] == 2.0**-6                    # smallest normal
    assert v[0x01] == 2.0**-9                    # smallest subnormal
    assert v[0x07] == 7 * 2.0**-9                # largest subnormal
    assert v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.isnan(v).sum() == 2                # no infinities, one NaN per sign
    fin = v[~np.isnan(v)]
    assert np.isfinite(fin).all()
    assert len(set(fin.tolist())) == 253         # 254 finite codes, +0 and -0 equal


def test_e4m3_round_trip_all_codes():
    c = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(c)
    fin = ~np.isnan(v)
    assert np.array_equal(oracle.e4m3_encode(v[fin].astype(np.float32)), c[fin])


def brute_force_code(y):
    """Nearest finite E4M3 code by exhaustive search; ties to the even code
    (mantissa bit 0 clear), saturating beyond 448."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    ok = ~np.isnan(vals)
    codes, vals = codes[ok], vals[ok]
    sign = np.signbit(y)
    a = min(abs(float(y)), 448.0)
    pos = vals >= 0
    c, v = codes[pos & ~np.signbit(vals)], vals[pos & ~np.signbit(vals)]
    d = np.abs(v - a)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:
        best = [b for b in best if (c[b] & 1) == 0]
    code = int(c[best[0]])
    return code | (0x80 if sign else 0)


def test_e4m3_encode_matches_brute_force():
    rng = np.random.default_rng(3)
    ys = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.uniform(-4, 2.8, 3000),
        # every midpoint between consecutive positive codes, and just beside it
        (lambda v: (v[1:] + v[:-1]) / 2)(np.sort(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)))),
        [448.0, 460.0, 464.0, 500.0, 1e6, -1e6, 2.0**-10, 2.0**-11, 3 * 2.0**-11],
    ]).astype(np.float32)
    got = oracle.e4m3_encode(ys)
    for y, g in zip(ys.tolist(), got.tolist()):
        assert g == brute_force_code(np.float32(y)), (y, g)


def test_e4m3_error_bound_and_monotone():
    rng = np.random.default_rng(4)
    y = np.sort(rng.uniform(2.0**-6, 440.0, 20000).astype(np.float32))
    q = oracle.e4m3_decode(oracle.e4m3_encode(y))
    assert (np.abs(q - y) <= 2.0**-4 * y).all()  # half a spacing of 2^-3 relative
    assert (np.diff(q) >= 0).all()


def test_quantize_uses_fp32_product():
    # the product is taken in fp32: x * fl32(1/3) rounds before the code does
    x = np.array([0x3F80, 0x4040], dtype=np.uint16)  # bf16 1.0, 3.0
    got = oracle.quantize_fp8(x, "bf16", 3.0)
    inv = np.float32(1.0) / np.float32(3.0)
    want = oracle.e4m3_encode(np.array([1.0, 3.0], np.float32) * inv)
    assert np.array_equal(got, want)
    assert oracle.e4m3_decode(got)[1] == 1.0       # 3 * fl32(1/3) rounds to 1


def test_cache_write_fp8_read_back():
    """The quantising cache write puts token t's K codes (K scale) and V codes
    (V scale) at (slot // B, head, slot % B); a negative slot writes nothing;
    every other byte of the pools is untouched.  Read back through the E4M3
    definition: |code value * scale - x| stays within half an E4M3 step."""
    rng = np.random.default_rng(9)
    NB, H, B, d, T = 6, 2, 16, 64, 5
    kp = rng.integers(0, 0x7f, (NB, H, B, d), dtype=np.uint8)
    vp = rng.integers(0, 0x7f, (NB, H, B, d), dtype=np.uint8)
    k0, v0 = kp.copy(), vp.copy()
    xk = rng.normal(0, 1, (T, H, d)).astype(np.float32)
    xv = rng.normal(0, 3, (T, H, d)).astype(np.float32)
    bf = lambda x: (x.view(np.uint32) >> 16).astype(np.uint16)  # truncation: exact bf16 values
    kb, vb = bf(xk), bf(xv)
    slots = np.array([17, 0, -1, 95, 40], dtype=np.int64)
    ks, vs = 0.0625, 0.5
    oracle.cache_write_fp8(kp, vp, kb, vb, slots, "bf16", ks, vs)
    touched = np.zeros((NB, B), bool)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        blk, off = slot // B, slot % B
        touched[blk, off] = True
        for pool, x, sc in ((kp, oracle.widen(kb[t], "bf16"), ks), (vp, oracle.widen(vb[t], "bf16"), vs)):
            got = oracle.e4m3_decode(pool[blk, :, off, :]) * sc
            # E4M3 has 3 mantissa bits: error <= 2^-4 relative, or half the
            # subnormal step (2^-10) times the scale near zero
            assert np.all(np.abs(got - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sc))
    for pool, p0 in ((kp, k0), (vp, v0)):
        mask = np.broadcast_to(touched[:, None, :, None], pool.shape)
        assert np.array_equal(pool[~mask], p0[~mask])
    # K and V are not swapped: the V codes carry the V scale
    assert not np.array_equal(kp[1, :, 1, :], vp[1, :, 1, :])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fp8_decode_reduces_to_16bit_decode(dtype):
    """Pools whose values E4M3 and the 16-bit type both hold exactly: the FP8
    decode with a power-of-two scale equals the 16-bit decode of the scaled
    values (the 16-bit decode is pinned elsewhere)."""
    import torch
    rng = np.random.default_rng(9)
    S, Hq, Hkv, d, B, NB = 3, 4, 2, 64, 16, 12
    codes_k = rng.integers(0, 0x7F, (NB, Hkv, B, d)).astype(np.uint8)  # positive finite codes
    codes_v = rng.integers(0, 0x7F, (NB, Hkv, B, d)).astype(np.uint8)
    codes_k |= (rng.integers(0, 2, codes_k.shape) << 7).astype(np.uint8)
    codes_v |= (rng.integers(0, 2, codes_v.shape) << 7).astype(np.uint8)
    ks, vs = 2.0**-3, 2.0**2
    tdt = torch.float16 if dtype == "f16" else torch.bfloat16

    def bits16(x):
        return torch.tensor(x, dtype=torch.float64).to(tdt).view(torch.int16).numpy().view(np.uint16)

    k16 = bits16(oracle.e4m3_decode(codes_k) * ks)
    v16 = bits16(oracle.e4m3_decode(codes_v) * vs)
    assert np.array_equal(oracle.widen(k16, dtype), oracle.e4m3_decode(codes_k) * ks)  # exact
    q = bits16(rng.standard_normal((S, Hq, d)))
    tables = rng.permutation(NB)[:S * 4].reshape(S, 4).astype(np.int32)
    lens = np.array([1, 37, 64], dtype=np.int32)
    a = oracle.decode_fp8(q, codes_k, codes_v, tables, lens, 0.125, dtype, ks, vs)
    b = oracle.decode(q, k16, v16, tables, lens, 0.125, dtype)
    assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_fp8_kv_bytes_formula():
    # b = 1 for FP8 in the pages' M_KV formula: half the 16-bit bytes
    assert oracle.kv_bytes_per_token(32, 8, 128, 1) == 65536
    assert oracle.kv_bytes_per_token(24, 2, 64, 1) * 2 == oracle.kv_bytes_per_token(24, 2, 64, 2)
