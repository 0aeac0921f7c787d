"""Plain, slow, obviously correct CPU oracle for the paged decode hot path.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference legs may import this package.  It shares no code with
the CUDA library (paged_kv_cache_64_gb300/csrc) and imports nothing from it.

Contents, each following the pages' definitions (page title, section):

* decode / partitions / reduce: fp64 C loops in pa_oracle.c (see the header
  there): the gather through the block table, softmax(scale * q K^T) V, and
  the split-KV partial + combine formula of "PagedAttention and Virtual Memory
  Management ..." (llms.blog) section 4, "Parallel Partitioning Across GPU
  Warps", step 3.
* cache_write: each new token's key and value vectors land in slot
  (slot // B, slot % B) of the pool ("Why AI servers waste memory, and how
  paging fixes it" (spicyshark.co), "The real implementation", the append
  step; llms.blog section 5 case 1; "2.1 PagedAttention" (infra-guide)
  section 5, physical_block_number / physical_block_offset).
* copy_blocks: the whole source block is copied onto the destination block
  (spicyshark.co, "The real implementation": the copy-on-write branch copies
  the whole block).  The llms.blog page (section 5) copies only the first o
  token vectors; copying the whole block is the reading taken: bytes past o
  are never read.
* translate / slot_of: logical block j = t // B, offset o = t % B, physical
  block T[j] (llms.blog section 3).
* kv_bytes_per_token: 2 * N_L * N_KV * d_h * b (llms.blog section 1;
  spicyshark.co "How big it gets").
* allocator.BlockAllocatorModel: the block manager semantics of the
  spicyshark.co page (free list, refcounts, fork, copy-on-write append).

Arrays of 16-bit elements are passed as numpy uint16 bit patterns; dtype is
"f16" or "bf16".
"""
import ctypes

import numpy as np

from . import allocator  # noqa: F401  (re-exported)
from . import build as _build

_DT = {"f16": 0, "bf16": 1}
_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if _build.is_stale():
        _build.build()
    lib = ctypes.CDLL(_build.LIB)
    dp = ctypes.POINTER(ctypes.c_double)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.pa_oracle_decode.restype = ctypes.c_int
    lib.pa_oracle_decode.argtypes = [dp, u16p, u16p, u16p, ctypes.c_int, i32p, ctypes.c_int, i32p,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, i32p, ctypes.c_int]
    lib.pa_oracle_partitions.restype = ctypes.c_int
    lib.pa_oracle_partitions.argtypes = [dp, dp, dp, u16p, u16p, u16p, ctypes.c_int, i32p,
                                         ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                         ctypes.c_int, ctypes.c_int]
    lib.pa_oracle_reduce.restype = None
    lib.pa_oracle_reduce.argtypes = [dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int, ctypes.c_int]
    lib.pa_oracle_widen.restype = None
    lib.pa_oracle_widen.argtypes = [dp, u16p, ctypes.c_int64, ctypes.c_int]
    u8p = ctypes.POINTER(ctypes.c_uint8)
    fp = ctypes.POINTER(ctypes.c_float)
    lib.pa_oracle_decode_fp8.restype = ctypes.c_int
    lib.pa_oracle_decode_fp8.argtypes = [dp, u16p, u8p, u8p, ctypes.c_int, ctypes.c_double,
                                         ctypes.c_double, i32p, ctypes.c_int, i32p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_double, i32p, ctypes.c_int]
    lib.pa_oracle_e4m3_decode.restype = None
    lib.pa_oracle_e4m3_decode.argtypes = [dp, u8p, ctypes.c_int64]
    lib.pa_oracle_e4m3_encode.restype = None
    lib.pa_oracle_e4m3_encode.argtypes = [u8p, fp, ctypes.c_int64]
    lib.pa_oracle_num_threads.restype = ctypes.c_int
    lib.pa_oracle_set_num_threads.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("16-bit element arrays must be passed as uint16 bit patterns")
    return a


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def num_threads():
    return _load().pa_oracle_num_threads()


def set_num_threads(n):
    _load().pa_oracle_set_num_threads(int(n))


def widen(bits, dtype):
    """Exact widening of f16 / bf16 bit patterns to float64."""
    bits = _u16(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().pa_oracle_widen(_ptr(out, ctypes.c_double), _ptr(bits, ctypes.c_uint16), bits.size,
                            _DT[dtype])
    return out


def decode(q, k_pool, v_pool, block_tables, seq_lens, scale, dtype, seqs=None):
    """Paged decode attention in fp64.

    q [S, Hq, d], pools [NB, Hkv, B, d] (uint16 bit patterns), block_tables
    int32 [S, max_blocks], seq_lens int32 [S].  Returns float64 [S, Hq, d];
    rows of sequences not in `seqs` (when given) are NaN.
    """
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, d = q.shape
    _, Hkv, B, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape and bt.shape[0] == S and sl.shape == (S,)
    out = np.full((S, Hq, d), np.nan)
    sub = None if seqs is None else _i32(seqs)
    rc = _load().pa_oracle_decode(
        _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(k_pool, ctypes.c_uint16),
        _ptr(v_pool, ctypes.c_uint16), _DT[dtype], _ptr(bt, ctypes.c_int32), bt.shape[1],
        _ptr(sl, ctypes.c_int32), S, Hq, Hkv, d, B, float(scale),
        None if sub is None else _ptr(sub, ctypes.c_int32), 0 if sub is None else sub.size)
    if rc:
        raise ValueError("oracle decode: bad dimensions")
    return out


def partitions(q, k_pool, v_pool, block_tables, seq_lens, scale, dtype, partition_tokens,
               max_partitions):
    """Split-KV partials: (m, l, o) with shapes [S, Hq, NP], [S, Hq, NP], [S, Hq, NP, d]."""
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, d = q.shape
    _, Hkv, B, _ = k_pool.shape
    m = np.empty((S, Hq, max_partitions))
    l = np.empty((S, Hq, max_partitions))
    o = np.empty((S, Hq, max_partitions, d))
    rc = _load().pa_oracle_partitions(
        _ptr(m, ctypes.c_double), _ptr(l, ctypes.c_double), _ptr(o, ctypes.c_double),
        _ptr(q, ctypes.c_uint16), _ptr(k_pool, ctypes.c_uint16), _ptr(v_pool, ctypes.c_uint16),
        _DT[dtype], _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), S, Hq, Hkv,
        d, B, float(scale), int(partition_tokens), int(max_partitions))
    if rc:
        raise ValueError("oracle partitions: bad arguments")
    return m, l, o


def reduce(m, l, o):
    """Cross-partition combine of partials shaped [..., NP] and [..., NP, d]."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    lead = m.shape[:-1]
    npart = m.shape[-1]
    d = o.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (d,))
    _load().pa_oracle_reduce(_ptr(out, ctypes.c_double), _ptr(m, ctypes.c_double),
                             _ptr(l, ctypes.c_double), _ptr(o, ctypes.c_double), rows, npart, d)
    return out


def translate(table, t, block_size):
    """Token position t -> (logical block j, offset o, physical block T[j])."""
    j = t // block_size
    o = t % block_size
    return j, o, int(table[j])


def slot_of(table, t, block_size):
    """Flat slot index (physical block * B + offset) of position t."""
    j, o, phys = translate(table, t, block_size)
    return phys * block_size + o


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, bytes_per_elem):
    """KV-cache bytes one token occupies: one key and one value vector per
    layer and KV head."""
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def cache_write(k_pool, v_pool, k_new, v_new, slot_mapping):
    """Write token t's K/V ([T, Hkv, d]) into slot slot_mapping[t] of the
    pools ([NB, Hkv, B, d]), in place.  A negative slot means "skip"."""
    B = k_pool.shape[2]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = slot // B, slot % B
        k_pool[blk, :, off, :] = k_new[t]
        v_pool[blk, :, off, :] = v_new[t]


def copy_blocks(pools, block_mapping):
    """For each (src, dst) pair, in order, copy block src onto block dst in
    every pool of the list (all layers' K and V pools), in place."""
    for src, dst in np.asarray(block_mapping).reshape(-1, 2).tolist():
        for pool in pools:
            pool[dst] = pool[src]


# ----------------------------------------------------------------- FP8 variant
def e4m3_decode(codes):
    """Values (float64) of OCP E4M3 codes (uint8)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().pa_oracle_e4m3_decode(_ptr(out, ctypes.c_double), _ptr(c, ctypes.c_uint8), c.size)
    return out


def e4m3_encode(values):
    """Nearest E4M3 codes (ties to even, saturating at +-448) of fp32 values."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().pa_oracle_e4m3_encode(_ptr(out, ctypes.c_uint8), _ptr(v, ctypes.c_float), v.size)
    return out


def quantize_fp8(bits, dtype, scale):
    """E4M3 codes of 16-bit values (bit patterns) under a pool scale: the fp32
    value times fl32(1 / scale), rounded to the nearest code."""
    x = widen(bits, dtype).astype(np.float32)  # exact: every 16-bit value is an fp32 value
    inv = np.float32(1.0) / np.float32(scale)
    return e4m3_encode(x * inv)


def cache_write_fp8(k_pool, v_pool, k_new, v_new, slot_mapping, dtype, k_scale, v_scale):
    """cache_write into E4M3 pools (uint8 [NB, Hkv, B, d]): token t's K/V
    (16-bit bit patterns [T, Hkv, d]) quantized with the pools' scales."""
    cache_write(k_pool, v_pool, quantize_fp8(k_new, dtype, k_scale),
                quantize_fp8(v_new, dtype, v_scale), slot_mapping)


def decode_fp8(q, k_pool, v_pool, block_tables, seq_lens, scale, dtype, k_scale, v_scale,
               seqs=None):
    """Paged decode attention in fp64 over E4M3 pools (uint8 codes): K element
    = k_scale * code value, V element = v_scale * code value.  q (16-bit bit
    patterns of `dtype`) as in decode()."""
    q = _u16(q)
    k_pool = np.ascontiguousarray(k_pool, dtype=np.uint8)
    v_pool = np.ascontiguousarray(v_pool, dtype=np.uint8)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, d = q.shape
    _, Hkv, B, d2 = k_pool.shape
    assert d2 == d and v_pool.shape == k_pool.shape and bt.shape[0] == S and sl.shape == (S,)
    out = np.full((S, Hq, d), np.nan)
    sub = None if seqs is None else _i32(seqs)
    rc = _load().pa_oracle_decode_fp8(
        _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(k_pool, ctypes.c_uint8),
        _ptr(v_pool, ctypes.c_uint8), _DT[dtype], float(k_scale), float(v_scale),
        _ptr(bt, ctypes.c_int32), bt.shape[1], _ptr(sl, ctypes.c_int32), S, Hq, Hkv, d, B,
        float(scale), None if sub is None else _ptr(sub, ctypes.c_int32),
        0 if sub is None else sub.size)
    if rc:
        raise ValueError("oracle decode: bad dimensions")
    return out
