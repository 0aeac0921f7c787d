"""Python binding of the C ABI (include/pa.h) for torch tensors.

Argument marshalling only: every function checks devices, dtypes, shapes and
contiguity, passes raw pointers and sizes to libpa.so, and raises on a
non-OK status.  All computation runs in the library's CUDA kernels; nothing
here computes on the host or falls back to PyTorch ops.
"""
import ctypes

import numpy as np
import torch

from . import _lib

_DTYPES = {torch.float16: _lib.PA_F16, torch.bfloat16: _lib.PA_BF16}


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t):
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported element type {t.dtype}; use float16 or bfloat16") from None


def _cuda(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def version():
    return _lib.load().pa_version()


def check_error(stream=None):
    """Synchronise the stream and raise if a kernel recorded a device error
    (PA_ERR_BAD_INDEX, PA_ERR_DEVICE_TIMEOUT)."""
    _lib.check("pa_check_error", _lib.load().pa_check_error(_stream_handle(stream)))


def selftest_wait_timeout(stream=None):
    """Launch the bounded-wait self-test kernel (see pa.h)."""
    _lib.check("pa_selftest_wait_timeout",
               _lib.load().pa_selftest_wait_timeout(_stream_handle(stream)))


def cache_write(k_new, v_new, slot_mapping, k_pool, v_pool, stream=None):
    """reshape_and_cache: k_new/v_new [T, Hkv, d] into pools [NB, Hkv, B, d]
    at slot_mapping (int64 [T]; slot = block * B + offset, < 0 skips)."""
    nb, hkv, bs, d = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape:
        raise ValueError("pool / new-token shapes differ")
    if k_new.dim() != 3 or k_new.shape[1:] != (hkv, d):
        raise ValueError(f"k_new must be [T, {hkv}, {d}], got {tuple(k_new.shape)}")
    T = k_new.shape[0]
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [T]")
    for t in (k_new, v_new, v_pool):
        if t.dtype != k_pool.dtype:
            raise TypeError("element types differ")
    rc = _lib.load().pa_cache_write(
        _cuda(k_new, "k_new"), _cuda(v_new, "v_new"),
        _cuda(slot_mapping, "slot_mapping", torch.int64), T,
        _cuda(k_pool, "k_pool", ndim=4), _cuda(v_pool, "v_pool", ndim=4), nb, hkv, d, bs,
        _dt(k_pool), _stream_handle(stream))
    _lib.check("pa_cache_write", rc)


def copy_blocks(k_pools, v_pools, block_mapping, stream=None):
    """Copy-on-write block copies: for each (src, dst) row of block_mapping
    (int64 [n, 2], CUDA), pool[dst] = pool[src] in every layer's K and V
    pool."""
    if len(k_pools) != len(v_pools) or not k_pools:
        raise ValueError("need the same non-zero number of K and V pools")
    shape, dtype = k_pools[0].shape, k_pools[0].dtype
    for t in list(k_pools) + list(v_pools):
        if t.shape != shape or t.dtype != dtype:
            raise ValueError("all pools must share shape and dtype")
    n = 0 if block_mapping.numel() == 0 else block_mapping.shape[0]
    if block_mapping.numel() and (block_mapping.dim() != 2 or block_mapping.shape[1] != 2):
        raise ValueError("block_mapping must be [n, 2]")
    L = len(k_pools)
    kp = (ctypes.c_void_p * L)(*[_cuda(t, "k_pool").value for t in k_pools])
    vp = (ctypes.c_void_p * L)(*[_cuda(t, "v_pool").value for t in v_pools])
    block_bytes = int(np.prod(shape[1:])) * k_pools[0].element_size()
    mp = _cuda(block_mapping, "block_mapping", torch.int64) if n else ctypes.c_void_p(0)
    rc = _lib.load().pa_copy_blocks(kp, vp, L, mp, n, shape[0], block_bytes,
                                    _stream_handle(stream))
    _lib.check("pa_copy_blocks", rc)


def _decode_dims(q, k_pool, block_tables, seq_lens):
    S, hq, d = q.shape
    nb, hkv, bs, d2 = k_pool.shape
    if d2 != d:
        raise ValueError("head_dim of q and pools differ")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], seq_lens [S]")
    return S, hq, hkv, d, nb, bs


def auto_partition(num_seqs, num_kv_heads, max_seq_len, head_dim, block_size, group, dtype,
                   fp8=False):
    """Partition size decode (fp8=False) or decode_fp8 (fp8=True) uses for
    partition_tokens=0; -1 for single pass."""
    fn = _lib.load().pa_decode_fp8_auto_partition if fp8 else _lib.load().pa_decode_auto_partition
    return fn(num_seqs, num_kv_heads, max_seq_len, head_dim, block_size, group, _DTYPES[dtype])


def partial_tokens(num_seqs, num_kv_heads, max_seq_len, head_dim, block_size, group, dtype,
                   partition_tokens=0, fp8=False):
    """Positions each split-KV partial of decode (or decode_fp8) covers: the
    partition size times the partitions one CTA merges; -1 for single pass."""
    return _lib.load().pa_decode_partial_tokens(num_seqs, num_kv_heads, max_seq_len, head_dim,
                                                block_size, group, int(partition_tokens),
                                                _DTYPES[dtype], int(bool(fp8)))


DECODE_IMPLS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2}


def set_decode_impl(name):
    """Select the decode kernel for later calls ("auto", "cuda_cores",
    "tensor_cores"); returns the previous name."""
    prev = _lib.load().pa_set_decode_impl(DECODE_IMPLS[name])
    if prev < 0:
        raise ValueError(name)
    return {v: k for k, v in DECODE_IMPLS.items()}[prev]


def get_decode_impl():
    return {v: k for k, v in DECODE_IMPLS.items()}[_lib.load().pa_get_decode_impl()]


def set_decode_span(span):
    """Split-KV partitions per tensor-core CTA for later calls (0 = automatic);
    returns the previous setting."""
    prev = _lib.load().pa_set_decode_span(int(span))
    if prev < 0:
        raise ValueError(span)
    return prev


def ctas_per_sm(head_dim, group, dtype):
    return _lib.load().pa_decode_ctas_per_sm(head_dim, group, _DTYPES[dtype])


def workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                   partition_tokens, dtype):
    return _lib.load().pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                block_size, max_seq_len, partition_tokens,
                                                _DTYPES[dtype])


def alloc_workspace(nbytes, device):
    """Device scratch for split-KV (256-byte aligned by the caching allocator)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def decode(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale,
           partition_tokens=0, workspace=None, stream=None):
    """Paged decode attention into out [S, Hq, d].  partition_tokens: -1
    single pass, 0 automatic, >0 split-KV partition size.  workspace: a
    device buffer of at least workspace_size(...) bytes (alloc_workspace);
    when it is missing or too small one is allocated here, so a decode loop
    passes its own.  Returns the workspace used."""
    S, hq, hkv, d, nb, bs = _decode_dims(q, k_pool, block_tables, seq_lens)
    if out.shape != q.shape or out.dtype != q.dtype or k_pool.dtype != q.dtype:
        raise ValueError("out/q/pool shapes or types differ")
    need = workspace_size(S, hq, hkv, d, bs, max_seq_len, partition_tokens, q.dtype)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = alloc_workspace(need, q.device)
    ws = _cuda(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.load().pa_decode(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_pool, "k_pool"), _cuda(v_pool, "v_pool"), nb,
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq, hkv, d, bs,
        float(scale), int(partition_tokens), ws, wbytes, _dt(q), _stream_handle(stream))
    _lib.check("pa_decode", rc)
    return workspace


def decode_step(out, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_tables, seq_lens,
                max_seq_len, scale, partition_tokens=0, workspace=None, stream=None):
    """One fused decode step: write each sequence's newest token (k_new /
    v_new [S, Hkv, d] at slot_mapping [S], the slot of position seq_lens-1)
    and attend over seq_lens positions, in one launch.  workspace as for
    decode."""
    S, hq, hkv, d, nb, bs = _decode_dims(q, k_pool, block_tables, seq_lens)
    if out.shape != q.shape or out.dtype != q.dtype or k_pool.dtype != q.dtype:
        raise ValueError("out/q/pool shapes or types differ")
    if k_new.shape != (S, hkv, d) or v_new.shape != k_new.shape or slot_mapping.shape != (S,):
        raise ValueError("k_new/v_new must be [S, Hkv, d] and slot_mapping [S]")
    need = workspace_size(S, hq, hkv, d, bs, max_seq_len, partition_tokens, q.dtype)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = alloc_workspace(need, q.device)
    ws = _cuda(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _lib.load().pa_decode_step(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_new, "k_new"), _cuda(v_new, "v_new"),
        _cuda(slot_mapping, "slot_mapping", torch.int64), _cuda(k_pool, "k_pool"),
        _cuda(v_pool, "v_pool"), nb, _cuda(block_tables, "block_tables", torch.int32),
        block_tables.shape[1], _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq,
        hkv, d, bs, float(scale), int(partition_tokens), ws, wbytes, _dt(q),
        _stream_handle(stream))
    _lib.check("pa_decode_step", rc)
    return workspace


def shared_prefix_len(block_tables, seq_lens, block_size):
    """Longest whole-block prefix that every sequence reaches through the
    same block-table entries (host arrays), capped by the shortest sequence:
    the prefix_len decode_cascade can be given for this batch
    (pa_shared_prefix_len)."""
    t = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if t.ndim != 2 or lens.shape != (t.shape[0],):
        raise ValueError("block_tables must be [S, max_blocks], seq_lens [S]")
    out = ctypes.c_int(0)
    rc = _lib.load().pa_shared_prefix_len(
        t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), t.shape[1],
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), t.shape[0], int(block_size),
        ctypes.byref(out))
    _lib.check("pa_shared_prefix_len", rc)
    return out.value


def cache_write_fp8(k_new, v_new, slot_mapping, k_pool, v_pool, k_scale, v_scale, stream=None):
    """reshape_and_cache into E4M3 pools (uint8 [NB, Hkv, B, d]): k_new /
    v_new (16-bit [T, Hkv, d]) quantised with the pools' scales."""
    nb, hkv, bs, d = k_pool.shape
    T = k_new.shape[0]
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8:
        raise ValueError("E4M3 pools are uint8 tensors of codes")
    if k_new.shape != (T, hkv, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [T, Hkv, d]")
    rc = _lib.load().pa_cache_write_fp8(
        _cuda(k_new, "k_new"), _cuda(v_new, "v_new"),
        _cuda(slot_mapping, "slot_mapping", torch.int64), T, _cuda(k_pool, "k_pool"),
        _cuda(v_pool, "v_pool"), nb, hkv, d, bs, float(k_scale), float(v_scale), _dt(k_new),
        _stream_handle(stream))
    _lib.check("pa_cache_write_fp8", rc)


def fp8_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_seq_len,
                       partition_tokens, dtype):
    return _lib.load().pa_decode_fp8_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                    head_dim, block_size, max_seq_len,
                                                    partition_tokens, _DTYPES[dtype])


def decode_fp8(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale, k_scale,
               v_scale, partition_tokens=0, k_new=None, v_new=None, slot_mapping=None,
               workspace=None, stream=None):
    """Paged decode over E4M3 pools (uint8 codes, element = scale * code);
    q / out 16-bit.  With k_new / v_new / slot_mapping, each sequence's newest
    token is quantised and written first (the fused step)."""
    S, hq, d = q.shape
    nb, hkv, bs, d2 = k_pool.shape
    if d2 != d or block_tables.dim() != 2 or block_tables.shape[0] != S or seq_lens.shape != (S,):
        raise ValueError("shapes of q, pools, block_tables, seq_lens disagree")
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    if k_pool.dtype != torch.uint8 or v_pool.dtype != torch.uint8:
        raise ValueError("E4M3 pools are uint8 tensors of codes")
    step = k_new is not None
    if step and (k_new.shape != (S, hkv, d) or v_new is None or v_new.shape != k_new.shape
                 or slot_mapping is None or slot_mapping.shape != (S,)):
        raise ValueError("k_new/v_new must be [S, Hkv, d] and slot_mapping [S]")
    need = fp8_workspace_size(S, hq, hkv, d, bs, max_seq_len, partition_tokens, q.dtype)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = alloc_workspace(need, q.device)
    ws = _cuda(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    null = ctypes.c_void_p(0)
    rc = _lib.load().pa_decode_fp8(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_new, "k_new") if step else null,
        _cuda(v_new, "v_new") if step else null,
        _cuda(slot_mapping, "slot_mapping", torch.int64) if step else null,
        _cuda(k_pool, "k_pool"), _cuda(v_pool, "v_pool"), nb,
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq, hkv, d, bs,
        float(scale), float(k_scale), float(v_scale), int(partition_tokens), ws, wbytes, _dt(q),
        _stream_handle(stream))
    _lib.check("pa_decode_fp8", rc)
    return workspace


def cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_seq_len, prefix_len, dtype):
    return _lib.load().pa_decode_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                        head_dim, block_size, max_seq_len,
                                                        prefix_len, _DTYPES[dtype])


def decode_cascade(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale,
                   prefix_len, k_new=None, v_new=None, slot_mapping=None, workspace=None,
                   stream=None):
    """Decode of a batch whose sequences share their first prefix_len
    positions (the same first prefix_len / block_size block-table entries):
    the prefix is attended once per KV head for every sequence's queries,
    each tail separately, and the two merged.  With k_new / v_new /
    slot_mapping, each sequence's newest token is written first, as in
    decode_step."""
    S, hq, hkv, d, nb, bs = _decode_dims(q, k_pool, block_tables, seq_lens)
    if out.shape != q.shape or out.dtype != q.dtype or k_pool.dtype != q.dtype:
        raise ValueError("out/q/pool shapes or types differ")
    step = k_new is not None
    if step and (k_new.shape != (S, hkv, d) or v_new is None or v_new.shape != k_new.shape
                 or slot_mapping is None or slot_mapping.shape != (S,)):
        raise ValueError("k_new/v_new must be [S, Hkv, d] and slot_mapping [S]")
    need = cascade_workspace_size(S, hq, hkv, d, bs, max_seq_len, prefix_len, q.dtype)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = alloc_workspace(need, q.device)
    ws = _cuda(workspace, "workspace") if workspace is not None else ctypes.c_void_p(0)
    wbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    null = ctypes.c_void_p(0)
    rc = _lib.load().pa_decode_cascade(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_new, "k_new") if step else null,
        _cuda(v_new, "v_new") if step else null,
        _cuda(slot_mapping, "slot_mapping", torch.int64) if step else null,
        _cuda(k_pool, "k_pool"), _cuda(v_pool, "v_pool"), nb,
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq, hkv, d, bs,
        float(scale), int(prefix_len), ws, wbytes, _dt(q), _stream_handle(stream))
    _lib.check("pa_decode_cascade", rc)
    return workspace


def decode_static_scratch(out, q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale,
                          partition_tokens=0, stream=None):
    """Same result as decode(), for callers that cannot allocate device
    memory: split-KV partials go to the library's fixed device array
    (_lib.STATIC_SCRATCH_BYTES per GPU) instead of a workspace.  Raises
    PagedAttentionError (PA_ERR_TOO_LARGE) when they would not fit; calls on
    one device share that array, so they must not overlap on the GPU."""
    S, hq, hkv, d, nb, bs = _decode_dims(q, k_pool, block_tables, seq_lens)
    if out.shape != q.shape or out.dtype != q.dtype or k_pool.dtype != q.dtype:
        raise ValueError("out/q/pool shapes or types differ")
    rc = _lib.load().pa_decode_static_scratch(
        _cuda(out, "out"), _cuda(q, "q"), _cuda(k_pool, "k_pool"), _cuda(v_pool, "v_pool"), nb,
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq, hkv, d, bs,
        float(scale), int(partition_tokens), _dt(q), _stream_handle(stream))
    _lib.check("pa_decode_static_scratch", rc)


def partition_count(max_seq_len, partition_tokens):
    return max(1, -(-int(max_seq_len) // int(partition_tokens)))


def partials_view(workspace, num_seqs, num_q_heads, head_dim, max_seq_len, partition_tokens):
    """Views (m, l, O) of the partials in a workspace, per the layout in pa.h."""
    NP = partition_count(max_seq_len, partition_tokens)
    rows = num_seqs * num_q_heads * NP
    a = lambda x: (x + 255) // 256 * 256
    m_off, l_off = 0, a(rows * 4)
    o_off = l_off + a(rows * 4)
    f = workspace.view(torch.uint8)
    m = f[m_off:m_off + rows * 4].view(torch.float32).view(num_seqs, num_q_heads, NP)
    l = f[l_off:l_off + rows * 4].view(torch.float32).view(num_seqs, num_q_heads, NP)
    o = f[o_off:o_off + rows * head_dim * 4].view(torch.float32).view(
        num_seqs, num_q_heads, NP, head_dim)
    return m, l, o


def decode_partitions(q, k_pool, v_pool, block_tables, seq_lens, max_seq_len, scale,
                      partition_tokens, workspace, stream=None):
    """Split-KV step 2 only: partials into the workspace."""
    S, hq, hkv, d, nb, bs = _decode_dims(q, k_pool, block_tables, seq_lens)
    rc = _lib.load().pa_decode_partitions(
        _cuda(q, "q"), _cuda(k_pool, "k_pool"), _cuda(v_pool, "v_pool"), nb,
        _cuda(block_tables, "block_tables", torch.int32), block_tables.shape[1],
        _cuda(seq_lens, "seq_lens", torch.int32), int(max_seq_len), S, hq, hkv, d, bs,
        float(scale), int(partition_tokens), _cuda(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _dt(q), _stream_handle(stream))
    _lib.check("pa_decode_partitions", rc)


def split_kv_reduce(out, workspace, seq_lens, max_seq_len, partition_tokens, stream=None):
    """Split-KV step 3 only: combine the partials in the workspace into out."""
    S, hq, d = out.shape
    rc = _lib.load().pa_split_kv_reduce(
        _cuda(out, "out"), _cuda(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _cuda(seq_lens, "seq_lens", torch.int32),
        int(max_seq_len), S, hq, d, int(partition_tokens), _dt(out), _stream_handle(stream))
    _lib.check("pa_split_kv_reduce", rc)


class BlockAllocator:
    """Host block allocator (free list, refcounts, fork, copy-on-write)."""

    def __init__(self, num_blocks, block_size, free_order=None):
        self._lib = _lib.load()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        handle = ctypes.c_void_p()
        order = None
        if free_order is not None:
            arr = np.ascontiguousarray(free_order, dtype=np.int32)
            if arr.shape != (self.num_blocks,):
                raise ValueError("free_order must list every block once")
            order = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        _lib.check("pa_alloc_create", self._lib.pa_alloc_create(
            self.num_blocks, self.block_size, order, ctypes.byref(handle)))
        self._h = handle

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_alloc_destroy(h)
            self._h = None

    def add(self, seq):
        _lib.check("pa_seq_add", self._lib.pa_seq_add(self._h, int(seq)))

    def append(self, seq, n=1):
        """Returns (slots, copies) like the allocator model: flat slots of the
        new tokens and the (src, dst) copy-on-write pair(s)."""
        slots = np.empty(max(int(n), 1), dtype=np.int64)
        pair = np.empty(2, dtype=np.int64)
        ncow = ctypes.c_int(0)
        rc = self._lib.pa_seq_append(
            self._h, int(seq), int(n), slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            pair.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), ctypes.byref(ncow))
        _lib.check("pa_seq_append", rc)
        copies = [(int(pair[0]), int(pair[1]))] if ncow.value else []
        return slots[:int(n)].tolist(), copies

    def fork(self, parent, child):
        _lib.check("pa_seq_fork", self._lib.pa_seq_fork(self._h, int(parent), int(child)))

    def release(self, seq):
        _lib.check("pa_seq_free", self._lib.pa_seq_free(self._h, int(seq)))

    def length(self, seq):
        v = ctypes.c_int64()
        _lib.check("pa_seq_len", self._lib.pa_seq_len(self._h, int(seq), ctypes.byref(v)))
        return v.value

    def table(self, seq):
        n = ctypes.c_int()
        cap = self.num_blocks
        out = np.empty(max(cap, 1), dtype=np.int32)
        rc = self._lib.pa_seq_block_table(self._h, int(seq),
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          cap, ctypes.byref(n))
        _lib.check("pa_seq_block_table", rc)
        return out[:n.value].tolist()

    def export(self, seqs, max_blocks_per_seq):
        """Dense int32 [n, max_blocks] tables and int32 [n] lengths."""
        ids = np.ascontiguousarray(seqs, dtype=np.int64)
        tables = np.zeros((len(ids), max(int(max_blocks_per_seq), 1)), dtype=np.int32)
        lens = np.zeros(len(ids), dtype=np.int32)
        rc = self._lib.pa_alloc_export(
            self._h, ids.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(ids),
            tables.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(max_blocks_per_seq),
            lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
        _lib.check("pa_alloc_export", rc)
        return tables[:, :int(max_blocks_per_seq)], lens

    def num_free(self):
        return self._lib.pa_alloc_num_free(self._h)

    def free_list(self):
        n = ctypes.c_int()
        out = np.empty(max(self.num_blocks, 1), dtype=np.int32)
        rc = self._lib.pa_alloc_free_list(self._h,
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                          self.num_blocks, ctypes.byref(n))
        _lib.check("pa_alloc_free_list", rc)
        return out[:n.value].tolist()

    def refcount(self, block):
        return self._lib.pa_block_refcount(self._h, int(block))


class PrefixCachePool:
    """Host block pool with automatic prefix caching (pa_pcache_*): requests
    whose prompts begin with cached full blocks share them; freed hashed
    blocks stay cached until the pool needs them (LRU)."""

    def __init__(self, num_blocks, block_size, free_order=None):
        self._lib = _lib.load()
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        handle = ctypes.c_void_p()
        order = None
        if free_order is not None:
            arr = np.ascontiguousarray(free_order, dtype=np.int32)
            if arr.shape != (self.num_blocks,):
                raise ValueError("free_order must list every block once")
            self._order = arr
            order = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        _lib.check("pa_pcache_create", self._lib.pa_pcache_create(
            self.num_blocks, self.block_size, order, ctypes.byref(handle)))
        self._h = handle

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_pcache_destroy(h)
            self._h = None

    @staticmethod
    def _tokens(tokens):
        arr = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def lookup(self, tokens, salt=0):
        """Number of leading full blocks of the prompt that are cached."""
        arr, ptr = self._tokens(tokens)
        n = ctypes.c_int()
        _lib.check("pa_pcache_lookup", self._lib.pa_pcache_lookup(
            self._h, ptr, arr.size, int(salt) & (2**64 - 1), ctypes.byref(n)))
        return n.value

    def add_request(self, seq, tokens, salt=0):
        """Returns (cached tokens, slot of every prompt position)."""
        arr, ptr = self._tokens(tokens)
        slots = np.empty(max(arr.size, 1), dtype=np.int64)
        cached = ctypes.c_int()
        _lib.check("pa_pcache_add", self._lib.pa_pcache_add(
            self._h, int(seq), ptr, arr.size, int(salt) & (2**64 - 1), ctypes.byref(cached),
            slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
        return cached.value, slots[:arr.size].tolist()

    def append(self, seq, token):
        slot = ctypes.c_int64()
        _lib.check("pa_pcache_append", self._lib.pa_pcache_append(
            self._h, int(seq), int(token), ctypes.byref(slot)))
        return slot.value

    def release(self, seq):
        _lib.check("pa_pcache_free", self._lib.pa_pcache_free(self._h, int(seq)))

    def table(self, seq):
        n = ctypes.c_int()
        out = np.empty(max(self.num_blocks, 1), dtype=np.int32)
        _lib.check("pa_pcache_block_table", self._lib.pa_pcache_block_table(
            self._h, int(seq), out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            self.num_blocks, ctypes.byref(n)))
        return out[:n.value].tolist()

    def length(self, seq):
        v = ctypes.c_int64()
        _lib.check("pa_pcache_len", self._lib.pa_pcache_len(self._h, int(seq), ctypes.byref(v)))
        return v.value

    def free_list(self):
        n = ctypes.c_int()
        out = np.empty(max(self.num_blocks, 1), dtype=np.int32)
        _lib.check("pa_pcache_free_queue", self._lib.pa_pcache_free_queue(
            self._h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), self.num_blocks,
            ctypes.byref(n)))
        return out[:n.value].tolist()

    def num_free(self):
        return self._lib.pa_pcache_num_free(self._h)

    def refcount(self, blk):
        return self._lib.pa_pcache_refcount(self._h, int(blk))

    def block_hash(self, blk):
        """The block's hash, or None when it is not cached."""
        h = ctypes.c_uint64()
        c = ctypes.c_int()
        _lib.check("pa_pcache_block_hash", self._lib.pa_pcache_block_hash(
            self._h, int(blk), ctypes.byref(h), ctypes.byref(c)))
        return h.value if c.value else None

    def hash_block(self, prev, tokens):
        arr, ptr = self._tokens(tokens)
        return int(self._lib.pa_pcache_hash_block(int(prev) & (2**64 - 1), ptr, arr.size))
