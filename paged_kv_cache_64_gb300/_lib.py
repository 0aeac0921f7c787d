"""ctypes declarations of the C ABI in include/pa.h (argument marshalling only).

The library is loaded lazily on first use.  If libpa.so has not been built the
load fails loudly with LibraryMissing: there is no fallback of any kind.
"""
import ctypes
import os

from . import build as _build

PA_OK = 0
STATUS = {
    0: "PA_OK",
    1: "PA_ERR_INVALID",
    2: "PA_ERR_OUT_OF_BLOCKS",
    3: "PA_ERR_UNSUPPORTED",
    4: "PA_ERR_CUDA",
    5: "PA_ERR_DEVICE_TIMEOUT",
    6: "PA_ERR_BAD_INDEX",
    7: "PA_ERR_NOT_FOUND",
    8: "PA_ERR_TOO_LARGE",
}
# Size of the fixed device scratch behind pa_decode_static_scratch (pa.h).
STATIC_SCRATCH_BYTES = 16 << 20
PA_F16, PA_BF16 = 0, 1

# Every symbol pa.h declares, with (restype, argtypes).
_c_int, _c_i64, _c_sz, _c_f = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_vp = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_intp = ctypes.POINTER(ctypes.c_int)

SIGNATURES = {
    "pa_version": (_c_int, []),
    "pa_status_string": (ctypes.c_char_p, [_c_int]),
    "pa_cache_write": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                _c_int, _vp]),
    "pa_copy_blocks": (_c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _c_int, _vp, _c_int,
                                _c_int, _c_sz, _vp]),
    "pa_decode": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp, _c_int, _c_int, _c_int,
                           _c_int, _c_int, _c_int, _c_f, _c_int, _vp, _c_sz, _c_int, _vp]),
    "pa_decode_step": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp,
                                _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_int, _vp,
                                _c_sz, _c_int, _vp]),
    "pa_decode_cascade": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int,
                                   _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f,
                                   _c_int, _vp, _c_sz, _c_int, _vp]),
    "pa_decode_cascade_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                 _c_int, _c_int]),
    "pa_pcache_create": (_c_int, [_c_int, _c_int, _i32p, ctypes.POINTER(_vp)]),
    "pa_pcache_destroy": (None, [_vp]),
    "pa_pcache_hash_block": (ctypes.c_uint64, [ctypes.c_uint64, _i32p, _c_int]),
    "pa_pcache_lookup": (_c_int, [_vp, _i32p, _c_int, ctypes.c_uint64, _intp]),
    "pa_pcache_add": (_c_int, [_vp, ctypes.c_int64, _i32p, _c_int, ctypes.c_uint64, _intp, _i64p]),
    "pa_pcache_append": (_c_int, [_vp, ctypes.c_int64, ctypes.c_int32, _i64p]),
    "pa_pcache_free": (_c_int, [_vp, ctypes.c_int64]),
    "pa_pcache_block_table": (_c_int, [_vp, ctypes.c_int64, _i32p, _c_int, _intp]),
    "pa_pcache_len": (_c_int, [_vp, ctypes.c_int64, _i64p]),
    "pa_pcache_num_free": (_c_int, [_vp]),
    "pa_pcache_free_queue": (_c_int, [_vp, _i32p, _c_int, _intp]),
    "pa_pcache_refcount": (_c_int, [_vp, _c_int]),
    "pa_pcache_block_hash": (_c_int, [_vp, _c_int, ctypes.POINTER(ctypes.c_uint64), _intp]),
    "pa_cache_write_fp8": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int,
                                    _c_int, _c_f, _c_f, _c_int, _vp]),
    "pa_decode_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp,
                               _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_f, _c_f,
                               _c_int, _vp, _c_sz, _c_int, _vp]),
    "pa_decode_fp8_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                             _c_int, _c_int]),
    "pa_decode_auto_partition": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          _c_int]),
    "pa_decode_fp8_auto_partition": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          _c_int]),
    "pa_decode_partial_tokens": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          _c_int, _c_int]),
    "pa_decode_ctas_per_sm": (_c_int, [_c_int, _c_int, _c_int]),
    "pa_set_decode_impl": (_c_int, [_c_int]),
    "pa_get_decode_impl": (_c_int, []),
    "pa_set_decode_span": (_c_int, [_c_int]),
    "pa_decode_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                         _c_int]),
    "pa_decode_partitions": (_c_int, [_vp, _vp, _vp, _c_int, _vp, _c_int, _vp, _c_int, _c_int,
                                      _c_int, _c_int, _c_int, _c_int, _c_f, _c_int, _vp, _c_sz,
                                      _c_int, _vp]),
    "pa_split_kv_reduce": (_c_int, [_vp, _vp, _c_sz, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _vp]),
    "pa_decode_static_scratch": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _vp, _c_int,
                                          _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_int,
                                          _c_int, _vp]),
    "pa_shared_prefix_len": (_c_int, [_i32p, _c_int, _i32p, _c_int, _c_int, _intp]),
    "pa_check_error": (_c_int, [_vp]),
    "pa_selftest_wait_timeout": (_c_int, [_vp]),
    "pa_alloc_create": (_c_int, [_c_int, _c_int, _i32p, ctypes.POINTER(_vp)]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_seq_add": (_c_int, [_vp, _c_i64]),
    "pa_seq_append": (_c_int, [_vp, _c_i64, _c_int, _i64p, _i64p, _intp]),
    "pa_seq_fork": (_c_int, [_vp, _c_i64, _c_i64]),
    "pa_seq_free": (_c_int, [_vp, _c_i64]),
    "pa_seq_len": (_c_int, [_vp, _c_i64, _i64p]),
    "pa_seq_block_table": (_c_int, [_vp, _c_i64, _i32p, _c_int, _intp]),
    "pa_alloc_export": (_c_int, [_vp, _i64p, _c_int, _i32p, _c_int, _i32p]),
    "pa_alloc_num_free": (_c_int, [_vp]),
    "pa_alloc_free_list": (_c_int, [_vp, _i32p, _c_int, _intp]),
    "pa_block_refcount": (_c_int, [_vp, _c_int]),
}


class LibraryMissing(RuntimeError):
    pass


class PagedAttentionError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")


class OutOfBlocks(PagedAttentionError):
    pass


_lib = None


def lib_path():
    return _build.LIB


def load():
    """Load libpa.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise LibraryMissing(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(fn_name, code):
    if code != PA_OK:
        if code == 2:
            raise OutOfBlocks(fn_name, code)
        raise PagedAttentionError(fn_name, code)
