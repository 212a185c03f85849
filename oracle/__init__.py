"""CPU oracle for the paged-KV decode path (fp64 attention, byte-exact copies).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg import this package.  The product
library never calls it, and it imports nothing from the product package.

Arrays are numpy.  bfloat16 data travels as ``uint16`` bit patterns and is
widened exactly inside the C code.  See ``oracle.c`` for the page citations of
every routine and ``block_manager.py`` for the host block manager model.
"""
import ctypes
import os

import numpy as np

from .build import build_oracle
from .block_manager import OracleBlockManager, pad_tables, run_script, sampling_memory

F32 = 0
BF16 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = build_oracle()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i32 = ctypes.c_int32
        i64 = ctypes.c_int64
        lib.orc_physical_index.restype = i64
        lib.orc_physical_index.argtypes = [p, i32, i64]
        lib.orc_slot_mapping.restype = None
        lib.orc_slot_mapping.argtypes = [p, i32, p, p, i32, i32, p]
        lib.orc_reshape_and_cache.restype = i32
        lib.orc_reshape_and_cache.argtypes = [p, p, p, i32, p, p, i32, i32, i32, i32, i32, i32]
        lib.orc_copy_blocks.restype = None
        lib.orc_copy_blocks.argtypes = [p, p, i64, p, i32]
        lib.orc_decode.restype = i32
        lib.orc_decode.argtypes = [p, i32, p, p, p, i32, i32, i32, i32, p, i32, p, i32, i32,
                                   ctypes.c_double, p, i32, i32, i32]
        _lib = lib
    return _lib


def _dtype_code(arr: np.ndarray) -> int:
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("oracle element arrays are float32 or uint16 (bfloat16 bits), got %s" % arr.dtype)


ROW = 0    # K and V [num_blocks, B, Hk, D]
SPLIT = 1  # K [num_blocks, Hk, D/x, B, x], V [num_blocks, Hk, D, B], x = 16 / element bytes


def cache_geometry(k_cache: np.ndarray, v_cache: np.ndarray):
    """(layout, num_blocks, B, Hk, D) read off the cache shapes."""
    if k_cache.ndim == 4:
        nb, bs, hk, d = k_cache.shape
        assert v_cache.shape == k_cache.shape
        return ROW, nb, bs, hk, d
    nb, hk, dx, bs, x = k_cache.shape
    assert x * k_cache.itemsize == 16 and v_cache.shape == (nb, hk, dx * x, bs)
    return SPLIT, nb, bs, hk, dx * x


def _ptr(arr: np.ndarray):
    return arr.ctypes.data_as(ctypes.c_void_p)


def _c(arr, dtype=None):
    return np.ascontiguousarray(arr if dtype is None else np.asarray(arr, dtype=dtype))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    u = bits.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def physical_index(table, block_size: int, pos: int) -> int:
    """PhysicalIndex of token ``pos`` through one block table."""
    t = _c(table, np.int32)
    return int(_load().orc_physical_index(_ptr(t), block_size, pos))


def slot_mapping(tables: np.ndarray, seq_ids, positions, block_size: int) -> np.ndarray:
    """Slots for new tokens (seq_ids[t], positions[t]) through [N, max_blocks] tables."""
    tables = _c(tables, np.int32)
    seq_ids = _c(seq_ids, np.int32)
    positions = _c(positions, np.int32)
    out = np.empty(seq_ids.shape[0], dtype=np.int64)
    _load().orc_slot_mapping(_ptr(tables), tables.shape[1], _ptr(seq_ids), _ptr(positions),
                             seq_ids.shape[0], block_size, _ptr(out))
    return out


def reshape_and_cache(k: np.ndarray, v: np.ndarray, slots, k_cache: np.ndarray,
                      v_cache: np.ndarray) -> int:
    """In-place cache write (k, v: [T, Hk, D]; caches in either layout).

    Returns the number of slots that lay beyond the pool (skipped)."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    code = _dtype_code(k_cache)
    k = _c(k, k_cache.dtype)
    v = _c(v, k_cache.dtype)
    slots = _c(slots, np.int64)
    layout, nb, bs, hk, d = cache_geometry(k_cache, v_cache)
    return int(_load().orc_reshape_and_cache(_ptr(k), _ptr(v), _ptr(slots), slots.shape[0],
                                             _ptr(k_cache), _ptr(v_cache), nb, bs, hk, d, code, layout))


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs) -> None:
    """In-place copy of whole blocks: for each (src, dst), block dst := block src."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    pairs = _c(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    block_bytes = k_cache[0].nbytes
    _load().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), block_bytes, _ptr(pairs), pairs.shape[0])


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
           seq_lens, scale: float, pairs=None, num_threads: int = 1) -> np.ndarray:
    """fp64 decode attention.  q: [N, H, D]; caches in either layout; tables [N, max_blocks].

    Returns float64 [N, H, D].  With ``pairs`` (a list of (seq, head)) only those
    entries are computed; the others are left as NaN."""
    code = _dtype_code(k_cache)
    q = _c(q, k_cache.dtype)
    k_cache = _c(k_cache)
    v_cache = _c(v_cache)
    tables = _c(block_tables, np.int32)
    lens = _c(seq_lens, np.int32)
    n, h, d = q.shape
    layout, nb, bs, hk, d2 = cache_geometry(k_cache, v_cache)
    assert d == d2 and tables.shape[0] == n and lens.shape[0] == n
    out = np.full((n, h, d), np.nan, dtype=np.float64)
    if pairs is None:
        pairs_arr = None
        npairs = 0
    else:
        # each (seq, head) once: the C loop writes a pair's row in place, and a
        # pair listed twice could be computed by two threads at the same time
        pairs_arr = _c(np.unique(np.asarray(pairs, dtype=np.int32).reshape(-1, 2), axis=0))
        npairs = pairs_arr.shape[0]
    rc = _load().orc_decode(_ptr(out), code, _ptr(q), _ptr(k_cache), _ptr(v_cache), nb, bs, hk, d,
                            _ptr(tables), tables.shape[1], _ptr(lens), n, h, float(scale),
                            None if pairs_arr is None else _ptr(pairs_arr), npairs,
                            int(num_threads), layout)
    if rc != 0:
        raise ValueError("oracle decode: a sequence length or block-table entry is out of range")
    return out


def available_threads() -> int:
    """Host threads the oracle may use for a timed baseline."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


__all__ = [
    "F32", "BF16", "ROW", "SPLIT", "cache_geometry", "OracleBlockManager", "run_script", "pad_tables",
    "bf16_bits_to_f64", "physical_index", "slot_mapping", "reshape_and_cache", "copy_blocks",
    "decode", "available_threads", "build_oracle",
]
