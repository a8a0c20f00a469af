"""CPU oracle for paged KV-cache decode -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this module.  It shares no code with the CUDA library; both sides
are fed by the seeded input generator alone.

Every function is a thin ctypes wrapper over oracle.c, which computes from the
plain definitions in fp64 (see the header of oracle.c for the passages of the
pages it follows and the readings it takes where the pages are silent):

- ``paged_decode``      softmax(scale * q K^T) V per (sequence, q head), with K
                        and V gathered in logical order through the block table
                        ("What Is vLLM", section "How does PagedAttention work?").
- ``partition_decode``  the same over ranges of P tokens, giving (m, l, o) per range.
- ``lse_merge``         the log-sum-exp combination of such partial results.
- ``Allocator``         block bookkeeping: a free-id stack and reference counts;
                        allocate for append (with copy-on-write of a shared
                        partly filled last block), fork, free ("vLLM in
                        Production", "PagedAttention - Virtual Memory for the KV
                        Cache"; "What Is vLLM", "How does PagedAttention work?").
- ``paged_decode_multi`` several new tokens per sequence, each attending causally
                        to the cache up to itself ("Serving models with vLLM":
                        chunked prefill, speculative decoding).
- ``slot_mapping``      slot = table[s][p // B] * B + p % B.
- ``kv_cache_write``    bit copy of new K/V rows into their slots.
- ``copy_blocks``       whole-block copy for copy-on-write of shared blocks
                        (same page, "Memory sharing").
- ``swap_blocks``       whole-block copy between two pools (device <-> host swap
                        of preempted sequences, same page, "What is continuous
                        batching in vLLM?").
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {"f32": F32, "f16": F16, "bf16": BF16}
_ELEM_BYTES = {F32: 4, F16: 2, BF16: 2}
_ERRORS = {1: "invalid argument", 2: "block id outside the pool or table", 3: "out of memory"}

_lib = None


def lib():
    global _lib
    if _lib is None:
        # ORACLE_LIB points the tests at a deliberately broken build of
        # oracle.c (the planted-mistake checks); normally the library is built here.
        path = os.environ.get("ORACLE_LIB") or _build.build()
        _lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        _lib.oracle_paged_decode.argtypes = [ctypes.c_int, P, P, i32, i32, i32, i32, P, i32, i32,
                                             P, i32, P, f32, P]
        _lib.oracle_partition_decode.argtypes = [ctypes.c_int, P, P, i32, i32, i32, i32, P, i32,
                                                 i32, P, i32, P, f32, i32, i32, P, P, P]
        _lib.oracle_lse_merge.argtypes = [i32, i32, i32, P, P, P, P]
        _lib.oracle_slot_mapping.argtypes = [P, i32, P, P, i32, i32, P]
        _lib.oracle_kv_cache_write.argtypes = [ctypes.c_int, P, P, i32, i32, i32, i32, P, P, P, i32]
        _lib.oracle_copy_blocks.argtypes = [P, P, i32, i64, P, i32]
        _lib.oracle_swap_blocks.argtypes = [P, P, i32, P, P, i32, i64, P, i32]
        _lib.oracle_allocator_reset.argtypes = [P, P, P, i32]
        _lib.oracle_allocate_for_append.argtypes = [P, P, P, i32, P, P, i64, i32, P, i32, P, P,
                                                    i32, P]
        _lib.oracle_fork_sequences.argtypes = [P, i32, i32, P, i32, P, P, i32]
        _lib.oracle_free_sequences.argtypes = [P, P, P, i32, i32, P, i32, P, P, i32]
        _lib.oracle_paged_decode_multi.argtypes = [ctypes.c_int, P, P, i32, i32, i32, i32, P, i32,
                                                   i32, i32, P, i32, P, f32, P]
        _lib.oracle_convert_to_double.argtypes = [ctypes.c_int, P, i64, P]
        _lib.oracle_num_threads.restype = ctypes.c_int
        _lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        for name in ("oracle_paged_decode", "oracle_partition_decode", "oracle_lse_merge",
                     "oracle_slot_mapping", "oracle_kv_cache_write", "oracle_copy_blocks",
                     "oracle_swap_blocks", "oracle_paged_decode_multi",
                     "oracle_allocate_for_append", "oracle_fork_sequences",
                     "oracle_free_sequences"):
            getattr(_lib, name).restype = ctypes.c_int
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc):
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, "error %d" % rc))


def _code(dtype):
    return _DTYPE_CODE[dtype] if isinstance(dtype, str) else int(dtype)


def _raw(a, itemsize=None):
    """Contiguous numpy view of element storage (fp16/bf16 as uint16 bits)."""
    a = np.ascontiguousarray(a)
    if itemsize is not None and a.dtype.itemsize != itemsize:
        raise ValueError("element size %d, expected %d" % (a.dtype.itemsize, itemsize))
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def num_threads():
    return lib().oracle_num_threads()


def set_num_threads(n):
    lib().oracle_set_num_threads(int(n))


def convert_to_double(dtype, bits):
    code = _code(dtype)
    bits = _raw(bits, _ELEM_BYTES[code])
    out = np.empty(bits.shape, dtype=np.float64)
    lib().oracle_convert_to_double(code, _ptr(bits), bits.size, _ptr(out))
    return out


def paged_decode(dtype, k_pool, v_pool, q, block_tables, context_lens, scale):
    """k_pool, v_pool: [N][Hkv][B][D] element storage; q: [S][Hq][D]; returns [S][Hq][D] float64."""
    code = _code(dtype)
    e = _ELEM_BYTES[code]
    k_pool, v_pool, q = _raw(k_pool, e), _raw(v_pool, e), _raw(q, e)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    N, Hkv, B, D = k_pool.shape
    S, Hq, Dq = q.shape
    assert Dq == D and v_pool.shape == k_pool.shape and bt.shape[0] == S and ctx.shape == (S,)
    out = np.zeros((S, Hq, D), dtype=np.float64)
    _check(lib().oracle_paged_decode(code, _ptr(k_pool), _ptr(v_pool), N, B, Hkv, D, _ptr(q), S, Hq,
                                     _ptr(bt), bt.shape[1], _ptr(ctx), float(np.float32(scale)),
                                     _ptr(out)))
    return out


def partition_decode(dtype, k_pool, v_pool, q, block_tables, context_lens, scale, partition_size,
                     max_parts=None):
    """Per-range partial results (m, l, o): m, l [S][Hq][max_parts], o [S][Hq][max_parts][D]."""
    code = _code(dtype)
    e = _ELEM_BYTES[code]
    k_pool, v_pool, q = _raw(k_pool, e), _raw(v_pool, e), _raw(q, e)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    N, Hkv, B, D = k_pool.shape
    S, Hq, _ = q.shape
    P = int(partition_size)
    if max_parts is None:
        max_parts = max(1, -(-int(ctx.max(initial=0)) // P))
    m = np.empty((S, Hq, max_parts), dtype=np.float64)
    l = np.empty((S, Hq, max_parts), dtype=np.float64)
    o = np.empty((S, Hq, max_parts, D), dtype=np.float64)
    _check(lib().oracle_partition_decode(code, _ptr(k_pool), _ptr(v_pool), N, B, Hkv, D, _ptr(q), S,
                                         Hq, _ptr(bt), bt.shape[1], _ptr(ctx),
                                         float(np.float32(scale)), P, max_parts, _ptr(m), _ptr(l),
                                         _ptr(o)))
    return m, l, o


def lse_merge(m, l, o):
    """m, l: [..., K]; o: [..., K, D] -> [..., D] float64."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    o = np.ascontiguousarray(o, dtype=np.float64)
    lead = m.shape[:-1]
    K = m.shape[-1]
    D = o.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (D,), dtype=np.float64)
    _check(lib().oracle_lse_merge(rows, K, D, _ptr(m), _ptr(l), _ptr(o), _ptr(out)))
    return out


def slot_mapping(block_tables, positions, block_size, token_seq=None):
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    ts = None if token_seq is None else np.ascontiguousarray(token_seq, dtype=np.int32)
    out = np.empty(pos.shape, dtype=np.int64)
    _check(lib().oracle_slot_mapping(_ptr(bt), bt.shape[1], _ptr(pos), _ptr(ts), pos.size,
                                     int(block_size), _ptr(out)))
    return out


def kv_cache_write(dtype, k_pool, v_pool, k_new, v_new, slots):
    """In-place on the (contiguous numpy) pools; k_new, v_new: [T][Hkv][D]."""
    code = _code(dtype)
    e = _ELEM_BYTES[code]
    for a in (k_pool, v_pool):
        if not a.flags.c_contiguous or a.dtype.itemsize != e:
            raise ValueError("pools must be contiguous element storage")
    k_new, v_new = _raw(k_new, e), _raw(v_new, e)
    sl = np.ascontiguousarray(slots, dtype=np.int64)
    N, Hkv, B, D = k_pool.shape
    _check(lib().oracle_kv_cache_write(code, _ptr(k_pool), _ptr(v_pool), N, B, Hkv, D, _ptr(k_new),
                                       _ptr(v_new), _ptr(sl), sl.size))


def copy_blocks(k_pool, v_pool, pairs):
    """In-place on the pools; pairs: [n][2] = (src, dst)."""
    for a in (k_pool, v_pool):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be contiguous")
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    N = k_pool.shape[0]
    block_bytes = k_pool.nbytes // N
    _check(lib().oracle_copy_blocks(_ptr(k_pool), _ptr(v_pool), N, block_bytes, _ptr(pr),
                                    pr.shape[0]))


def swap_blocks(src_k, src_v, dst_k, dst_v, pairs):
    """Block dst of (dst_k, dst_v) <- block src of (src_k, src_v) for each (src, dst) pair."""
    for a in (src_k, src_v, dst_k, dst_v):
        if not a.flags.c_contiguous:
            raise ValueError("pools must be contiguous")
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype.itemsize != dst_k.dtype.itemsize:
        raise ValueError("pools must have the same block geometry")
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    block_bytes = src_k.nbytes // src_k.shape[0]
    _check(lib().oracle_swap_blocks(_ptr(src_k), _ptr(src_v), src_k.shape[0], _ptr(dst_k),
                                    _ptr(dst_v), dst_k.shape[0], block_bytes, _ptr(pr), pr.shape[0]))


def paged_decode_multi(dtype, k_pool, v_pool, q, block_tables, context_lens, scale):
    """q: [S][nq][Hq][D]; the last nq positions are the new tokens; returns [S][nq][Hq][D]."""
    code = _code(dtype)
    e = _ELEM_BYTES[code]
    k_pool, v_pool, q = _raw(k_pool, e), _raw(v_pool, e), _raw(q, e)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    N, Hkv, B, D = k_pool.shape
    S, nq, Hq, _ = q.shape
    out = np.zeros((S, nq, Hq, D), dtype=np.float64)
    _check(lib().oracle_paged_decode_multi(code, _ptr(k_pool), _ptr(v_pool), N, B, Hkv, D, _ptr(q),
                                           S, nq, Hq, _ptr(bt), bt.shape[1], _ptr(ctx),
                                           float(np.float32(scale)), _ptr(out)))
    return out


class Allocator:
    """Host state of the block bookkeeping, updated one sequence after another."""

    def __init__(self, num_blocks):
        self.num_blocks = int(num_blocks)
        self.free_ids = np.zeros(num_blocks, np.int32)
        self.free_count = np.zeros(1, np.int32)
        self.refcount = np.zeros(num_blocks, np.int32)
        lib().oracle_allocator_reset(_ptr(self.free_ids), _ptr(self.free_count),
                                     _ptr(self.refcount), self.num_blocks)

    def allocate_for_append(self, k_pool, v_pool, block_size, block_tables, old_lens, new_lens):
        """In place on block_tables (contiguous int32) and the pools; returns statuses."""
        assert block_tables.dtype == np.int32 and block_tables.flags.c_contiguous
        old = np.ascontiguousarray(old_lens, np.int32)
        new = np.ascontiguousarray(new_lens, np.int32)
        status = np.zeros(old.shape, np.int32)
        block_bytes = k_pool.nbytes // k_pool.shape[0]
        _check(lib().oracle_allocate_for_append(
            _ptr(self.free_ids), _ptr(self.free_count), _ptr(self.refcount), self.num_blocks,
            _ptr(k_pool), _ptr(v_pool), block_bytes, int(block_size), _ptr(block_tables),
            block_tables.shape[1], _ptr(old), _ptr(new), old.size, _ptr(status)))
        return status

    def fork(self, block_size, block_tables, pairs, lens):
        pr = np.ascontiguousarray(pairs, np.int32).reshape(-1, 2)
        ln = np.ascontiguousarray(lens, np.int32)
        _check(lib().oracle_fork_sequences(_ptr(self.refcount), self.num_blocks, int(block_size),
                                           _ptr(block_tables), block_tables.shape[1], _ptr(pr),
                                           _ptr(ln), pr.shape[0]))

    def free(self, block_size, block_tables, seqs, lens):
        sq = np.ascontiguousarray(seqs, np.int32)
        ln = np.ascontiguousarray(lens, np.int32)
        _check(lib().oracle_free_sequences(_ptr(self.free_ids), _ptr(self.free_count),
                                           _ptr(self.refcount), self.num_blocks, int(block_size),
                                           _ptr(block_tables), block_tables.shape[1], _ptr(sq),
                                           _ptr(ln), sq.size))
