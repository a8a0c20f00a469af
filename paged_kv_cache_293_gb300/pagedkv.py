"""ctypes binding of libpagedkv.so (include/pagedkv.h), same entry-point names.

Argument marshalling only: torch tensors in, raw device pointers, sizes and
the caller's CUDA stream out to the C ABI.  Every step of the path runs in the
library's kernels.  Importing this module fails when the library has not been
built (``python -m paged_kv_cache_293_gb300._build`` or
``__graft_entry__.build()``); there is no fallback.
"""
import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "pagedkv.h")

if not os.path.exists(LIB_PATH):
    raise ImportError("libpagedkv.so is not built (%s); run python -m paged_kv_cache_293_gb300._build"
                      % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

PKV_OK, PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA, PKV_ERR_DEVICE = range(6)
PKV_F32, PKV_F16, PKV_BF16 = 0, 1, 2
DEVERR = {"BLOCK_ID": 0x1, "SLOT": 0x2, "CONTEXT": 0x4, "TIMEOUT": 0x8, "POSITION": 0x10,
          "PAIR": 0x20, "PREFIX": 0x40}

_DTYPE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}


class pkv_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class pkv_block_allocator(ctypes.Structure):
    _fields_ = [("free_ids", ctypes.c_void_p), ("free_count", ctypes.c_void_p),
                ("refcount", ctypes.c_void_p), ("num_blocks", ctypes.c_int32)]


_P, _i32, _i64, _sz, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_PP = ctypes.POINTER(pkv_pool)
_PA = ctypes.POINTER(pkv_block_allocator)
_SIGS = {
    "pkv_slot_mapping": (_i32, [_P, _i32, _i32, _P, _P, _i32, _i32, _P, _P]),
    "pkv_kv_cache_write": (_i32, [_PP, _P, _P, _P, _i32, _P]),
    "pkv_choose_partition_size": (_i32, [_PP, _i32, _i32, _i32]),
    "pkv_decode_workspace_bytes": (_sz, [_PP, _i32, _i32, _i32, _i32]),
    "pkv_partition_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "pkv_paged_attention_decode": (_i32, [_PP, _P, _i32, _i32, _P, _i32, _P, _i32, _f32, _P, _i32,
                                          _i32, _P, _sz, _P]),
    "pkv_paged_attention_decode_static_workspace": (_i32, [_PP, _P, _i32, _i32, _P, _i32, _P,
                                                           _i32, _f32, _P, _i32, _i32, _P]),
    "pkv_paged_attention_decode_append": (_i32, [_PP, _P, _P, _P, _i32, _i32, _P, _i32, _P, _i32,
                                                 _f32, _P, _i32, _i32, _P, _sz, _P, _P]),
    "pkv_paged_attention_decode_multi": (_i32, [_PP, _P, _i32, _i32, _i32, _P, _i32, _P, _i32,
                                                _f32, _P, _i32, _i32, _P, _sz, _P]),
    "pkv_paged_attention_decode_multi_append": (_i32, [_PP, _P, _P, _P, _i32, _i32, _i32, _P,
                                                       _i32, _P, _i32, _f32, _P, _i32, _i32, _P,
                                                       _sz, _P, _P]),
    "pkv_cascade_workspace_bytes": (_sz, [_PP, _i32, _i32, _i32, _i32, _i32]),
    "pkv_paged_attention_decode_cascade": (_i32, [_PP, _P, _i32, _i32, _P, _i32, _P, _i32, _f32,
                                                  _i32, _P, _i32, _i32, _P, _P, _P, _P, _sz, _P]),
    "pkv_paged_attention_partitions": (_i32, [_PP, _P, _i32, _i32, _P, _i32, _P, _i32, _f32, _i32,
                                              _P, _sz, _P]),
    "pkv_lse_merge": (_i32, [_P, _sz, _i32, _i32, _i32, _P, _i32, _i32, _P, _i32, _P]),
    "pkv_copy_blocks": (_i32, [_PP, _P, _i32, _P]),
    "pkv_swap_blocks": (_i32, [_PP, _PP, _P, _i32, _P]),
    "pkv_get_device_error": (_i32, [ctypes.POINTER(ctypes.c_uint32), _P]),
    "pkv_allocator_reset": (_i32, [_PA, _P]),
    "pkv_allocate_for_append": (_i32, [_PA, _PP, _P, _i32, _P, _P, _i32, _P, _P]),
    "pkv_fork_sequences": (_i32, [_PA, _i32, _P, _i32, _P, _P, _i32, _P]),
    "pkv_free_sequences": (_i32, [_PA, _i32, _P, _i32, _P, _P, _i32, _P]),
    "pkv_status_str": (ctypes.c_char_p, [_i32]),
    "pkv_version": (_i32, []),
    "pkv_set_decode_engine": (_i32, [_i32]),
    "pkv_get_decode_engine": (_i32, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def declared_functions(header=HEADER_PATH):
    """Names of the functions include/pagedkv.h declares."""
    with open(header) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


class PagedKVError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, pkv_status_str(status), status))


def _check(status, where):
    if status != PKV_OK:
        raise PagedKVError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, ref=None):
    if stream is None:
        if ref is not None and ref.is_cuda:
            return ctypes.c_void_p(torch.cuda.current_stream(ref.device).cuda_stream)
        return None
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors passed to libpagedkv must be contiguous")


def make_pool(k_pool, v_pool):
    """pkv_pool view of two [N][Hkv][B][D] tensors."""
    _contig(k_pool, v_pool)
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or k_pool.dim() != 4:
        raise ValueError("k_pool and v_pool must be matching [N][Hkv][B][D] tensors")
    N, Hkv, B, D = k_pool.shape
    return pkv_pool(k_pool.data_ptr(), v_pool.data_ptr(), N, B, Hkv, D, _DTYPE[k_pool.dtype])


def pkv_status_str(status):
    return lib.pkv_status_str(int(status)).decode()


def pkv_version():
    return lib.pkv_version()


ENGINE_AUTO, ENGINE_CUDA_CORES, ENGINE_TENSOR_CORES = 0, 1, 2


def pkv_set_decode_engine(engine):
    _check(lib.pkv_set_decode_engine(int(engine)), "pkv_set_decode_engine")


def pkv_get_decode_engine():
    return lib.pkv_get_decode_engine()


def pkv_slot_mapping(block_tables, positions, block_size, slot_mapping, token_seq=None,
                     stream=None):
    _contig(block_tables, positions, slot_mapping, token_seq)
    S, M = block_tables.shape
    _check(lib.pkv_slot_mapping(_ptr(block_tables), M, S, _ptr(positions), _ptr(token_seq),
                                positions.numel(), int(block_size), _ptr(slot_mapping),
                                _stream(stream, block_tables)), "pkv_slot_mapping")


def pkv_kv_cache_write(k_pool, v_pool, k_new, v_new, slot_mapping, stream=None):
    _contig(k_new, v_new, slot_mapping)
    pool = make_pool(k_pool, v_pool)
    _check(lib.pkv_kv_cache_write(ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
                                  slot_mapping.numel(), _stream(stream, k_pool)),
           "pkv_kv_cache_write")


def pkv_choose_partition_size(k_pool, num_seqs, num_q_heads, max_context_len):
    pool = make_pool(k_pool, k_pool)
    return lib.pkv_choose_partition_size(ctypes.byref(pool), num_seqs, num_q_heads, max_context_len)


def pkv_decode_workspace_bytes(k_pool, num_seqs, num_q_heads, max_context_len, partition_size=0):
    pool = make_pool(k_pool, k_pool)
    return lib.pkv_decode_workspace_bytes(ctypes.byref(pool), num_seqs, num_q_heads,
                                          max_context_len, partition_size)


def pkv_partition_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                  partition_size):
    return lib.pkv_partition_workspace_bytes(num_seqs, num_q_heads, head_dim, max_context_len,
                                             partition_size)


def pkv_paged_attention_decode(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                               max_context_len, partition_size=0, workspace=None, stream=None):
    _contig(q, block_tables, context_lens, out, workspace)
    pool = make_pool(k_pool, v_pool)
    S, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode(ctypes.byref(pool), _ptr(q), S, Hq, _ptr(block_tables),
                                          block_tables.shape[1], _ptr(context_lens),
                                          int(max_context_len), float(scale), _ptr(out),
                                          _DTYPE[out.dtype], int(partition_size), _ptr(workspace),
                                          ws_bytes, _stream(stream, q)),
           "pkv_paged_attention_decode")


def pkv_paged_attention_decode_append(q, k_pool, v_pool, k_new, v_new, block_tables,
                                      context_lens, scale, out, max_context_len,
                                      partition_size=0, workspace=None, slot_mapping=None,
                                      stream=None):
    _contig(q, k_new, v_new, block_tables, context_lens, out, workspace, slot_mapping)
    pool = make_pool(k_pool, v_pool)
    S, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_append(
        ctypes.byref(pool), _ptr(q), _ptr(k_new), _ptr(v_new), S, Hq, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _DTYPE[out.dtype], int(partition_size), _ptr(workspace), ws_bytes, _ptr(slot_mapping),
        _stream(stream, q)), "pkv_paged_attention_decode_append")


def pkv_paged_attention_decode_multi(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                                     max_context_len, partition_size=0, workspace=None,
                                     stream=None):
    """q, out: [num_seqs][num_queries][num_q_heads][head_dim]."""
    _contig(q, block_tables, context_lens, out, workspace)
    pool = make_pool(k_pool, v_pool)
    S, NQ, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_multi(
        ctypes.byref(pool), _ptr(q), NQ, S, Hq, _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), float(scale), _ptr(out), _DTYPE[out.dtype],
        int(partition_size), _ptr(workspace), ws_bytes, _stream(stream, q)),
        "pkv_paged_attention_decode_multi")


def pkv_paged_attention_decode_multi_append(q, k_pool, v_pool, k_new, v_new, block_tables,
                                            context_lens, scale, out, max_context_len,
                                            partition_size=0, workspace=None, slot_mapping=None,
                                            stream=None):
    """q, out: [num_seqs][num_queries][num_q_heads][head_dim]; k_new, v_new:
    [num_seqs][num_queries][num_kv_heads][head_dim], written to the pools at the last
    num_queries positions of each context in the same launch."""
    _contig(q, k_new, v_new, block_tables, context_lens, out, workspace, slot_mapping)
    pool = make_pool(k_pool, v_pool)
    S, NQ, Hq, _ = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_multi_append(
        ctypes.byref(pool), _ptr(q), _ptr(k_new), _ptr(v_new), NQ, S, Hq, _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), int(max_context_len), float(scale), _ptr(out),
        _DTYPE[out.dtype], int(partition_size), _ptr(workspace), ws_bytes, _ptr(slot_mapping),
        _stream(stream, q)), "pkv_paged_attention_decode_multi_append")


def pkv_cascade_workspace_bytes(k_pool, num_seqs, num_q_heads, max_context_len, prefix_len,
                                partition_size=0):
    pool = make_pool(k_pool, k_pool)
    return lib.pkv_cascade_workspace_bytes(ctypes.byref(pool), num_seqs, num_q_heads,
                                           max_context_len, prefix_len, partition_size)


def pkv_paged_attention_decode_cascade(q, k_pool, v_pool, block_tables, context_lens, scale, out,
                                       max_context_len, prefix_len, workspace, partition_size=0,
                                       k_new=None, v_new=None, slot_mapping=None, stream=None):
    """Decode for a batch whose sequences all share their first prefix_len tokens' blocks."""
    _contig(q, block_tables, context_lens, out, workspace, k_new, v_new, slot_mapping)
    pool = make_pool(k_pool, v_pool)
    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_decode_cascade(
        ctypes.byref(pool), _ptr(q), S, Hq, _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), float(scale), int(prefix_len), _ptr(out),
        _DTYPE[out.dtype], int(partition_size), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
        _ptr(workspace), ws_bytes, _stream(stream, q)), "pkv_paged_attention_decode_cascade")


def pkv_paged_attention_decode_static_workspace(q, k_pool, v_pool, block_tables, context_lens,
                                                scale, out, max_context_len, partition_size=0,
                                                stream=None):
    """Decode for callers that cannot allocate device memory: the partition scratch is a
    fixed array inside the library (PKV_STATIC_WORKSPACE_BYTES) shared by all calls."""
    _contig(q, block_tables, context_lens, out)
    pool = make_pool(k_pool, v_pool)
    S, Hq, _ = q.shape
    _check(lib.pkv_paged_attention_decode_static_workspace(
        ctypes.byref(pool), _ptr(q), S, Hq, _ptr(block_tables), block_tables.shape[1],
        _ptr(context_lens), int(max_context_len), float(scale), _ptr(out), _DTYPE[out.dtype],
        int(partition_size), _stream(stream, q)), "pkv_paged_attention_decode_static_workspace")


STATIC_WORKSPACE_BYTES = 32 << 20


def pkv_paged_attention_partitions(q, k_pool, v_pool, block_tables, context_lens, scale,
                                   max_context_len, partition_size, workspace, stream=None):
    _contig(q, block_tables, context_lens, workspace)
    pool = make_pool(k_pool, v_pool)
    S, Hq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.pkv_paged_attention_partitions(ctypes.byref(pool), _ptr(q), S, Hq,
                                              _ptr(block_tables), block_tables.shape[1],
                                              _ptr(context_lens), int(max_context_len),
                                              float(scale), int(partition_size), _ptr(workspace),
                                              ws_bytes, _stream(stream, q)),
           "pkv_paged_attention_partitions")


def pkv_lse_merge(workspace, num_seqs, num_q_heads, head_dim, context_lens, max_context_len,
                  partition_size, out, stream=None):
    _contig(workspace, context_lens, out)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib.pkv_lse_merge(_ptr(workspace), ws_bytes, num_seqs, num_q_heads, head_dim,
                             _ptr(context_lens), int(max_context_len), int(partition_size),
                             _ptr(out), _DTYPE[out.dtype], _stream(stream, out)), "pkv_lse_merge")


def pkv_copy_blocks(k_pool, v_pool, src_dst_pairs, stream=None):
    _contig(src_dst_pairs)
    pool = make_pool(k_pool, v_pool)
    n = src_dst_pairs.numel() // 2
    _check(lib.pkv_copy_blocks(ctypes.byref(pool), _ptr(src_dst_pairs), n, _stream(stream, k_pool)),
           "pkv_copy_blocks")


def pkv_swap_blocks(src_k, src_v, dst_k, dst_v, src_dst_pairs, stream=None):
    """Blocks between two pools (device or pinned host tensors); pairs on the device or pinned."""
    _contig(src_dst_pairs)
    src = make_pool(src_k, src_v)
    dst = make_pool(dst_k, dst_v)
    ref = src_k if src_k.is_cuda else dst_k
    n = src_dst_pairs.numel() // 2
    _check(lib.pkv_swap_blocks(ctypes.byref(src), ctypes.byref(dst), _ptr(src_dst_pairs), n,
                               _stream(stream, ref)), "pkv_swap_blocks")


class BlockAllocator:
    """Device arrays of the block bookkeeping (free-id stack, count, reference counts)."""

    def __init__(self, num_blocks, device):
        self.free_ids = torch.empty(num_blocks, dtype=torch.int32, device=device)
        self.free_count = torch.zeros(1, dtype=torch.int32, device=device)
        self.refcount = torch.zeros(num_blocks, dtype=torch.int32, device=device)
        self.num_blocks = int(num_blocks)

    def struct(self):
        return pkv_block_allocator(self.free_ids.data_ptr(), self.free_count.data_ptr(),
                                   self.refcount.data_ptr(), self.num_blocks)


def pkv_allocator_reset(alloc, stream=None):
    a = alloc.struct()
    _check(lib.pkv_allocator_reset(ctypes.byref(a), _stream(stream, alloc.refcount)),
           "pkv_allocator_reset")


def pkv_allocate_for_append(alloc, k_pool, v_pool, block_tables, old_lens, new_lens, seq_status,
                            stream=None):
    _contig(block_tables, old_lens, new_lens, seq_status)
    a, pool = alloc.struct(), make_pool(k_pool, v_pool)
    S, M = block_tables.shape
    _check(lib.pkv_allocate_for_append(ctypes.byref(a), ctypes.byref(pool), _ptr(block_tables), M,
                                       _ptr(old_lens), _ptr(new_lens), S, _ptr(seq_status),
                                       _stream(stream, block_tables)), "pkv_allocate_for_append")


def pkv_fork_sequences(alloc, block_size, block_tables, src_dst_seqs, lens, stream=None):
    _contig(block_tables, src_dst_seqs, lens)
    a = alloc.struct()
    _check(lib.pkv_fork_sequences(ctypes.byref(a), int(block_size), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(src_dst_seqs), _ptr(lens),
                                  src_dst_seqs.numel() // 2, _stream(stream, block_tables)),
           "pkv_fork_sequences")


def pkv_free_sequences(alloc, block_size, block_tables, seqs, lens, stream=None):
    _contig(block_tables, seqs, lens)
    a = alloc.struct()
    _check(lib.pkv_free_sequences(ctypes.byref(a), int(block_size), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(seqs), _ptr(lens), seqs.numel(),
                                  _stream(stream, block_tables)), "pkv_free_sequences")


def pkv_get_device_error(stream=None, device=None):
    """Synchronise the stream, return and clear the device error word (0 = none)."""
    flags = ctypes.c_uint32(0)
    ref = None
    if stream is None and torch.cuda.is_available():
        ref = torch.empty(0, device=device or "cuda")
    st = lib.pkv_get_device_error(ctypes.byref(flags), _stream(stream, ref))
    if st not in (PKV_OK, PKV_ERR_DEVICE):
        raise PagedKVError(st, "pkv_get_device_error")
    return flags.value


def workspace_tensor(nbytes, device):
    """A device byte buffer for the workspace (16-byte aligned, as torch allocations are)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
