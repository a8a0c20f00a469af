"""Decode through pkv_paged_attention_decode_static_workspace, the entry point for
callers that cannot allocate device memory (a host engine that owns every
allocation and forbids new ones while it enqueues work, or a caller behind a
foreign-function layer without a device allocator).  Its partition scratch is a
fixed array inside the library instead of a caller-provided workspace.

Calls the C ABI directly.  Each result must be bit-identical to the regular
pkv_paged_attention_decode (torch-allocated workspace, same partition size, so
the same kernels run on the same inputs) and within the stated tolerance of the
oracle.  Calls come in a row on different batches -- one merged by the kernel for
up to 8 partitions a row, one with dozens of partitions a row (the other merge
kernel), then the first again -- so each call reads an array that still holds
the previous call's partials.  Once every kernel involved has run, repeated calls
must leave both the device's free memory and torch's allocation count unchanged.
This file is named to be collected last; it also passes on its own in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_293_gb300 import workloads
from gpu_helpers import TOL, dev_i32, host, max_abs, pkv

pytestmark = pytest.mark.gpu

DEV = "cuda"


class StaticCall:
    """Inputs of one static-workspace call, all allocated up front, so that the call itself
    touches no allocator."""

    def __init__(self, P, w, psize):
        self.P, self.w, self.psize = P, w, psize
        self.pool = P.make_pool(w.k_pool, w.v_pool)
        self.bt, self.ctx = dev_i32(w.block_tables), dev_i32(w.context_lens)
        self.out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"),
                              dtype=torch.float32, device=DEV)

    def __call__(self):
        w, P = self.w, self.P
        self.out.fill_(float("nan"))
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        status = P.lib.pkv_paged_attention_decode_static_workspace(
            ctypes.byref(self.pool), ctypes.c_void_p(w.q.data_ptr()), w.num_seqs, w.num_q_heads,
            ctypes.c_void_p(self.bt.data_ptr()), w.max_blocks_per_seq,
            ctypes.c_void_p(self.ctx.data_ptr()), w.max_context_len, w.scale,
            ctypes.c_void_p(self.out.data_ptr()), P.PKV_F32, self.psize, stream)
        torch.cuda.synchronize()
        return status


def _decode_with_workspace(P, w, psize):
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32, device=DEV)
    nbytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads,
                                          w.max_context_len, psize)
    assert nbytes > 0, "the batch should need partition scratch"
    ws = P.workspace_tensor(nbytes, DEV)
    P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                 dev_i32(w.context_lens), w.scale, out, w.max_context_len, psize,
                                 ws)
    torch.cuda.synchronize()
    return out


def test_static_workspace_decode_matches_regular_decode_and_oracle_in_a_row():
    P = pkv()
    a = workloads.build("noalloc_a", dtype="f16", num_q_heads=40, num_kv_heads=40, head_dim=128,
                        block_size=16, context_lens=[4096, 17, 1500, 700, 2049, 1], seed=21,
                        device=DEV)
    b = workloads.build("noalloc_b", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[600, 64, 1025], seed=22, device=DEV)
    calls = [StaticCall(P, a, 512),     # up to 8 partitions a row
             StaticCall(P, b, 16),      # up to 65 partitions a row
             StaticCall(P, a, 512)]     # the first batch again, over the second's leftovers
    want = {id(c): _decode_with_workspace(P, c.w, c.psize) for c in calls}
    ref = {id(c.w): oracle.paged_decode(c.w.dtype, host(c.w.k_pool), host(c.w.v_pool),
                                        host(c.w.q), c.w.block_tables, c.w.context_lens,
                                        c.w.scale) for c in calls}
    for c in calls:
        assert c() == P.PKV_OK
        assert torch.equal(c.out, want[id(c)])
        assert max_abs(c.out, ref[id(c.w)]) <= TOL[c.w.dtype]
        assert P.pkv_get_device_error() == 0
    # every kernel of these calls has run now: further calls allocate nothing
    free0, torch0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    for c in calls:
        assert c() == P.PKV_OK
    free1, torch1 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
    assert (free1, torch1) == (free0, torch0)
    for c in calls[1:]:
        assert torch.equal(c.out, want[id(c)])


def test_static_workspace_rejects_requests_larger_than_the_array():
    P = pkv()
    w = workloads.build("noalloc_big", dtype="f16", num_q_heads=40, num_kv_heads=40, head_dim=128,
                        block_size=16, context_lens=[4096] * 8, seed=23, device=DEV)
    need = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, w.max_context_len,
                                        16)
    assert need > P.STATIC_WORKSPACE_BYTES
    c = StaticCall(P, w, 16)
    c.out.zero_()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = P.lib.pkv_paged_attention_decode_static_workspace(
        ctypes.byref(c.pool), ctypes.c_void_p(w.q.data_ptr()), w.num_seqs, w.num_q_heads,
        ctypes.c_void_p(c.bt.data_ptr()), w.max_blocks_per_seq, ctypes.c_void_p(c.ctx.data_ptr()),
        w.max_context_len, w.scale, ctypes.c_void_p(c.out.data_ptr()), P.PKV_F32, 16, stream)
    torch.cuda.synchronize()
    assert status == P.PKV_ERR_WORKSPACE
    assert torch.count_nonzero(c.out).item() == 0       # nothing was launched
