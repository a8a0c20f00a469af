"""Decode through pkv_paged_attention_decode_static_workspace, the entry point for
callers that cannot allocate device memory (a host engine that owns every
allocation and forbids new ones while it enqueues work, or a caller behind a
foreign-function layer without a device allocator).  Its partition scratch is a
fixed array inside the library instead of a caller-provided workspace.

Calls the C ABI directly and checks each result against the regular
pkv_paged_attention_decode (with a torch-allocated workspace) on the same
inputs, for two calls in a row on different batches, so that the second call
must not be disturbed by what the first left in the shared array.  This file
is named to be collected last; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_cache_293_gb300 import workloads
from gpu_helpers import dev_i32, pkv

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_SAME_PATH = 1e-5   # fp32 output, same kernels on both sides


def _decode_static(P, w, out, psize):
    """The no-allocation entry point, called through the C ABI."""
    pool = P.make_pool(w.k_pool, w.v_pool)
    bt, ctx = dev_i32(w.block_tables), dev_i32(w.context_lens)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = P.lib.pkv_paged_attention_decode_static_workspace(
        ctypes.byref(pool), ctypes.c_void_p(w.q.data_ptr()), w.num_seqs, w.num_q_heads,
        ctypes.c_void_p(bt.data_ptr()), w.max_blocks_per_seq, ctypes.c_void_p(ctx.data_ptr()),
        w.max_context_len, w.scale, ctypes.c_void_p(out.data_ptr()), P.PKV_F32, psize, stream)
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


def test_static_workspace_decode_matches_regular_decode_twice_in_a_row():
    P = pkv()
    batches = [
        workloads.build("noalloc_a", dtype="f16", num_q_heads=40, num_kv_heads=40, head_dim=128,
                        block_size=16, context_lens=[4096, 17, 1500, 700, 2049, 1], seed=21,
                        device=DEV),
        workloads.build("noalloc_b", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[3000, 64, 1025], seed=22, device=DEV),
    ]
    for w in batches:                       # two calls in a row
        want = _decode_with_workspace(P, w, 512)
        got = torch.full_like(want, float("nan"))
        assert _decode_static(P, w, got, 512) == P.PKV_OK
        err = (got.double() - want.double()).abs().max().item()
        assert err <= TOL_SAME_PATH, err
        assert P.pkv_get_device_error() == 0


def test_static_workspace_rejects_requests_larger_than_the_array():
    P = pkv()
    w = workloads.build("noalloc_big", dtype="f16", num_q_heads=40, num_kv_heads=40, head_dim=128,
                        block_size=16, context_lens=[4096] * 8, seed=23, device=DEV)
    need = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, w.max_context_len,
                                        16)
    assert need > P.STATIC_WORKSPACE_BYTES
    out = torch.zeros((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32, device=DEV)
    assert _decode_static(P, w, out, 16) == P.PKV_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0       # nothing was launched
