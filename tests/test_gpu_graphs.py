"""The decode-step calls captured into a CUDA graph and replayed, as a serving loop
does for its decode steps: every launch of a call is enqueued on the caller's stream
with no host synchronisation and no allocation, so a captured call replays with new
inputs (the same buffers, new contents) and gives what a direct call gives."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_293_gb300 import workloads
from gpu_helpers import TOL, dev_i32, host, max_abs, pkv

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    return pkv()


def _capture(fn):
    """Capture fn() (after one direct warm-up call, which does the library's one-time
    set-up) into a graph on a side stream."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("dtype,Hq,Hkv,psize", [("f16", 8, 8, 512), ("bf16", 32, 8, 0)])
def test_fused_decode_step_replays_from_a_graph(P, dtype, Hq, Hkv, psize):
    """Append + attention + merge (partitions of 512 tokens for the first case)."""
    w = workloads.build("graph", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                        block_size=16, context_lens=[1, 700, 1500, 33, 2048], seed=61,
                        device=DEV)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    bt, cl = dev_i32(w.block_tables), dev_i32(w.context_lens)
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, Hq, mcl, psize)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.zeros((w.num_seqs, Hq, 128), dtype=torch.float32, device=DEV)
    slots = torch.zeros(w.num_seqs, dtype=torch.int64, device=DEV)

    def step():
        P.pkv_paged_attention_decode_append(w.q, w.k_pool, w.v_pool, w.k_new, w.v_new, bt, cl,
                                            w.scale, out, mcl, psize, ws, slot_mapping=slots)

    g = _capture(step)
    gen = torch.Generator(device=DEV).manual_seed(9)
    tdt = workloads.TORCH_DTYPE[dtype]
    for _ in range(3):
        w.q.copy_(torch.randn(w.q.shape, generator=gen, device=DEV).to(tdt))
        w.k_new.copy_(torch.randn(w.k_new.shape, generator=gen, device=DEV).to(tdt))
        w.v_new.copy_(torch.randn(w.v_new.shape, generator=gen, device=DEV).to(tdt))
        w.k_pool.copy_(k0)
        w.v_pool.copy_(v0)
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        got, got_k, got_v = out.clone(), w.k_pool.clone(), w.v_pool.clone()
        w.k_pool.copy_(k0)
        w.v_pool.copy_(v0)
        out.zero_()
        step()
        torch.cuda.synchronize()
        assert torch.equal(got, out)
        assert torch.equal(got_k, w.k_pool) and torch.equal(got_v, w.v_pool)
    ref = oracle.paged_decode(dtype, host(w.k_pool), host(w.v_pool), host(w.q), w.block_tables,
                              w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL[dtype]
    assert P.pkv_get_device_error() == 0


def test_cascade_replays_from_a_graph(P):
    """Suffix decode, prefix pass behind it (programmatic dependent launch) and merge."""
    ctx = [200, 260, 333, 1000, 129, 700]
    w = workloads.build("graph_cascade", dtype="bf16", num_q_heads=32, num_kv_heads=8,
                        head_dim=128, block_size=16, context_lens=ctx, seed=62, device=DEV,
                        shared_prefix_blocks=8)
    prefix = 8 * 16
    bt, cl = dev_i32(w.block_tables), dev_i32(w.context_lens)
    mcl = w.max_context_len
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 32, mcl,
                                                          prefix, 0), DEV)
    out = torch.zeros((w.num_seqs, 32, 128), dtype=torch.float32, device=DEV)

    def step():
        P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, bt, cl, w.scale, out, mcl,
                                             prefix, ws)

    g = _capture(step)
    gen = torch.Generator(device=DEV).manual_seed(10)
    for _ in range(3):
        w.q.copy_(torch.randn(w.q.shape, generator=gen, device=DEV).to(torch.bfloat16))
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        out.zero_()
        step()
        torch.cuda.synchronize()
        assert torch.equal(got, out)
    ref = oracle.paged_decode("bf16", host(w.k_pool), host(w.v_pool), host(w.q), w.block_tables,
                              w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL["bf16"]
    assert P.pkv_get_device_error() == 0


def test_multi_query_append_replays_from_a_graph(P):
    w = workloads.build("graph_multi", dtype="f16", num_q_heads=16, num_kv_heads=8,
                        head_dim=128, block_size=16, context_lens=[40, 1300, 17, 2500], seed=63,
                        device=DEV)
    nq, S = 4, w.num_seqs
    gen = torch.Generator(device=DEV).manual_seed(11)
    q = torch.randn((S, nq, 16, 128), generator=gen, device=DEV).half()
    kn = torch.randn((S, nq, 8, 128), generator=gen, device=DEV).half()
    vn = torch.randn_like(kn)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    bt, cl = dev_i32(w.block_tables), dev_i32(w.context_lens)
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, S * nq, 16, mcl, 1024)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.zeros((S, nq, 16, 128), dtype=torch.float32, device=DEV)

    def step():
        P.pkv_paged_attention_decode_multi_append(q, w.k_pool, w.v_pool, kn, vn, bt, cl, w.scale,
                                                  out, mcl, 1024, ws)

    g = _capture(step)
    for _ in range(2):
        q.copy_(torch.randn(q.shape, generator=gen, device=DEV).half())
        kn.copy_(torch.randn(kn.shape, generator=gen, device=DEV).half())
        w.k_pool.copy_(k0)
        w.v_pool.copy_(v0)
        g.replay()
        torch.cuda.synchronize()
        got, got_k = out.clone(), w.k_pool.clone()
        w.k_pool.copy_(k0)
        w.v_pool.copy_(v0)
        step()
        torch.cuda.synchronize()
        assert torch.equal(got, out) and torch.equal(got_k, w.k_pool)
    ref = oracle.paged_decode_multi("f16", host(w.k_pool), host(w.v_pool), host(q),
                                    w.block_tables, w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL["f16"]
    assert P.pkv_get_device_error() == 0
