"""Device-side block bookkeeping against the sequential oracle (GPU).

Which free id a request gets depends on the order the GPU serves the atomics
in, so ids are not compared.  What is unique is: statuses, how many blocks are
taken, the multiset of reference counts, and every sequence's contents; the rest must be valid: counts equal table references and the free
stack holds exactly the unreferenced blocks.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_293_gb300 import workloads
from gpu_helpers import check_allocator_invariants, dev_i32, host, pkv

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    return pkv()


def state(alloc):
    return (alloc.free_ids.cpu().numpy(), int(alloc.free_count.item()),
            alloc.refcount.cpu().numpy())


def test_prefill_fork_append_free_cycle(P):
    B, N, M, S = 16, 600, 40, 12
    rng = np.random.default_rng(7)
    w = workloads.build("alloc", dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                        block_size=B, context_lens=[1], seed=3, device=DEV, num_blocks=N)
    w.k_pool.normal_()
    w.v_pool.normal_()
    alloc = P.BlockAllocator(N, DEV)
    P.pkv_allocator_reset(alloc)
    ref = oracle.Allocator(N)
    tables = torch.full((S, M), -1, dtype=torch.int32, device=DEV)
    ref_tables = np.full((S, M), -1, np.int32)
    status = torch.empty(S, dtype=torch.int32, device=DEV)
    kh, vh = host(w.k_pool).copy(), host(w.v_pool).copy()

    # 1. prefill sequences 0..5; 6..11 stay empty
    lens = np.zeros(S, np.int32)
    lens[:6] = rng.integers(1, 300, 6)
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(np.zeros(S)),
                              dev_i32(lens), status)
    st_ref = ref.allocate_for_append(kh, vh, B, ref_tables, np.zeros(S), lens)
    torch.cuda.synchronize()
    assert np.array_equal(status.cpu().numpy(), st_ref)
    fi, fc, rc = state(alloc)
    assert fc == int(ref.free_count[0]) == N - int(sum(-(-L // B) for L in lens))
    check_allocator_invariants(fi, fc, rc, tables.cpu().numpy(), lens, B)

    # 2. sequences 6, 7, 8 share sequence 0's blocks; 9 shares sequence 1's
    pairs = np.array([[0, 6], [0, 7], [0, 8], [1, 9]], np.int32)
    flens = lens[pairs[:, 0]]
    P.pkv_fork_sequences(alloc, B, tables, dev_i32(pairs), dev_i32(flens))
    ref.fork(B, ref_tables, pairs, flens)
    lens[pairs[:, 1]] = flens
    torch.cuda.synchronize()
    fi, fc, rc = state(alloc)
    check_allocator_invariants(fi, fc, rc, tables.cpu().numpy(), lens, B)
    assert fc == int(ref.free_count[0])

    # 3. every live sequence appends 1..20 tokens, except 8 (a holder that stays put):
    #    holders of a shared partly filled block copy it, the last reference keeps it
    q = torch.randn((S, 8, 128), device=DEV).to(torch.bfloat16)
    live = lens > 0
    before = oracle.paged_decode("bf16", host(w.k_pool), host(w.v_pool), host(q)[live],
                                 tables.cpu().numpy()[live], lens[live], 0.1)
    grow = np.where(live, rng.integers(1, 21, S), 0).astype(np.int32)
    grow[8] = 0
    new = (lens + grow).astype(np.int32)
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(lens), dev_i32(new),
                              status)
    st_ref = ref.allocate_for_append(kh, vh, B, ref_tables, lens, new)
    torch.cuda.synchronize()
    assert np.array_equal(status.cpu().numpy(), st_ref) and np.all(st_ref == 0)
    fi, fc, rc = state(alloc)
    assert fc == int(ref.free_count[0])                     # same number of blocks taken
    # the ids differ from the oracle's, the multiset of counts does not
    assert np.array_equal(np.sort(rc), np.sort(ref.refcount))
    check_allocator_invariants(fi, fc, rc, tables.cpu().numpy(), new, B)
    after = oracle.paged_decode("bf16", host(w.k_pool), host(w.v_pool), host(q)[live],
                                tables.cpu().numpy()[live], lens[live], 0.1)
    assert np.array_equal(before, after)                    # nobody's tokens moved or changed

    # 4. everything back
    P.pkv_free_sequences(alloc, B, tables, dev_i32(np.arange(S)), dev_i32(new))
    torch.cuda.synchronize()
    fi, fc, rc = state(alloc)
    assert fc == N and np.all(rc == 0) and np.array_equal(np.sort(fi), np.arange(N))
    assert torch.all(tables == -1)
    assert P.pkv_get_device_error() == 0


def test_running_out_of_blocks_reports_and_stays_consistent(P):
    B, N, M, S = 16, 20, 8, 4
    w = workloads.build("short", dtype="f16", num_q_heads=4, num_kv_heads=4, head_dim=64,
                        block_size=B, context_lens=[1], seed=1, device=DEV, num_blocks=N)
    alloc = P.BlockAllocator(N, DEV)
    P.pkv_allocator_reset(alloc)
    tables = torch.full((S, M), -1, dtype=torch.int32, device=DEV)
    status = torch.empty(S, dtype=torch.int32, device=DEV)
    want = np.array([100, 100, 100, 100], np.int32)         # 7 blocks each, 28 > 20
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(np.zeros(S)),
                              dev_i32(want), status)
    torch.cuda.synchronize()
    st = status.cpu().numpy()
    fi, fc, rc = state(alloc)
    assert fc == 0 and np.all(np.isin(st, [0, 1])) and np.sum(st == 1) >= 1
    tb = tables.cpu().numpy()
    got = (tb >= 0).sum(axis=1)
    assert got.sum() == N and np.all(got[st == 0] == 7)
    for s in range(S):                                       # allocated entries form a prefix
        assert np.all(tb[s, :got[s]] >= 0) and np.all(tb[s, got[s]:] == -1)
    check_allocator_invariants(fi, fc, rc, tb, got * B, B)
    # an impossible request (table row too short) is refused for that sequence alone
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(got * B),
                              dev_i32(got * B + np.array([0, 0, 0, 1000])), status)
    torch.cuda.synchronize()
    assert status.cpu().numpy()[3] == 2
    assert P.pkv_get_device_error() == 0


def test_one_decode_step_driven_by_the_device_allocator(P):
    """Allocate for each sequence's new token on the device, then slot mapping, cache write
    and decode: the result equals the oracle's run of the same step."""
    B, N, M = 16, 400, 64
    lens = np.array([15, 16, 17, 300, 1, 32], np.int32)
    S = len(lens)
    w = workloads.build("step", dtype="f16", num_q_heads=8, num_kv_heads=8, head_dim=128,
                        block_size=B, context_lens=[1], seed=9, device=DEV, num_blocks=N)
    w.k_pool.normal_()
    w.v_pool.normal_()
    alloc = P.BlockAllocator(N, DEV)
    P.pkv_allocator_reset(alloc)
    tables = torch.full((S, M), -1, dtype=torch.int32, device=DEV)
    status = torch.empty(S, dtype=torch.int32, device=DEV)
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(np.zeros(S)),
                              dev_i32(lens), status)
    new = lens + 1
    P.pkv_allocate_for_append(alloc, w.k_pool, w.v_pool, tables, dev_i32(lens), dev_i32(new),
                              status)
    slots = torch.empty(S, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(tables, dev_i32(lens), B, slots)     # the new token's position = old length
    k_new = torch.randn((S, 8, 128), device=DEV).half()
    v_new = torch.randn((S, 8, 128), device=DEV).half()
    q = torch.randn((S, 8, 128), device=DEV).half()
    kh, vh = host(w.k_pool).copy(), host(w.v_pool).copy()
    P.pkv_kv_cache_write(w.k_pool, w.v_pool, k_new, v_new, slots)
    out = torch.empty((S, 8, 128), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode(q, w.k_pool, w.v_pool, tables, dev_i32(new), w.scale, out,
                                 int(new.max()))
    torch.cuda.synchronize()
    assert np.all(status.cpu().numpy() == 0)
    tb = tables.cpu().numpy()
    ref_slots = oracle.slot_mapping(tb, lens, B)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    oracle.kv_cache_write("f16", kh, vh, host(k_new), host(v_new), ref_slots)
    ref = oracle.paged_decode("f16", kh, vh, host(q), tb, new, w.scale)
    assert float(np.abs(out.double().cpu().numpy() - ref).max()) <= 2e-3
    assert P.pkv_get_device_error() == 0
