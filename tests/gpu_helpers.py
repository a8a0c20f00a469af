"""Shared helpers for the GPU parity tests: move workloads between the CUDA path
(through the C ABI binding) and the oracle (host numpy copies)."""
import numpy as np
import torch

import oracle
from paged_kv_cache_293_gb300 import workloads

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}


def pkv():
    from paged_kv_cache_293_gb300 import _build
    _build.build()
    from paged_kv_cache_293_gb300 import pagedkv
    return pagedkv


def dev_i32(a, device="cuda"):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=device)


def host(t):
    return workloads.storage_numpy(t)


def compact_for_oracle(w, seqs, block_tables=None):
    """Host copies of just the blocks the chosen sequences use, with their table rows renumbered
    into the compact pool (physical placement does not change the result)."""
    bt = w.block_tables if block_tables is None else block_tables
    seqs = np.asarray(seqs)
    rows = bt[seqs]
    ctx = w.context_lens[seqs]
    nb = workloads.blocks_for(ctx, w.block_size)
    used = np.unique(np.concatenate([rows[i, :nb[i]] for i in range(len(seqs))]))
    idx = torch.as_tensor(used, dtype=torch.long, device=w.k_pool.device)
    k = host(w.k_pool.index_select(0, idx))
    v = host(w.v_pool.index_select(0, idx))
    new_rows = np.full_like(rows, -1)
    for i in range(len(seqs)):
        new_rows[i, :nb[i]] = np.searchsorted(used, rows[i, :nb[i]])
    q = host(w.q)[seqs]
    return k, v, new_rows.astype(np.int32), ctx, q


def max_abs(gpu, ref):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


def check_allocator_invariants(free_ids, free_count, refcount, tables, lens, block_size):
    """Counts equal the table references of the live positions; the free stack holds exactly
    the unreferenced blocks, each once."""
    N = refcount.size
    refs = np.zeros(N, np.int64)
    for s, L in enumerate(lens):
        nb = -(-int(L) // block_size)
        row = tables[s, :nb]
        assert np.all((row >= 0) & (row < N)), "sequence %d has a bad table entry" % s
        np.add.at(refs, row, 1)
    assert np.array_equal(refs, refcount.astype(np.int64))
    n = int(free_count)
    free = np.sort(free_ids[:n])
    assert np.array_equal(free, np.flatnonzero(refs == 0)), "free stack != unreferenced blocks"
