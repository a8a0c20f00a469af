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


class OracleStep:
    """The oracle's side of one decode step, taken from host copies made BEFORE the GPU step,
    so that nothing the CUDA path writes ever feeds the oracle.

    It copies the blocks the chosen sequences use (plus `extra_blocks`, e.g. copy-on-write
    targets) into a compact host pool, renumbers the table rows into it (physical placement
    does not change the result), and applies the oracle's own slot mapping and cache write
    of each sequence's new token (its K/V rows at position ctx - 1) to those copies.
    Afterwards `check_pools` compares the GPU pool's same blocks bit for bit, `decode` runs
    the oracle's attention on the oracle-written copies, and `device_expected_pools` gives
    the whole expected pool on the device (the untouched blocks from a device clone taken
    before the step, the touched ones from the oracle)."""

    def __init__(self, w, seqs=None, extra_blocks=(), keep_device_clone=False):
        seqs = np.arange(w.num_seqs) if seqs is None else np.asarray(seqs)
        self.seqs, self.dtype, self.scale, self.B = seqs, w.dtype, w.scale, w.block_size
        rows = w.block_tables[seqs]
        self.ctx = w.context_lens[seqs]
        nb = workloads.blocks_for(self.ctx, w.block_size)
        used = np.unique(np.concatenate([rows[i, :nb[i]] for i in range(len(seqs))]
                                        + [np.asarray(extra_blocks, np.int64)]).astype(np.int64))
        self.used = used
        self.idx = torch.as_tensor(used, dtype=torch.long, device=w.k_pool.device)
        self.k = host(w.k_pool.index_select(0, self.idx)).copy()
        self.v = host(w.v_pool.index_select(0, self.idx)).copy()
        self.clone = (w.k_pool.clone(), w.v_pool.clone()) if keep_device_clone else None
        compact = np.full_like(rows, -1)
        for i in range(len(seqs)):
            compact[i, :nb[i]] = np.searchsorted(used, rows[i, :nb[i]])
        self.bt = compact.astype(np.int32)
        self.q = host(w.q)[seqs]
        # slots in the whole pool (what the GPU reports) and in the compact copy
        self.slots = oracle.slot_mapping(rows, w.positions[seqs], w.block_size)
        self._cslots = oracle.slot_mapping(self.bt, w.positions[seqs], w.block_size)
        self._k_new = host(w.k_new)[seqs]
        self._v_new = host(w.v_new)[seqs]

    def compact_ids(self, ids):
        ids = np.asarray(ids, np.int64)
        pos = np.searchsorted(self.used, ids)
        assert np.all(self.used[pos] == ids), "block outside the compact pool"
        return pos.astype(np.int32)

    def copy_blocks(self, pairs):
        """The oracle's copy-on-write copy of (src, dst) pool blocks on the compact copy."""
        pairs = np.asarray(pairs, np.int32).reshape(-1, 2)
        oracle.copy_blocks(self.k, self.v,
                           np.stack([self.compact_ids(pairs[:, 0]), self.compact_ids(pairs[:, 1])],
                                    1).astype(np.int32))

    def write(self):
        """The oracle's cache write of the new tokens into the compact copy."""
        oracle.kv_cache_write(self.dtype, self.k, self.v, self._k_new, self._v_new, self._cslots)

    def check_pools(self, w):
        """The GPU pool's copies of the same blocks equal the oracle's, bit for bit."""
        assert np.array_equal(host(w.k_pool.index_select(0, self.idx)), self.k)
        assert np.array_equal(host(w.v_pool.index_select(0, self.idx)), self.v)

    def check_whole_pools(self, w):
        """Every other block of the GPU pools is as it was before the step."""
        k, v = self.clone
        dev = k.device
        as_t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        k.index_copy_(0, self.idx, as_t(self.k).view(k.dtype).to(dev))
        v.index_copy_(0, self.idx, as_t(self.v).view(v.dtype).to(dev))
        assert torch.equal(k, w.k_pool) and torch.equal(v, w.v_pool)
        self.clone = None

    def decode(self):
        return oracle.paged_decode(self.dtype, self.k, self.v, self.q, self.bt, self.ctx,
                                   self.scale)


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
