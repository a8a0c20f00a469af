"""Host-side batch helpers of the workload module (CPU only)."""
import numpy as np

from paged_kv_cache_293_gb300 import workloads


def test_shortest_last_order():
    rng = np.random.default_rng(3)
    ctx = rng.integers(1, 5000, size=103)
    o = workloads.shortest_last_order(ctx, 0.2)
    assert sorted(o.tolist()) == list(range(103))
    k = round(0.2 * 103)
    tail, head = o[-k:], o[:-k]
    assert np.all(np.diff(ctx[tail]) <= 0)                   # longest of the short ones first
    assert ctx[tail].max() <= ctx[head].min()                # the shortest fifth
    assert np.all(np.diff(head) > 0)                         # the others in the given order
    assert np.array_equal(workloads.shortest_last_order(ctx, 0.0), np.arange(103))


def test_reorder_moves_every_per_sequence_input_together():
    w = workloads.build("re", dtype="f16", num_q_heads=4, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=[40, 300, 17, 90, 33, 64, 129, 16],
                        seed=5, shared_prefix_blocks=1, cow_fraction=0.5)
    o = workloads.shortest_last_order(w.context_lens, 0.25)
    r = workloads.reorder(w, o)
    assert np.array_equal(r.context_lens, w.context_lens[o])
    assert np.array_equal(r.block_tables, w.block_tables[o])
    assert np.array_equal(r.positions, w.positions[o])
    for name in ("q", "k_new", "v_new"):
        assert np.array_equal(workloads.storage_numpy(getattr(r, name)),
                              workloads.storage_numpy(getattr(w, name))[o])
    assert np.array_equal(r.block_tables_after_cow(), w.block_tables_after_cow()[o])
    assert r.k_pool is w.k_pool and r.v_pool is w.v_pool
