"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test ties the oracle to something it does not compute itself: a library
routine on a special case (dense attention from torch, float conversions from
numpy / torch), the pages' worked numbers (fixtures under tests/golden/),
closed forms, and invariants the pages fix (physical placement does not
matter; shared blocks behave like private copies).  The planted-mistake test
in test_oracle_mutants.py checks that plausible mistakes in oracle.c fail here.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_293_gb300 import accounting, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ helpers (test-side only)

def rand_storage(rng, shape, dtype):
    """(element storage for the oracle, exact float64 values) of N(0,1) draws."""
    x = rng.standard_normal(shape).astype(np.float32)
    if dtype == "f32":
        return x, x.astype(np.float64)
    if dtype == "f16":
        h = x.astype(np.float16)
        return h.view(np.uint16), h.astype(np.float64)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.to(torch.float64).numpy()


def paged_from_dense(dense, tables, B, N):
    """Lay dense per-sequence rows [ctx][Hkv][D] out as a pool [N][Hkv][B][D] by padding each
    sequence to whole blocks, cutting it into [blocks][B][Hkv][D] and moving the head axis
    in front of the row axis; block j of sequence s goes to physical block tables[s][j]."""
    Hkv, D = dense[0].shape[1:]
    pool = np.zeros((N, Hkv, B, D), dtype=dense[0].dtype)
    for s, rows in enumerate(dense):
        ctx = rows.shape[0]
        nb = -(-ctx // B)
        padded = np.zeros((nb * B, Hkv, D), dtype=rows.dtype)
        padded[:ctx] = rows
        pool[tables[s, :nb]] = padded.reshape(nb, B, Hkv, D).transpose(0, 2, 1, 3)
    return pool


def random_case(rng, dtype, ctx, Hq, Hkv, D, B, extra_blocks=3):
    """Dense K/V (storage + exact), q, and a random physical placement."""
    S = len(ctx)
    nb = [-(-c // B) for c in ctx]
    N = sum(nb) + extra_blocks
    perm = rng.permutation(N)
    M = max(max(nb), 1)
    tables = np.full((S, M), -1, np.int32)
    cur = 0
    for s in range(S):
        tables[s, :nb[s]] = perm[cur:cur + nb[s]]
        cur += nb[s]
    ks, kx, vs, vx = [], [], [], []
    for c in ctx:
        a, ax = rand_storage(rng, (c, Hkv, D), dtype)
        b, bx = rand_storage(rng, (c, Hkv, D), dtype)
        ks.append(a); kx.append(ax); vs.append(b); vx.append(bx)
    qs, qx = rand_storage(rng, (S, Hq, D), dtype)
    k_pool = paged_from_dense(ks, tables, B, N)
    v_pool = paged_from_dense(vs, tables, B, N)
    return dict(k_pool=k_pool, v_pool=v_pool, q=qs, qx=qx, kx=kx, vx=vx, tables=tables,
                ctx=np.asarray(ctx, np.int32), N=N)


def dense_attention_torch(qx, kx, vx, scale, G):
    """torch's scaled_dot_product_attention in float64 on the dense rows of one sequence."""
    q = torch.from_numpy(qx)[:, None, :]                       # [Hq, 1, D]
    K = torch.from_numpy(kx).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, ctx, D]
    V = torch.from_numpy(vx).permute(1, 0, 2).repeat_interleave(G, dim=0)
    out = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
    return out[:, 0, :].numpy()


# ------------------------------------------------------------------ element conversions

def test_f16_conversion_matches_numpy_on_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.convert_to_double("f16", bits)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_conversion_matches_torch_on_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.convert_to_double("bf16", bits)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# ------------------------------------------------------------------ attention vs library

CASES = [
    # dtype, ctx, Hq, Hkv, D, B
    ("f32", [1, 17, 50, 100], 4, 4, 64, 16),
    ("f16", [5, 16, 33, 64], 8, 2, 128, 16),
    ("bf16", [31, 32, 70], 8, 8, 64, 32),
    ("f16", [40, 3], 4, 1, 128, 32),
]


@pytest.mark.parametrize("dtype,ctx,Hq,Hkv,D,B", CASES)
def test_decode_equals_dense_sdpa(dtype, ctx, Hq, Hkv, D, B):
    rng = np.random.default_rng(11)
    c = random_case(rng, dtype, ctx, Hq, Hkv, D, B)
    scale = float(np.float32(0.37))
    got = oracle.paged_decode(dtype, c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], scale)
    for s in range(len(ctx)):
        want = dense_attention_torch(c["qx"][s], c["kx"][s], c["vx"][s], scale, Hq // Hkv)
        np.testing.assert_allclose(got[s], want, rtol=0, atol=1e-12)


def test_single_block_equals_textbook_softmax():
    """One block with B >= ctx: paged decode is dense softmax(qK^T * scale) V (scipy softmax)."""
    from scipy.special import softmax
    rng = np.random.default_rng(5)
    c = random_case(rng, "f32", [13], 2, 2, 64, 16)
    scale = float(np.float32(0.125))
    got = oracle.paged_decode("f32", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], scale)
    K, V, q = c["kx"][0], c["vx"][0], c["qx"][0]
    for h in range(2):
        w = softmax(scale * (K[:, h, :] @ q[h]))
        np.testing.assert_allclose(got[0, h], w @ V[:, h, :], rtol=0, atol=1e-13)


# ------------------------------------------------------------------ special cases with exact answers

def test_context_of_one_returns_that_value_row():
    rng = np.random.default_rng(1)
    c = random_case(rng, "f16", [1, 1, 1], 4, 2, 128, 16)
    got = oracle.paged_decode("f16", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.088)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(got[s, h], c["vx"][s][0, h // 2])


def test_equal_value_rows_return_that_row():
    rng = np.random.default_rng(2)
    c = random_case(rng, "f32", [37, 64], 2, 2, 64, 16)
    row = rng.standard_normal(64).astype(np.float32)
    v_pool = np.broadcast_to(row, c["v_pool"].shape).copy()
    got = oracle.paged_decode("f32", c["k_pool"], v_pool, c["q"], c["tables"], c["ctx"], 0.5)
    np.testing.assert_allclose(got, np.broadcast_to(row.astype(np.float64), got.shape),
                               rtol=4e-16 * 64, atol=0)


def test_zero_query_gives_mean_of_values():
    """All scores equal -> uniform weights -> the mean of the cached V rows."""
    rng = np.random.default_rng(3)
    c = random_case(rng, "bf16", [29, 48], 4, 4, 64, 16)
    q0 = np.zeros_like(c["q"])
    got = oracle.paged_decode("bf16", c["k_pool"], c["v_pool"], q0, c["tables"], c["ctx"], 1.0)
    for s in range(2):
        np.testing.assert_allclose(got[s], c["vx"][s].mean(axis=0), rtol=0, atol=1e-14)


def test_dominant_key_selects_its_value_row():
    """A key far more aligned with q than the rest takes all the weight."""
    rng = np.random.default_rng(4)
    ctx, D = 20, 64
    k = np.zeros((ctx, 1, D), np.float32)
    k[7, 0, 0] = 1.0
    v = rng.standard_normal((ctx, 1, D)).astype(np.float32)
    tables = np.array([[1, 0]], np.int32)
    k_pool = paged_from_dense([k], tables, 16, 2)
    v_pool = paged_from_dense([v], tables, 16, 2)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    got = oracle.paged_decode("f32", k_pool, v_pool, q, tables, [ctx], 2000.0)
    np.testing.assert_array_equal(got[0, 0], v[7, 0].astype(np.float64))


def test_empty_context_gives_zeros():
    rng = np.random.default_rng(6)
    c = random_case(rng, "f16", [0, 5], 2, 1, 64, 16)
    got = oracle.paged_decode("f16", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.1)
    assert np.all(got[0] == 0.0)
    assert np.all(np.isfinite(got[1]))


# ------------------------------------------------------------------ invariants the pages fix

def test_physical_permutation_leaves_output_unchanged():
    """Blocks may live anywhere in the pool: moving them (and their table entries) is a no-op."""
    rng = np.random.default_rng(7)
    c = random_case(rng, "f16", [45, 100, 16], 4, 4, 128, 16, extra_blocks=5)
    base = oracle.paged_decode("f16", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.09)
    perm = rng.permutation(c["N"])             # old physical id -> new physical id
    kp = np.empty_like(c["k_pool"]); kp[perm] = c["k_pool"]
    vp = np.empty_like(c["v_pool"]); vp[perm] = c["v_pool"]
    tables = np.where(c["tables"] >= 0, perm[np.maximum(c["tables"], 0)], -1).astype(np.int32)
    moved = oracle.paged_decode("f16", kp, vp, c["q"], tables, c["ctx"], 0.09)
    assert np.array_equal(base, moved)


def test_shared_prefix_blocks_equal_private_copies():
    w = workloads.build("shared", dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=[70, 90, 64], seed=3,
                        shared_prefix_blocks=4, num_blocks=40)
    k = workloads.storage_numpy(w.k_pool).copy()
    v = workloads.storage_numpy(w.v_pool).copy()
    q = workloads.storage_numpy(w.q)
    shared = oracle.paged_decode("bf16", k, v, q, w.block_tables, w.context_lens, w.scale)
    # give every sequence its own copy of the prefix blocks
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    bt = w.block_tables.copy()
    for s in range(1, w.num_seqs):
        for j in range(4):
            dst = free.pop()
            k[dst] = k[bt[s, j]]
            v[dst] = v[bt[s, j]]
            bt[s, j] = dst
    assert len(set(bt[:, :4].ravel().tolist())) == 4 * w.num_seqs
    private = oracle.paged_decode("bf16", k, v, q, bt, w.context_lens, w.scale)
    assert np.array_equal(shared, private)


def test_copy_on_write_then_redirect_is_a_no_op():
    w = workloads.build("cow", dtype="bf16", num_q_heads=4, num_kv_heads=4, head_dim=64,
                        block_size=16, context_lens=[40, 50, 33, 64], seed=9,
                        shared_prefix_blocks=2, cow_fraction=0.5)
    k = workloads.storage_numpy(w.k_pool).copy()
    v = workloads.storage_numpy(w.v_pool).copy()
    q = workloads.storage_numpy(w.q)
    before = oracle.paged_decode("bf16", k, v, q, w.block_tables, w.context_lens, w.scale)
    k0, v0 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, w.cow_pairs)
    for src, dst in w.cow_pairs:
        assert np.array_equal(k[dst], k[src]) and np.array_equal(v[dst], v[src])
    untouched = np.setdiff1d(np.arange(w.num_blocks), w.cow_pairs[:, 1])
    assert np.array_equal(k[untouched], k0[untouched]) and np.array_equal(v[untouched], v0[untouched])
    after = oracle.paged_decode("bf16", k, v, q, w.block_tables_after_cow(), w.context_lens, w.scale)
    assert np.array_equal(before, after)


def test_grouped_query_equals_mha_on_repeated_kv_heads():
    """G q heads per kv head = plain multi-head attention with each kv head repeated G times."""
    rng = np.random.default_rng(8)
    G = 4
    c = random_case(rng, "f16", [30, 77], 8, 2, 64, 16)
    gqa = oracle.paged_decode("f16", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.2)
    k_rep = np.repeat(c["k_pool"], G, axis=1)
    v_rep = np.repeat(c["v_pool"], G, axis=1)
    mha = oracle.paged_decode("f16", k_rep, v_rep, c["q"], c["tables"], c["ctx"], 0.2)
    assert np.array_equal(gqa, mha)


# ------------------------------------------------------------------ partitions and their merge

@pytest.mark.parametrize("P", [16, 48, 64, 512])
def test_partition_merge_equals_whole_context(P):
    rng = np.random.default_rng(12)
    c = random_case(rng, "f32", [1, 47, 200, 130], 4, 2, 64, 16)
    whole = oracle.paged_decode("f32", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.3)
    m, l, o = oracle.partition_decode("f32", c["k_pool"], c["v_pool"], c["q"], c["tables"],
                                      c["ctx"], 0.3, P)
    merged = oracle.lse_merge(m, l, o)
    np.testing.assert_allclose(merged, whole, rtol=0, atol=1e-13)
    # empty ranges carry no weight
    parts = -(-c["ctx"] // P)
    for s in range(4):
        assert np.all(l[s, :, parts[s]:] == 0) and np.all(np.isneginf(m[s, :, parts[s]:]))


def test_single_partition_holds_max_and_normaliser():
    """With one range covering the context: m = the largest score, o / l = the output."""
    rng = np.random.default_rng(13)
    c = random_case(rng, "f32", [25], 2, 2, 64, 16)
    scale = 0.25
    m, l, o = oracle.partition_decode("f32", c["k_pool"], c["v_pool"], c["q"], c["tables"],
                                      c["ctx"], scale, 32)
    K, q = c["kx"][0], c["qx"][0]
    for h in range(2):
        x = scale * (K[:, h, :] @ q[h])
        assert m[0, h, 0] == pytest.approx(x.max(), abs=1e-13)
        assert l[0, h, 0] == pytest.approx(np.exp(x - x.max()).sum(), rel=1e-13)
    whole = oracle.paged_decode("f32", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], scale)
    np.testing.assert_allclose(o[0, :, 0] / l[0, :, 0][:, None], whole[0], atol=1e-13, rtol=0)


def test_merge_of_hand_made_partials():
    """Two ranges with known (m, l, o): the merge weights them by exp(m_k - M)."""
    D = 4
    m = np.array([[0.0, math.log(3.0)]])
    l = np.array([[2.0, 1.0]])
    o = np.array([[[2.0, 0, 0, 4.0], [0, 1.0, 0, 1.0]]])
    # exp weights 1 and 3: numerator = o0 + 3 o1, denominator = 2 + 3
    want = (o[0, 0] + 3 * o[0, 1]) / 5.0
    got = oracle.lse_merge(m, l, o)
    np.testing.assert_allclose(got[0], want, atol=1e-15)
    assert got.shape == (1, D)


# ------------------------------------------------------------------ slot mapping and the write

@pytest.mark.parametrize("dtype,B", [("f16", 16), ("f32", 32), ("bf16", 16)])
def test_token_by_token_append_rebuilds_the_dense_sequence(dtype, B):
    """Appending each token through slot mapping + write, then laying the pool out the dense
    way, gives back the sequence; the blocks are allocated one at a time as tokens arrive."""
    rng = np.random.default_rng(21)
    Hkv, D, S = 2, 64, 3
    ctx = [B * 2 + 5, 1, B * 3]
    N = 20
    free = list(rng.permutation(N))
    M = 4
    tables = np.full((S, M), -1, np.int32)
    k_dense = [rand_storage(rng, (c, Hkv, D), dtype)[0] for c in ctx]
    v_dense = [rand_storage(rng, (c, Hkv, D), dtype)[0] for c in ctx]
    edt = k_dense[0].dtype
    k_pool = np.zeros((N, Hkv, B, D), edt)
    v_pool = np.zeros((N, Hkv, B, D), edt)
    for p in range(max(ctx)):
        seqs = [s for s in range(S) if p < ctx[s]]
        for s in seqs:
            if p % B == 0:
                tables[s, p // B] = free.pop()
        pos = np.array([p] * len(seqs), np.int32)
        slots = oracle.slot_mapping(tables, pos, B, token_seq=np.array(seqs, np.int32))
        kn = np.stack([k_dense[s][p] for s in seqs])
        vn = np.stack([v_dense[s][p] for s in seqs])
        oracle.kv_cache_write(dtype, k_pool, v_pool, kn, vn, slots)
    assert np.array_equal(k_pool, paged_from_dense(k_dense, tables, B, N))
    assert np.array_equal(v_pool, paged_from_dense(v_dense, tables, B, N))


def test_negative_slots_are_skipped():
    k = np.arange(2 * 1 * 16 * 8, dtype=np.float32).reshape(2, 1, 16, 8)
    v = -k
    k0, v0 = k.copy(), v.copy()
    oracle.kv_cache_write("f32", k, v, np.ones((2, 1, 8), np.float32), np.ones((2, 1, 8), np.float32),
                          np.array([-1, -1], np.int64))
    assert np.array_equal(k, k0) and np.array_equal(v, v0)
    pos = oracle.slot_mapping(np.array([[1, 0]], np.int32), np.array([-1], np.int32), 16)
    assert pos.tolist() == [-1]


# ------------------------------------------------------------------ the pages' worked numbers

def test_hundred_token_sequence_reads_exactly_four_blocks():
    g = golden("hundred_tokens_four_blocks.json")
    B, n, blocks = g["block_size"], g["tokens"], g["blocks"]
    assert int(workloads.blocks_for(n, B)) == blocks
    rng = np.random.default_rng(0)
    k_pool = rng.standard_normal((8, 1, B, 64)).astype(np.float32)
    v_pool = rng.standard_normal((8, 1, B, 64)).astype(np.float32)
    q = rng.standard_normal((1, 1, 64)).astype(np.float32)
    table = np.array([[5, 2, 7, 0] + [-1] * 4], np.int32)      # nothing past block `blocks`
    out = oracle.paged_decode("f32", k_pool, v_pool, q, table, [n], 0.125)
    assert np.all(np.isfinite(out))
    short = table.copy()
    short[0, blocks - 1] = -1                                    # one block too few
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode("f32", k_pool, v_pool, q, short, [n], 0.125)


def test_toy_simulation_kv_slot_totals():
    g = golden("toy_kv_slots.json")
    lens = [g["prompt_tokens"] + n for n in g["output_lengths"]]
    assert workloads.allocated_slots(lens, g["block_size"]) == g["paged_slots"]
    assert len(lens) * g["naive_reserved_per_request"] == g["naive_slots"]
    # waste is confined to each sequence's last block
    waste = workloads.allocated_slots(lens, g["block_size"]) - sum(lens)
    assert 0 <= waste < len(lens) * g["block_size"]


def test_llama13b_kv_bytes_per_sequence():
    g = golden("llama13b_kv_per_sequence.json")
    per_tok = accounting.kv_bytes_per_token(g["kv_heads"], g["head_dim"], g["elem_bytes"])
    total = per_tok * g["layers"] * g["tokens"]
    assert abs(total / 1e9 - g["quoted_gb"]) <= g["quoted_precision_gb"]


def test_out_of_pool_block_is_an_error():
    k = np.zeros((2, 1, 16, 64), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode("f32", k, k, np.zeros((1, 1, 64), np.float32),
                            np.array([[3]], np.int32), [5], 1.0)


def test_swap_out_and_back_in_restores_the_pool():
    """Moving blocks to a second (host) pool and back into fresh blocks, then pointing the
    table at them, leaves decode unchanged; with one pool it is the block copy."""
    w = workloads.build("swap", dtype="f16", num_q_heads=4, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=[40, 70], seed=12, num_blocks=20)
    k = workloads.storage_numpy(w.k_pool).copy()
    v = workloads.storage_numpy(w.v_pool).copy()
    q = workloads.storage_numpy(w.q)
    before = oracle.paged_decode("f16", k, v, q, w.block_tables, w.context_lens, w.scale)
    used = w.block_tables[1, :5]
    hk = np.zeros((8,) + k.shape[1:], k.dtype)
    hv = np.zeros_like(hk)
    oracle.swap_blocks(k, v, hk, hv, np.stack([used, np.arange(5)], 1))
    assert np.array_equal(hk[:5], k[used]) and np.array_equal(hv[:5], v[used])
    free = np.setdiff1d(np.arange(20), w.block_tables[w.block_tables >= 0])[:5]
    k[used] = 0
    v[used] = 0
    oracle.swap_blocks(hk, hv, k, v, np.stack([np.arange(5), free], 1))
    bt = w.block_tables.copy()
    bt[1, :5] = free
    after = oracle.paged_decode("f16", k, v, q, bt, w.context_lens, w.scale)
    assert np.array_equal(before, after)
    k1, v1 = k.copy(), v.copy()
    pairs = np.array([[free[0], used[0]], [free[1], used[1]]], np.int32)
    oracle.copy_blocks(k, v, pairs)
    oracle.swap_blocks(k1.copy(), v1.copy(), k1, v1, pairs)
    assert np.array_equal(k, k1) and np.array_equal(v, v1)


# ------------------------------------------------------------------ several new tokens per sequence

@pytest.mark.parametrize("dtype,ctx,nq,Hq,Hkv,D,B", [
    ("f16", [20, 64, 9], 4, 8, 2, 64, 16),
    ("bf16", [33, 5], 3, 4, 4, 128, 32),
    ("f32", [3, 40], 5, 2, 1, 64, 16),       # first sequence: two queries see nothing
])
def test_multi_query_equals_causal_sdpa(dtype, ctx, nq, Hq, Hkv, D, B):
    """The tail queries against torch SDPA with an explicit causal mask over the dense rows."""
    rng = np.random.default_rng(14)
    c = random_case(rng, dtype, ctx, Hq, Hkv, D, B)
    qs, qx = rand_storage(rng, (len(ctx), nq, Hq, D), dtype)
    scale = float(np.float32(0.2))
    got = oracle.paged_decode_multi(dtype, c["k_pool"], c["v_pool"], qs, c["tables"], c["ctx"], scale)
    G = Hq // Hkv
    for s, L in enumerate(ctx):
        K = torch.from_numpy(c["kx"][s]).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        V = torch.from_numpy(c["vx"][s]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        q = torch.from_numpy(qx[s]).permute(1, 0, 2)                                  # [Hq, nq, D]
        pos = torch.arange(L)[None, :]
        lim = (L - nq + torch.arange(nq))[:, None]
        mask = pos <= lim                                                          # [nq, L]
        for j in range(nq):
            if L - nq + 1 + j <= 0:
                assert np.all(got[s, j] == 0)
                continue
            want = torch.nn.functional.scaled_dot_product_attention(
                q[:, j:j + 1], K, V, attn_mask=mask[j:j + 1], scale=scale)[:, 0].numpy()
            np.testing.assert_allclose(got[s, j], want, rtol=0, atol=1e-12)


def test_multi_query_with_one_query_is_decode():
    rng = np.random.default_rng(15)
    c = random_case(rng, "f16", [17, 90], 8, 2, 128, 16)
    one = oracle.paged_decode_multi("f16", c["k_pool"], c["v_pool"], c["q"][:, None], c["tables"],
                                    c["ctx"], 0.1)
    dec = oracle.paged_decode("f16", c["k_pool"], c["v_pool"], c["q"], c["tables"], c["ctx"], 0.1)
    assert np.array_equal(one[:, 0], dec)


# ------------------------------------------------------------------ block bookkeeping

def test_toy_simulation_blocks_allocated_token_by_token():
    """Growing the toy's eight requests (100 prompt tokens + their outputs) one token at a
    time allocates blocks holding exactly the 960 slots the page prints, ceil(len/16) each."""
    from gpu_helpers import check_allocator_invariants
    g = golden("toy_kv_slots.json")
    B = g["block_size"]
    lens = np.array([g["prompt_tokens"] + n for n in g["output_lengths"]], np.int32)
    N = 100
    alloc = oracle.Allocator(N)
    k = np.zeros((N, 1, B, 8), np.float32)
    tables = np.full((len(lens), 16), -1, np.int32)
    cur = np.zeros(len(lens), np.int32)
    while np.any(cur < lens):
        nxt = np.minimum(cur + 1, lens).astype(np.int32)
        st = alloc.allocate_for_append(k, k, B, tables, cur, nxt)
        assert np.all(st == 0)
        cur = nxt
    assert (N - int(alloc.free_count[0])) * B == g["paged_slots"]
    for s, L in enumerate(lens):
        assert np.sum(tables[s] >= 0) == -(-L // B)
    check_allocator_invariants(alloc.free_ids, alloc.free_count[0], alloc.refcount, tables, lens, B)
    alloc.free(B, tables, np.arange(len(lens)), lens)
    assert int(alloc.free_count[0]) == N and np.all(alloc.refcount == 0)


def test_hundred_tokens_take_four_blocks_of_32():
    g = golden("hundred_tokens_four_blocks.json")
    alloc = oracle.Allocator(10)
    k = np.zeros((10, 1, g["block_size"], 8), np.float32)
    tables = np.full((1, 8), -1, np.int32)
    alloc.allocate_for_append(k, k, g["block_size"], tables, [0], [g["tokens"]])
    assert 10 - int(alloc.free_count[0]) == g["blocks"]


def test_fork_append_copy_on_write_free_keeps_every_sequence_intact():
    """Prefix sharing by fork, then appends into the shared partly filled block: every holder
    but the last reference gets a private copy, and each sequence still reads its own tokens."""
    from gpu_helpers import check_allocator_invariants
    B, N, M = 16, 64, 8
    rng = np.random.default_rng(3)
    alloc = oracle.Allocator(N)
    k = rng.standard_normal((N, 2, B, 64)).astype(np.float32)
    v = rng.standard_normal((N, 2, B, 64)).astype(np.float32)
    tables = np.full((4, M), -1, np.int32)
    lens = np.array([40, 0, 0, 0], np.int32)                 # sequence 0: 40 tokens, 3 blocks
    assert np.all(alloc.allocate_for_append(k, v, B, tables, [0, 0, 0, 0], lens) == 0)
    alloc.fork(B, tables, [[0, 1], [0, 2]], [40, 40])          # 1 and 2 share all of 0's blocks
    lens = np.array([40, 40, 40, 0], np.int32)
    check_allocator_invariants(alloc.free_ids, alloc.free_count[0], alloc.refcount, tables, lens, B)
    q = rng.standard_normal((4, 2, 64)).astype(np.float32)
    before = oracle.paged_decode("f32", k, v, q[:3], tables[:3], lens[:3], 0.125)
    shared_last = tables[0, 2]
    used_before = N - int(alloc.free_count[0])
    new = np.array([41, 45, 40, 0], np.int32)                # 0 and 1 append, 2 does not
    assert np.all(alloc.allocate_for_append(k, v, B, tables, lens, new) == 0)
    # both appenders copy (sequence 2 still holds the original), nothing else is allocated
    assert N - int(alloc.free_count[0]) == used_before + 2
    assert tables[2, 2] == shared_last and tables[0, 2] != shared_last != tables[1, 2]
    assert np.array_equal(k[tables[0, 2]], k[shared_last]) and np.array_equal(v[tables[1, 2]], v[shared_last])
    after = oracle.paged_decode("f32", k, v, q[:3], tables[:3], lens[:3], 0.125)
    assert np.array_equal(before, after)
    check_allocator_invariants(alloc.free_ids, alloc.free_count[0], alloc.refcount, tables, new, B)
    alloc.free(B, tables, [0, 1, 2], new[:3])
    assert int(alloc.free_count[0]) == N and np.all(alloc.refcount == 0)
    assert np.all(tables == -1)                              # freed sequences hold no blocks


def test_last_reference_keeps_its_block():
    B, N = 16, 8
    alloc = oracle.Allocator(N)
    k = np.zeros((N, 1, B, 8), np.float32)
    tables = np.full((2, 10), -1, np.int32)
    alloc.allocate_for_append(k, k, B, tables, [0, 0], [20, 0])
    alloc.fork(B, tables, [[0, 1]], [20])
    alloc.free(B, tables, [1], [20])
    assert np.all(tables[1] == -1) and np.all(tables[0, :2] >= 0)
    owned = tables[0, 1]
    assert np.all(alloc.allocate_for_append(k, k, B, tables, [20, 0], [21, 0]) == 0)
    assert tables[0, 1] == owned                            # refcount 1: written in place
    st = alloc.allocate_for_append(k, k, B, tables, [21, 0], [21 + 16 * 7, 0])
    assert st[0] == 1                                        # only 6 free blocks were left
