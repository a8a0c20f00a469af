"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Bit-exact for slot mapping, cache write and block copy; max-abs 1e-5 (fp32
KV) / 2e-3 (fp16, bf16 KV) for attention with fp32 output; a 16-bit output
must equal the oracle rounded to that type within one unit in the last place.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_293_gb300 import workloads
from gpu_helpers import TOL, OracleStep, dev_i32, host, max_abs, pkv

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def P():
    return pkv()


@pytest.fixture
def engine(P, request):
    """Run the test with the decode engine given by the parameter, then restore auto."""
    P.pkv_set_decode_engine(request.param)
    yield request.param
    P.pkv_set_decode_engine(P.ENGINE_AUTO)


ENGINES = [0, 1, 2]          # auto, CUDA cores, tensor cores
ENGINE_IDS = ["auto", "cuda_cores", "tensor_cores"]


def run_decode(P, w, partition_size=None, out_dtype=torch.float32, block_tables=None,
               context_lens=None, max_context_len=None):
    bt = dev_i32(w.block_tables if block_tables is None else block_tables)
    ctx_np = w.context_lens if context_lens is None else context_lens
    ctx = dev_i32(ctx_np)
    mcl = int(np.max(ctx_np, initial=0)) if max_context_len is None else max_context_len
    ps = w.partition_size if partition_size is None else partition_size
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"), dtype=out_dtype,
                     device=DEV)
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, mcl, ps)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, bt, ctx, w.scale, out, mcl, ps, ws)
    torch.cuda.synchronize()
    return out


def oracle_decode(w, block_tables=None):
    bt = w.block_tables if block_tables is None else block_tables
    return oracle.paged_decode(w.dtype, host(w.k_pool), host(w.v_pool), host(w.q), bt,
                               w.context_lens, w.scale)


def assert_no_device_error(P):
    assert P.pkv_get_device_error() == 0


# ------------------------------------------------------------------ small, many shapes

SMALL = [
    # dtype, Hq, Hkv, D, B, context lengths (ragged, partial chunks, 1 token, empty)
    ("f32", 4, 4, 64, 16, [1, 17, 50, 100]),
    ("f32", 8, 2, 128, 32, [0, 33, 64, 300, 15]),
    ("f16", 8, 8, 128, 16, [1, 16, 17, 31, 32, 33, 511, 513, 1000]),
    ("f16", 16, 2, 64, 32, [5, 64, 65, 700]),
    ("bf16", 32, 8, 128, 16, [3, 48, 160, 1100]),
    ("bf16", 8, 1, 64, 16, [2, 250]),
    ("f16", 32, 4, 128, 32, [90, 1999]),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,ctx", SMALL)
@pytest.mark.parametrize("psize", [0, 64, 512, 4096])
@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS, indirect=True)
def test_decode_matches_oracle_small(P, engine, dtype, Hq, Hkv, D, B, ctx, psize):
    if psize and psize % B:
        pytest.skip("partition must be a multiple of the block size")
    if dtype == "f32" and engine == 2:
        pytest.skip("fp32 pools always use the CUDA-core kernel")
    w = workloads.build("small", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=B, context_lens=ctx, seed=len(ctx) + D, device=DEV)
    got = run_decode(P, w, partition_size=psize)
    ref = oracle_decode(w)
    assert max_abs(got, ref) <= TOL[dtype]
    assert_no_device_error(P)


@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_split_equals_single_pass(P, engine):
    w = workloads.build("split", dtype="f16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                        block_size=16, context_lens=[4000, 700, 1, 2048, 513], seed=3, device=DEV)
    single = run_decode(P, w, partition_size=4096)
    for ps in (16, 128, 512, 1024):
        split = run_decode(P, w, partition_size=ps)
        assert max_abs(split, single.double().cpu().numpy()) <= 1e-5
    assert_no_device_error(P)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_16bit_output_is_oracle_rounded_within_one_ulp(P, engine, dtype):
    w = workloads.build("out16", dtype=dtype, num_q_heads=8, num_kv_heads=2, head_dim=128,
                        block_size=16, context_lens=[7, 300, 1500], seed=5, device=DEV)
    tdt = workloads.TORCH_DTYPE[dtype]
    got = run_decode(P, w, out_dtype=tdt, partition_size=512)
    _assert_16bit_close(got, oracle_decode(w), dtype)


@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_engines_agree_and_hold_nan_rows_past_the_context(P, engine):
    """Rows past a sequence's end in its last block may hold anything (here NaN and
    inf); neither kernel lets them into the result."""
    w = workloads.build("nanrows", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=32, context_lens=[5, 47, 1000, 70], seed=19, device=DEV)
    for s, c in enumerate(w.context_lens):
        last = w.block_tables[s, (c - 1) // 32]
        w.k_pool[last, :, c % 32:] = float("nan") if c % 32 else w.k_pool[last, :, c % 32:]
        w.v_pool[last, :, c % 32:] = float("inf") if c % 32 else w.v_pool[last, :, c % 32:]
    got = run_decode(P, w, partition_size=0)
    assert torch.isfinite(got).all()
    assert max_abs(got, oracle_decode(w)) <= TOL["bf16"]


@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_block_permutation_gives_bit_identical_output(P, engine):
    w = workloads.build("perm", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[40, 900, 1234, 17], seed=8, device=DEV)
    base = run_decode(P, w, partition_size=512)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1))
    k2 = torch.empty_like(w.k_pool)
    v2 = torch.empty_like(w.v_pool)
    k2[perm.to(DEV)] = w.k_pool
    v2[perm.to(DEV)] = w.v_pool
    bt = np.where(w.block_tables >= 0, perm.numpy()[np.maximum(w.block_tables, 0)], -1)
    w.k_pool, w.v_pool = k2, v2
    moved = run_decode(P, w, partition_size=512, block_tables=bt)
    assert torch.equal(base, moved)


@pytest.mark.parametrize("Pz", [256, 64])   # up to 8 partitions a row, and up to 32
@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_partitions_and_merge_match_oracle(P, engine, Pz):
    w = workloads.build("parts", dtype="f16", num_q_heads=8, num_kv_heads=4, head_dim=64,
                        block_size=16, context_lens=[0, 5, 512, 1025, 2000], seed=9, device=DEV)
    mcl = int(w.context_lens.max())
    nparts = -(-mcl // Pz)
    ws = P.workspace_tensor(P.pkv_partition_workspace_bytes(w.num_seqs, w.num_q_heads,
                                                            w.head_dim, mcl, Pz), DEV)
    ctx = dev_i32(w.context_lens)
    P.pkv_paged_attention_partitions(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables), ctx,
                                     w.scale, mcl, Pz, ws)
    torch.cuda.synchronize()
    rows = w.num_seqs * w.num_q_heads * nparts
    a = (rows * 4 + 15) // 16 * 16
    wsf = ws.cpu().numpy()
    m = wsf[:rows * 4].view(np.float32).reshape(w.num_seqs, w.num_q_heads, nparts)
    l = wsf[a:a + rows * 4].view(np.float32).reshape(w.num_seqs, w.num_q_heads, nparts)
    o = wsf[2 * a:2 * a + rows * w.head_dim * 4].view(np.float32).reshape(
        w.num_seqs, w.num_q_heads, nparts, w.head_dim)
    rm, rl, ro = oracle.partition_decode(w.dtype, host(w.k_pool), host(w.v_pool), host(w.q),
                                         w.block_tables, w.context_lens, w.scale, Pz, nparts)
    for s, c in enumerate(w.context_lens):
        k = max(1, -(-int(c) // Pz))
        if c == 0:
            assert np.all(l[s, :, 0] == 0) and np.all(np.isneginf(m[s, :, 0]))
            continue
        np.testing.assert_allclose(m[s, :, :k], rm[s, :, :k], atol=2e-5, rtol=0)
        np.testing.assert_allclose(l[s, :, :k], rl[s, :, :k], rtol=2e-5, atol=0)
        np.testing.assert_allclose(o[s, :, :k] / l[s, :, :k, None],
                                   ro[s, :, :k] / rl[s, :, :k, None], atol=2e-3, rtol=0)
    # the merge entry point on the oracle's own partial results
    ws2 = torch.zeros_like(ws)
    buf = np.zeros(ws.numel(), np.uint8)
    rm2 = np.where(np.isneginf(rm), -np.inf, rm).astype(np.float32)
    buf[:rows * 4] = rm2.ravel().view(np.uint8)
    buf[a:a + rows * 4] = rl.astype(np.float32).ravel().view(np.uint8)
    buf[2 * a:2 * a + rows * w.head_dim * 4] = ro.astype(np.float32).ravel().view(np.uint8)
    ws2.copy_(torch.from_numpy(buf))
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32, device=DEV)
    P.pkv_lse_merge(ws2, w.num_seqs, w.num_q_heads, w.head_dim, ctx, mcl, Pz, out)
    torch.cuda.synchronize()
    ref = oracle.lse_merge(rm, rl, ro)
    assert max_abs(out, ref) <= 1e-5
    assert_no_device_error(P)


# ------------------------------------------------------------------ write, slot mapping, copy

@pytest.mark.parametrize("dtype,B,D", [("f32", 16, 64), ("f16", 32, 128), ("bf16", 16, 128)])
def test_slot_mapping_and_write_bit_exact(P, dtype, B, D):
    w = workloads.build("write", dtype=dtype, num_q_heads=8, num_kv_heads=8, head_dim=D,
                        block_size=B, context_lens=[1, 16, 17, 33, 200, 64], seed=2, device=DEV)
    pos = w.positions.copy()
    pos[3] = -1                                   # a padding token
    slots = torch.empty(w.num_seqs, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(dev_i32(w.block_tables), dev_i32(pos), B, slots)
    torch.cuda.synchronize()
    ref_slots = oracle.slot_mapping(w.block_tables, pos, B)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    k_ref, v_ref = host(w.k_pool).copy(), host(w.v_pool).copy()
    oracle.kv_cache_write(dtype, k_ref, v_ref, host(w.k_new), host(w.v_new), ref_slots)
    P.pkv_kv_cache_write(w.k_pool, w.v_pool, w.k_new, w.v_new, slots)
    torch.cuda.synchronize()
    assert np.array_equal(host(w.k_pool), k_ref) and np.array_equal(host(w.v_pool), v_ref)
    assert_no_device_error(P)


def test_slot_mapping_with_token_sequence_index(P):
    bt = np.array([[3, 1, -1], [0, 2, 4]], np.int32)
    pos = np.array([0, 15, 16, 17, 40, -1], np.int32)
    seq = np.array([0, 1, 0, 1, 1, 0], np.int32)
    slots = torch.empty(6, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(dev_i32(bt), dev_i32(pos), 16, slots, token_seq=dev_i32(seq))
    torch.cuda.synchronize()
    assert np.array_equal(slots.cpu().numpy(), oracle.slot_mapping(bt, pos, 16, token_seq=seq))


def test_copy_blocks_bit_exact_and_cow_is_a_no_op(P):
    w = workloads.build("cow", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=list(range(520, 1800, 80)), seed=4,
                        device=DEV, shared_prefix_blocks=32, cow_fraction=0.25)
    before = run_decode(P, w, partition_size=512)
    k_ref, v_ref = host(w.k_pool).copy(), host(w.v_pool).copy()
    oracle.copy_blocks(k_ref, v_ref, w.cow_pairs)
    P.pkv_copy_blocks(w.k_pool, w.v_pool, dev_i32(w.cow_pairs))
    torch.cuda.synchronize()
    assert np.array_equal(host(w.k_pool), k_ref) and np.array_equal(host(w.v_pool), v_ref)
    after = run_decode(P, w, partition_size=512, block_tables=w.block_tables_after_cow())
    assert torch.equal(before, after)
    assert_no_device_error(P)


# ------------------------------------------------------------------ the largest batch the grid takes

@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
@pytest.mark.parametrize("psize", [0, 16])
def test_largest_batch_the_grid_takes(P, engine, psize):
    """65535 sequences (one grid row each; one more is refused on the host), ragged contexts
    of 0-40 tokens; with partitions of one block most rows go through the merge."""
    ctx = np.random.default_rng(71).integers(0, 41, size=65535)
    w = workloads.build("maxgrid", dtype="bf16", num_q_heads=4, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=ctx, seed=71, device=DEV)
    out = run_decode(P, w, partition_size=psize)
    assert max_abs(out, oracle_decode(w)) <= TOL["bf16"]
    assert torch.all(out[torch.as_tensor(ctx == 0, device=DEV)] == 0)
    assert_no_device_error(P)


# ------------------------------------------------------------------ device-side error reporting

def test_bad_block_id_sets_flag_without_faulting(P):
    w = workloads.build("bad", dtype="f16", num_q_heads=4, num_kv_heads=4, head_dim=128,
                        block_size=16, context_lens=[40, 40], seed=1, device=DEV)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks + 5                    # outside the pool
    run_decode(P, w, partition_size=0, block_tables=bt)
    assert P.pkv_get_device_error() & P.DEVERR["BLOCK_ID"]
    assert P.pkv_get_device_error() == 0           # reading clears it


def test_slot_past_pool_sets_flag(P):
    w = workloads.build("badslot", dtype="f16", num_q_heads=4, num_kv_heads=4, head_dim=128,
                        block_size=16, context_lens=[5], seed=1, device=DEV)
    k0 = w.k_pool.clone()
    slots = torch.tensor([w.num_blocks * 16 + 3], dtype=torch.int64, device=DEV)
    P.pkv_kv_cache_write(w.k_pool, w.v_pool, w.k_new, w.v_new, slots)
    assert P.pkv_get_device_error() & P.DEVERR["SLOT"]
    assert torch.equal(k0, w.k_pool)


def test_context_beyond_table_sets_flag(P):
    w = workloads.build("badctx", dtype="f16", num_q_heads=4, num_kv_heads=4, head_dim=128,
                        block_size=16, context_lens=[30], seed=1, device=DEV)
    run_decode(P, w, partition_size=0, context_lens=np.array([100], np.int32), max_context_len=100)
    assert P.pkv_get_device_error() & P.DEVERR["CONTEXT"]


def test_host_checks_return_status_before_launch(P):
    w = workloads.build("args", dtype="f16", num_q_heads=6, num_kv_heads=4, head_dim=128,
                        block_size=16, context_lens=[30], seed=1, device=DEV)
    out = torch.empty((1, 6, 128), device=DEV)
    with pytest.raises(P.PagedKVError) as e:   # 6 % 4 != 0
        P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                     dev_i32(w.context_lens), w.scale, out, 30)
    assert e.value.status == P.PKV_ERR_INVALID
    w2 = workloads.build("args2", dtype="f16", num_q_heads=8, num_kv_heads=4, head_dim=128,
                         block_size=16, context_lens=[3000], seed=1, device=DEV)
    out2 = torch.empty((1, 8, 128), device=DEV)
    with pytest.raises(P.PagedKVError) as e:   # needs a workspace
        P.pkv_paged_attention_decode(w2.q, w2.k_pool, w2.v_pool, dev_i32(w2.block_tables),
                                     dev_i32(w2.context_lens), w2.scale, out2, 3000, 512, None)
    assert e.value.status == P.PKV_ERR_WORKSPACE


# ------------------------------------------------------------------ the five batches at full size

def full_step(P, w):
    """slot mapping -> cache write -> decode, as one decode step of a layer runs it."""
    bt = dev_i32(w.block_tables)
    pos = dev_i32(w.positions)
    ctx = dev_i32(w.context_lens)
    slots = torch.empty(w.num_seqs, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(bt, pos, w.block_size, slots)
    P.pkv_kv_cache_write(w.k_pool, w.v_pool, w.k_new, w.v_new, slots)
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=torch.float32, device=DEV)
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, mcl,
                                            w.partition_size)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, bt, ctx, w.scale, out, mcl,
                                 w.partition_size, ws)
    torch.cuda.synchronize()
    return slots, out


@pytest.mark.parametrize("name", ["tiny", "llama7b", "llama13b_b16", "llama13b_b32", "gqa_prefix"])
def test_full_config_step_matches_oracle(P, name):
    assert P.pkv_get_decode_engine() == P.ENGINE_AUTO
    w = workloads.make(name, seed=0, device=DEV)
    k0, v0 = host(w.k_pool).copy(), host(w.v_pool).copy()
    slots, out = full_step(P, w)
    ref_slots = oracle.slot_mapping(w.block_tables, w.positions, w.block_size)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    oracle.kv_cache_write(w.dtype, k0, v0, host(w.k_new), host(w.v_new), ref_slots)
    assert np.array_equal(host(w.k_pool), k0) and np.array_equal(host(w.v_pool), v0)
    ref = oracle.paged_decode(w.dtype, k0, v0, host(w.q), w.block_tables, w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL[w.dtype]
    if len(w.cow_pairs):
        P.pkv_copy_blocks(w.k_pool, w.v_pool, dev_i32(w.cow_pairs))
        oracle.copy_blocks(k0, v0, w.cow_pairs)
        torch.cuda.synchronize()
        assert np.array_equal(host(w.k_pool), k0) and np.array_equal(host(w.v_pool), v0)
        after = run_decode(P, w, block_tables=w.block_tables_after_cow())
        assert torch.equal(after, out)
    assert_no_device_error(P)


def test_long_context_split_matches_oracle_on_every_sequence(P):
    """The long-context batch (8 sequences of 32k-128k tokens, partitions of 512, ~20 GB
    pool): slot mapping, cache write and decode as three launches.  The oracle's inputs are
    host copies of every block the batch uses, taken before the GPU step, with the oracle's
    own write applied; the GPU's written blocks must equal them bit for bit, no other block
    may change, and all 8 sequences' attention must be within 2e-3 of the oracle's."""
    w = workloads.make("long_splitk", seed=0, device=DEV)
    ref = OracleStep(w, keep_device_clone=True)
    ref.write()
    slots, out = full_step(P, w)
    assert np.array_equal(slots.cpu().numpy(), ref.slots)
    ref.check_pools(w)
    ref.check_whole_pools(w)
    assert out.shape[0] == 8
    assert max_abs(out, ref.decode()) <= TOL[w.dtype]
    assert_no_device_error(P)


# ------------------------------------------------------------------ fused append + decode

@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,ctx,psize", [
    ("f16", 8, 8, 128, 16, [1, 16, 17, 300, 1025, 0], 0),
    ("bf16", 32, 8, 128, 32, [33, 64, 2000, 5], 512),
    ("f32", 4, 4, 64, 16, [1, 17, 50, 100], 0),
    ("f16", 16, 2, 64, 16, [700, 31, 4096], 256),
])
@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS, indirect=True)
def test_fused_append_decode_equals_write_then_decode(P, engine, dtype, Hq, Hkv, D, B, ctx,
                                                      psize):
    w = workloads.build("fused", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=B, context_lens=ctx, seed=31, device=DEV)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    mcl = w.max_context_len
    bt, cl = dev_i32(w.block_tables), dev_i32(w.context_lens)
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, mcl, psize)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.full((w.num_seqs, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    slots = torch.full((w.num_seqs,), -7, dtype=torch.int64, device=DEV)
    P.pkv_paged_attention_decode_append(w.q, w.k_pool, w.v_pool, w.k_new, w.v_new, bt, cl,
                                        w.scale, out, mcl, psize, ws, slot_mapping=slots)
    torch.cuda.synchronize()
    # oracle: slot mapping, write, decode
    ref_slots = oracle.slot_mapping(w.block_tables, w.positions, B)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    kr, vr = host(k0).copy(), host(v0).copy()
    oracle.kv_cache_write(dtype, kr, vr, host(w.k_new), host(w.v_new), ref_slots)
    assert np.array_equal(host(w.k_pool), kr) and np.array_equal(host(w.v_pool), vr)
    ref = oracle.paged_decode(dtype, kr, vr, host(w.q), w.block_tables, w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL[dtype]
    # and bit-identical to the three-launch path on the GPU
    w.k_pool, w.v_pool = k0, v0
    s2 = torch.empty(w.num_seqs, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(bt, dev_i32(w.positions), B, s2)
    P.pkv_kv_cache_write(w.k_pool, w.v_pool, w.k_new, w.v_new, s2)
    out2 = run_decode(P, w, partition_size=psize)
    assert torch.equal(out, out2)
    assert_no_device_error(P)


# ------------------------------------------------------------------ swap to host and back

def test_swap_blocks_to_pinned_host_and_back(P):
    w = workloads.build("swapg", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[300, 1000, 45], seed=13, device=DEV,
                        num_blocks=200)
    before = run_decode(P, w, partition_size=0)
    seq, nb = 1, 63
    used = w.block_tables[seq, :nb].copy()
    hk = torch.zeros((nb + 5,) + tuple(w.k_pool.shape[1:]), dtype=w.k_pool.dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = np.stack([used, np.arange(nb) + 2], 1).astype(np.int32)
    P.pkv_swap_blocks(w.k_pool, w.v_pool, hk, hv, dev_i32(out_pairs))
    torch.cuda.synchronize()
    rk, rv = host(hk).copy() * 0, host(hv).copy() * 0
    oracle.swap_blocks(host(w.k_pool), host(w.v_pool), rk, rv, out_pairs)
    assert np.array_equal(host(hk), rk) and np.array_equal(host(hv), rv)
    # the preempted sequence's blocks are reused, then it is swapped back into other blocks
    w.k_pool[torch.as_tensor(used, device=DEV).long()] = 0
    w.v_pool[torch.as_tensor(used, device=DEV).long()] = 0
    free = np.setdiff1d(np.arange(w.num_blocks), w.block_tables[w.block_tables >= 0])[:nb]
    in_pairs = np.stack([np.arange(nb) + 2, free], 1).astype(np.int32)
    pairs_pinned = torch.from_numpy(in_pairs).pin_memory()      # pairs may live on the host too
    P.pkv_swap_blocks(hk, hv, w.k_pool, w.v_pool, pairs_pinned)
    torch.cuda.synchronize()
    bt = w.block_tables.copy()
    bt[seq, :nb] = free
    after = run_decode(P, w, partition_size=0, block_tables=bt)
    assert torch.equal(before, after)
    assert_no_device_error(P)
    with pytest.raises(P.PagedKVError):                        # pageable host memory is refused
        P.pkv_swap_blocks(w.k_pool, w.v_pool, torch.zeros_like(hk), torch.zeros_like(hv),
                          dev_i32(out_pairs))


# ------------------------------------------------------------------ several query rows per sequence

@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,ctx,nq,psize", [
    ("f16", 8, 8, 128, 16, [40, 300, 17, 1500], 4, 0),      # MHA: all 4 queries in one pass
    ("bf16", 32, 8, 128, 16, [5, 700, 64, 2000], 3, 512),   # G=4: 2 queries per pass, 2 passes
    ("bf16", 16, 2, 64, 32, [33, 1025, 3], 2, 256),         # G=8: 1 query per pass; a row sees nothing
    ("f16", 16, 8, 128, 16, [1, 9, 4096], 8, 1024),         # G=2, 8 queries -> 2 passes
])
def test_multi_query_decode_matches_oracle(P, dtype, Hq, Hkv, D, B, ctx, nq, psize):
    w = workloads.build("multi", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=B, context_lens=ctx, seed=41, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    tdt = workloads.TORCH_DTYPE[dtype]
    q = torch.randn((w.num_seqs, nq, Hq, D), generator=g, device=DEV).to(tdt)
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs * nq, Hq, mcl, psize)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.full((w.num_seqs, nq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_multi(q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                       dev_i32(w.context_lens), w.scale, out, mcl, psize, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_decode_multi(dtype, host(w.k_pool), host(w.v_pool), host(q),
                                    w.block_tables, w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL[dtype]
    # the last query of each sequence sees the whole context: plain decode
    P.pkv_set_decode_engine(P.ENGINE_TENSOR_CORES)
    try:
        w.q = q[:, -1].contiguous()
        last = run_decode(P, w, partition_size=psize)
    finally:
        P.pkv_set_decode_engine(P.ENGINE_AUTO)
    assert max_abs(out[:, -1], last.double().cpu().numpy()) <= 1e-5
    assert_no_device_error(P)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,ctx,nq,psize", [
    ("f16", 8, 8, 128, 16, [40, 300, 17, 1500, 4], 4, 0),   # MHA; a context of exactly nq
    ("bf16", 32, 8, 128, 16, [5, 700, 64, 2000], 3, 512),   # G=4: 2 queries per pass
    ("bf16", 16, 2, 64, 32, [33, 1025, 3, 0], 2, 256),      # G=8; an empty sequence
    ("f16", 16, 8, 128, 16, [1, 9, 4096, 31], 8, 1024),     # G=2, 8 queries; ctx < nq
    ("bf16", 8, 4, 64, 16, [17, 18, 47, 48, 49], 16, 0),    # 16 new rows across block edges
])
def test_multi_query_fused_append_equals_write_then_decode(P, dtype, Hq, Hkv, D, B, ctx, nq,
                                                           psize):
    w = workloads.build("multiapp", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=B, context_lens=ctx, seed=43, device=DEV)
    g = torch.Generator(device=DEV).manual_seed(7)
    tdt = workloads.TORCH_DTYPE[dtype]
    S = w.num_seqs
    q = torch.randn((S, nq, Hq, D), generator=g, device=DEV).to(tdt)
    kn = torch.randn((S, nq, Hkv, D), generator=g, device=DEV).to(tdt)
    vn = torch.randn((S, nq, Hkv, D), generator=g, device=DEV).to(tdt)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    mcl = w.max_context_len
    bt, cl = dev_i32(w.block_tables), dev_i32(w.context_lens)
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, S * nq, Hq, mcl, psize)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.full((S, nq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    slots = torch.full((S, nq), -7, dtype=torch.int64, device=DEV)
    P.pkv_paged_attention_decode_multi_append(q, w.k_pool, w.v_pool, kn, vn, bt, cl, w.scale,
                                              out, mcl, psize, ws, slot_mapping=slots)
    torch.cuda.synchronize()
    # oracle: the new tokens sit at the last nq positions of each context
    pos = (w.context_lens[:, None] - nq + np.arange(nq)[None, :]).astype(np.int32)
    seq = np.repeat(np.arange(S, dtype=np.int32), nq)
    ref_slots = oracle.slot_mapping(w.block_tables, pos.reshape(-1), B, token_seq=seq)
    assert np.array_equal(slots.cpu().numpy().reshape(-1), ref_slots)
    kr, vr = host(k0).copy(), host(v0).copy()
    oracle.kv_cache_write(dtype, kr, vr, host(kn).reshape(S * nq, Hkv, D),
                          host(vn).reshape(S * nq, Hkv, D), ref_slots)
    assert np.array_equal(host(w.k_pool), kr) and np.array_equal(host(w.v_pool), vr)
    ref = oracle.paged_decode_multi(dtype, kr, vr, host(q), w.block_tables, w.context_lens,
                                    w.scale)
    live = (pos >= 0)
    assert not np.isnan(host(out)[~live]).any()             # rows that see nothing are written too
    assert max_abs(out, ref) <= TOL[dtype]
    # bit-identical to slot mapping + cache write + multi-query decode on the GPU
    k2, v2 = k0.clone(), v0.clone()
    s2 = torch.empty(S * nq, dtype=torch.int64, device=DEV)
    P.pkv_slot_mapping(bt, dev_i32(pos.reshape(-1)), B, s2, token_seq=dev_i32(seq))
    P.pkv_kv_cache_write(k2, v2, kn.reshape(S * nq, Hkv, D), vn.reshape(S * nq, Hkv, D), s2)
    out2 = torch.full_like(out, float("nan"))
    P.pkv_paged_attention_decode_multi(q, k2, v2, bt, cl, w.scale, out2, mcl, psize, ws)
    torch.cuda.synchronize()
    assert torch.equal(k2, w.k_pool) and torch.equal(v2, w.v_pool)
    assert torch.equal(out, out2)
    assert_no_device_error(P)


def test_multi_query_fused_append_flags_a_bad_table_entry(P):
    w = workloads.build("multiapp_bad", dtype="f16", num_q_heads=8, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[40, 100], seed=44, device=DEV)
    nq = 4
    bt = w.block_tables.copy()
    bt[1, (100 - 1) // 16] = -1                         # the block the new rows of seq 1 land in
    g = torch.Generator(device=DEV).manual_seed(8)
    q = torch.randn((2, nq, 8, 128), generator=g, device=DEV).half()
    kn = torch.randn((2, nq, 8, 128), generator=g, device=DEV).half()
    vn = torch.randn_like(kn)
    k0 = w.k_pool.clone()
    out = torch.zeros((2, nq, 8, 128), dtype=torch.float32, device=DEV)
    slots = torch.full((2, nq), -7, dtype=torch.int64, device=DEV)
    P.pkv_paged_attention_decode_multi_append(q, w.k_pool, w.v_pool, kn, vn, dev_i32(bt),
                                              dev_i32(w.context_lens), w.scale, out, 100, 0,
                                              None, slot_mapping=slots)
    torch.cuda.synchronize()
    s = slots.cpu().numpy()
    assert np.all(s[1] == -1) and np.all(s[0] >= 0)
    err = P.pkv_get_device_error()
    assert err & P.DEVERR["BLOCK_ID"]
    # the first sequence's rows went in; nothing was written through the bad entry
    k_expect = host(k0).copy()
    for j in range(nq):
        sl = int(s[0, j])
        k_expect[sl // 16, :, sl % 16, :] = host(kn)[0, j]
    assert np.array_equal(host(w.k_pool), k_expect)


# ------------------------------------------------------------------ exactly what bench.py times

def _assert_16bit_close(got, ref, dtype):
    """A 16-bit output: within the stated tolerance of the unrounded oracle plus half a unit
    in the last place of the output type (the rounding of the result itself), and within
    one unit of the oracle rounded to that type."""
    tdt = workloads.TORCH_DTYPE[dtype]
    ref_r = torch.from_numpy(ref).to(tdt).double()
    mant, floor = (10, 2.0 ** -24) if dtype == "f16" else (7, 2.0 ** -133)
    ulp = (ref_r.abs().clamp_min(1e-38).log2().floor() - mant).exp2().clamp_min(floor)
    err = (got.double().cpu() - torch.from_numpy(ref)).abs() - 0.5 * ulp
    assert err.max().item() <= TOL[dtype], err.max().item()
    assert _ulp_excess(got, ref, dtype) <= 0


def _ulp_excess(got, ref, dtype, ulps=1, abs_floor=1e-5):
    """How far the 16-bit output lies beyond `ulps` units in the last place of the oracle
    rounded to that type, plus `abs_floor` (<= 0: within).  The floor covers outputs near
    zero, whose units in the last place are far below the fp32 accumulation error, which
    scales with the terms summed, not with their (cancelling) sum."""
    tdt = workloads.TORCH_DTYPE[dtype]
    ref_t = torch.from_numpy(ref)
    ref_r = ref_t.to(tdt).double()
    mant, floor = (10, 2.0 ** -24) if dtype == "f16" else (7, 2.0 ** -133)
    ulp = (ref_r.abs().clamp_min(1e-38).log2().floor() - mant).exp2().clamp_min(floor)
    return ((got.double().cpu() - ref_r).abs() - ulps * ulp - abs_floor).max().item()


@pytest.mark.parametrize("out_dtype", ["pool", "f32"])
@pytest.mark.parametrize("name", ["llama13b_b16", "gqa_prefix", "long_splitk"])
def test_bench_step_matches_oracle_at_full_size(P, name, out_dtype):
    """bench.py's own Step (the copy-on-write copy where the batch has one, then the decode
    launch with the append fused into it, the partition size and engine bench.py uses) on
    the full batch, every sequence.  The oracle's inputs are host copies of every block the
    batch uses, taken before the step, with the oracle's own copy-on-write copy and cache
    write applied: the GPU's pools must equal them bit for bit (and no other block may
    change), and the output must match the oracle's attention on them.  With the output in
    fp32 the bound is the plain max-abs 2e-3; with the output in the pool's 16-bit type (what
    bench.py times) it is 2e-3 plus the output's own rounding, and one unit in the last
    place of the oracle rounded to that type (with the absolute floor `_ulp_excess` states)."""
    import bench
    w = workloads.make(name, seed=0, device=DEV)
    st = bench.Step(P, w, torch.device(DEV), fused=True, cascade=False)
    assert st.prefix_len == 0                     # bench.py's default: no cascade
    if out_dtype == "f32":
        st.out = torch.full_like(st.out, float("nan"), dtype=torch.float32)
    pairs = w.cow_pairs if len(w.cow_pairs) else np.zeros((0, 2), np.int32)
    ref = OracleStep(w, extra_blocks=pairs[:, 1], keep_device_clone=True)
    if len(pairs):
        ref.copy_blocks(pairs)
    ref.write()
    st.pre_decode()
    st.decode()
    torch.cuda.synchronize()
    assert np.array_equal(st.slots.cpu().numpy(), ref.slots)
    ref.check_pools(w)
    ref.check_whole_pools(w)
    want = ref.decode()
    if out_dtype == "f32":
        assert max_abs(st.out, want) <= TOL[w.dtype]
    else:
        assert st.out.dtype == w.q.dtype
        _assert_16bit_close(st.out, want, w.dtype)
    assert_no_device_error(P)


@pytest.mark.parametrize("nq", [4, 8])
def test_multi_query_append_at_full_size_matches_oracle(P, nq):
    """bench.py --path multi's launch (the new tokens' K/V written by the causal multi-query
    decode launch itself, the library's automatic partitions) on the full LLaMA-13B-shaped
    batch: every sequence's slots and the pools bit-exact, every query row within 2e-3
    (fp32 output) of the oracle's attention on the oracle-written pools."""
    w = workloads.make("llama13b_b16", seed=0, device=DEV)
    S, Hq, Hkv, D, B = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    g = torch.Generator(device=DEV).manual_seed(17 + nq)
    q = torch.randn((S, nq, Hq, D), generator=g, device=DEV).half()
    kn = torch.randn((S * nq, Hkv, D), generator=g, device=DEV).half()
    vn = torch.randn((S * nq, Hkv, D), generator=g, device=DEV).half()
    kr, vr = host(w.k_pool).copy(), host(w.v_pool).copy()      # before the GPU step
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, S * nq, Hq, mcl, 0)
    ws = P.workspace_tensor(ws_bytes, DEV) if ws_bytes else None
    out = torch.full((S, nq, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    slots = torch.full((S, nq), -7, dtype=torch.int64, device=DEV)
    P.pkv_paged_attention_decode_multi_append(q, w.k_pool, w.v_pool, kn, vn,
                                              dev_i32(w.block_tables), dev_i32(w.context_lens),
                                              w.scale, out, mcl, 0, ws, slot_mapping=slots)
    torch.cuda.synchronize()
    pos = (w.context_lens[:, None] - nq + np.arange(nq)[None, :]).astype(np.int32)
    seq = np.repeat(np.arange(S, dtype=np.int32), nq)
    ref_slots = oracle.slot_mapping(w.block_tables, pos.reshape(-1), B, token_seq=seq)
    assert np.array_equal(slots.cpu().numpy().reshape(-1), ref_slots)
    oracle.kv_cache_write("f16", kr, vr, host(kn), host(vn), ref_slots)
    assert np.array_equal(host(w.k_pool), kr) and np.array_equal(host(w.v_pool), vr)
    ref = oracle.paged_decode_multi("f16", kr, vr, host(q), w.block_tables, w.context_lens,
                                    w.scale)
    assert max_abs(out, ref) <= TOL["f16"]
    assert_no_device_error(P)


def test_swap_at_full_size_matches_oracle(P):
    """bench.py --path swap's moves on the full LLaMA-13B-shaped batch: a seeded quarter of
    the blocks in use out to a pinned host pool (compared bit for bit with the oracle's
    copy of the same blocks), the device blocks overwritten, then back in."""
    w = workloads.make("llama13b_b16", seed=0, device=DEV)
    used = np.unique(np.concatenate([w.block_tables[s, :-(-int(c) // w.block_size)]
                                     for s, c in enumerate(w.context_lens)]))
    rng = np.random.default_rng(11)
    moved = np.sort(rng.choice(used, size=len(used) // 4, replace=False)).astype(np.int32)
    n = len(moved)
    shape = (n,) + tuple(w.k_pool.shape[1:])
    hk = torch.zeros(shape, dtype=w.k_pool.dtype).pin_memory()
    hv = torch.zeros(shape, dtype=w.v_pool.dtype).pin_memory()
    out_pairs = np.stack([moved, np.arange(n, dtype=np.int32)], 1).astype(np.int32)
    k0, v0 = host(w.k_pool).copy(), host(w.v_pool).copy()
    P.pkv_swap_blocks(w.k_pool, w.v_pool, hk, hv, dev_i32(out_pairs))
    torch.cuda.synchronize()
    rk, rv = np.zeros_like(host(hk)), np.zeros_like(host(hv))
    oracle.swap_blocks(k0, v0, rk, rv, out_pairs)
    assert np.array_equal(host(hk), rk) and np.array_equal(host(hv), rv)
    idx = torch.as_tensor(moved, device=DEV).long()
    w.k_pool[idx] = 0
    w.v_pool[idx] = 0
    in_pairs = np.stack([np.arange(n, dtype=np.int32), moved], 1).astype(np.int32)
    P.pkv_swap_blocks(hk, hv, w.k_pool, w.v_pool, dev_i32(in_pairs))
    torch.cuda.synchronize()
    assert np.array_equal(host(w.k_pool), k0) and np.array_equal(host(w.v_pool), v0)
    assert_no_device_error(P)


def test_bench_step_in_shortest_last_order_matches_oracle(P):
    """bench.py --order shortest-last: the same batch with its shortest fifth last; every
    sequence's slot, write and attention still match the oracle."""
    import bench
    w = workloads.make("gqa_prefix", seed=0, device=DEV)
    w = workloads.reorder(w, workloads.shortest_last_order(w.context_lens))
    st = bench.Step(P, w, torch.device(DEV), fused=True, cascade=False)
    st.out = torch.full_like(st.out, float("nan"), dtype=torch.float32)
    ref = OracleStep(w, extra_blocks=w.cow_pairs[:, 1], keep_device_clone=True)
    ref.copy_blocks(w.cow_pairs)
    ref.write()
    st.pre_decode()
    st.decode()
    torch.cuda.synchronize()
    assert np.array_equal(st.slots.cpu().numpy(), ref.slots)
    ref.check_pools(w)
    ref.check_whole_pools(w)
    assert max_abs(st.out, ref.decode()) <= TOL[w.dtype]
    assert_no_device_error(P)


# ------------------------------------------------------------------ shared-prefix (cascade) decode

def test_cascade_step_is_deterministic(P):
    """The cascade's three launches overlap (the prefix pass starts while the suffix decode's
    last CTAs run), and every floating-point result depends only on the inputs: repeated
    steps on the full shared-prefix GQA batch give bit-identical output and partials.  (A
    prefix-pass CTA that staged its output over the area where its warps exchange row sums
    once showed up here as 4-8 rows differing in about one step in three.)"""
    import bench
    w = workloads.make("gqa_prefix", seed=0, device=DEV)
    k0, v0 = w.k_pool.clone(), w.v_pool.clone()
    st = bench.Step(P, w, torch.device(DEV), fused=True, cascade=True)
    assert st.prefix_len > 0
    first = None
    for _ in range(8):
        w.k_pool.copy_(k0)
        w.v_pool.copy_(v0)
        st.ws.zero_()
        st.pre_decode()
        st.decode()
        torch.cuda.synchronize()
        got = (st.out.clone(), st.ws.clone())
        if first is None:
            first = got
        else:
            assert torch.equal(got[0], first[0]) and torch.equal(got[1], first[1])
    assert_no_device_error(P)



@pytest.mark.parametrize("dtype,Hq,Hkv,D,B,prefix_blocks,suffix,psize", [
    ("bf16", 32, 8, 128, 16, 4, [1, 30, 700, 2000, 16], 0),     # tensor-core suffix, G = 4
    ("f16", 8, 8, 128, 32, 3, [5, 64, 1100, 33], 512),         # CUDA-core suffix (MHA), B = 32
    ("f16", 16, 2, 64, 16, 2, [0, 9, 300], 256),               # a sequence that is all prefix
    ("f16", 8, 8, 128, 16, 2, [0, 7, 100], 0),                 # CUDA-core suffix finishing rows
])
def test_cascade_decode_matches_oracle_and_plain_decode(P, dtype, Hq, Hkv, D, B, prefix_blocks,
                                                        suffix, psize):
    Lp = prefix_blocks * B
    ctx = [Lp + x for x in suffix]
    w = workloads.build("cascade", dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=B, context_lens=ctx, seed=51, device=DEV,
                        shared_prefix_blocks=prefix_blocks)
    mcl = w.max_context_len
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, Hq, mcl, Lp,
                                                          psize), DEV)
    out = torch.full((w.num_seqs, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                         dev_i32(w.context_lens), w.scale, out, mcl, Lp, ws,
                                         psize)
    torch.cuda.synchronize()
    ref = oracle_decode(w)
    assert max_abs(out, ref) <= TOL[dtype]
    plain = run_decode(P, w, partition_size=psize)
    assert max_abs(out, plain.double().cpu().numpy()) <= 1e-5
    assert_no_device_error(P)


def test_cascade_with_fused_append_matches_oracle(P):
    w = workloads.build("cascade_app", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                        block_size=16, context_lens=[100, 600, 1500, 65], seed=52, device=DEV,
                        shared_prefix_blocks=4)
    Lp, mcl = 64, w.max_context_len
    k0, v0 = host(w.k_pool).copy(), host(w.v_pool).copy()
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 32, mcl, Lp), DEV)
    out = torch.empty((w.num_seqs, 32, 128), dtype=torch.bfloat16, device=DEV)
    slots = torch.empty(w.num_seqs, dtype=torch.int64, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                         dev_i32(w.context_lens), w.scale, out, mcl, Lp, ws,
                                         k_new=w.k_new, v_new=w.v_new, slot_mapping=slots)
    torch.cuda.synchronize()
    ref_slots = oracle.slot_mapping(w.block_tables, w.positions, 16)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    oracle.kv_cache_write("bf16", k0, v0, host(w.k_new), host(w.v_new), ref_slots)
    assert np.array_equal(host(w.k_pool), k0) and np.array_equal(host(w.v_pool), v0)
    ref = oracle.paged_decode("bf16", k0, v0, host(w.q), w.block_tables, w.context_lens, w.scale)
    _assert_16bit_close(out, ref, "bf16")
    assert_no_device_error(P)


def test_cascade_flags_a_sequence_with_other_prefix_blocks(P):
    w = workloads.build("cascade_bad", dtype="f16", num_q_heads=8, num_kv_heads=2, head_dim=128,
                        block_size=16, context_lens=[80, 90, 100], seed=53, device=DEV,
                        shared_prefix_blocks=2)
    bt = w.block_tables.copy()
    bt[2, 1] = bt[2, 3]                                     # sequence 2 no longer shares block 1
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, 3, 8, 100, 32), DEV)
    out = torch.empty((3, 8, 128), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(bt),
                                         dev_i32(w.context_lens), w.scale, out, 100, 32, ws)
    assert P.pkv_get_device_error() & P.DEVERR["PREFIX"]


def test_cascade_flags_a_prefix_block_outside_the_pool(P):
    """Every sequence's third prefix block names a block past the pool: the prefix pass
    copies nothing for it, sets BLOCK_ID, and the call still returns."""
    w = workloads.build("cascade_badid", dtype="bf16", num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=16, context_lens=[100, 120], seed=57,
                        device=DEV, shared_prefix_blocks=4)
    bt = w.block_tables.copy()
    bt[:, 2] = w.num_blocks + 5
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, 2, 8, 120, 64), DEV)
    out = torch.empty((2, 8, 128), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(bt),
                                         dev_i32(w.context_lens), w.scale, out, 120, 64, ws)
    torch.cuda.synchronize()
    flags = P.pkv_get_device_error()
    assert flags & P.DEVERR["BLOCK_ID"] and not flags & P.DEVERR["TIMEOUT"]


def test_cascade_prefix_pass_rescales_when_scores_grow(P):
    """Keys scaled by 1 + 15 t / 640 along a 640-token shared prefix: each row's
    maximum keeps rising, so the prefix pass raises its reference maximum and
    rescales the accumulated O on later chunks (250 sequences x G = 4: eight tiles,
    the last partial, and splits of three 64-token chunks)."""
    B, nb = 16, 40
    ctx = [nb * B + x for x in (3, 17, 64, 200, 1)] * 50
    w = workloads.build("cascade_grow", dtype="bf16", num_q_heads=16, num_kv_heads=4,
                        head_dim=128, block_size=B, context_lens=ctx, seed=54, device=DEV,
                        shared_prefix_blocks=nb)
    blocks = torch.as_tensor(w.block_tables[0, :nb].astype(np.int64), device=DEV)
    t = torch.arange(nb * B, device=DEV, dtype=torch.float32)
    w.k_pool[blocks] = (w.k_pool[blocks].float() * (1 + 15 * t / (nb * B)).view(nb, 1, B, 1)).to(
        w.k_pool.dtype)
    Lp, mcl = nb * B, w.max_context_len
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 16, mcl, Lp), DEV)
    out = torch.full((w.num_seqs, 16, 128), float("nan"), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                         dev_i32(w.context_lens), w.scale, out, mcl, Lp, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_decode("bf16", host(w.k_pool), host(w.v_pool), host(w.q), w.block_tables,
                              w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL["bf16"]
    # both paths carry each weight as a 16-bit pair (relative error <= 2^-18) against
    # V rows of magnitude up to about 4, on attention concentrated on a few tokens
    plain = run_decode(P, w)
    assert max_abs(out, plain.double().cpu().numpy()) <= 5e-5
    assert_no_device_error(P)


def test_cascade_long_prefix_few_sequences(P):
    """A 4096-token prefix shared by three sequences: a few CTAs per kv head, so the
    prefix is cut into many splits, each its own slot in the merge."""
    B, nb = 16, 256
    w = workloads.build("cascade_long", dtype="bf16", num_q_heads=16, num_kv_heads=4,
                        head_dim=128, block_size=B, context_lens=[nb * B + x for x in (5, 100, 1000)],
                        seed=55, device=DEV, shared_prefix_blocks=nb)
    Lp, mcl = nb * B, w.max_context_len
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 16, mcl, Lp), DEV)
    out = torch.full((w.num_seqs, 16, 128), float("nan"), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                         dev_i32(w.context_lens), w.scale, out, mcl, Lp, ws)
    torch.cuda.synchronize()
    assert max_abs(out, oracle_decode(w)) <= TOL["bf16"]
    plain = run_decode(P, w)
    assert max_abs(out, plain.double().cpu().numpy()) <= 1e-5
    assert_no_device_error(P)


def test_cascade_head_dim_64_rescales_when_scores_grow(P):
    """head_dim 64 (one 128-byte column per row) with keys growing along the prefix,
    so later chunks raise the reference maximum and rescale the half-width O."""
    B, nb = 32, 24
    ctx = [nb * B + x for x in (1, 40, 300)] * 30
    w = workloads.build("cascade_d64", dtype="f16", num_q_heads=8, num_kv_heads=2, head_dim=64,
                        block_size=B, context_lens=ctx, seed=56, device=DEV,
                        shared_prefix_blocks=nb)
    blocks = torch.as_tensor(w.block_tables[0, :nb].astype(np.int64), device=DEV)
    t = torch.arange(nb * B, device=DEV, dtype=torch.float32)
    w.k_pool[blocks] = (w.k_pool[blocks].float() * (1 + 12 * t / (nb * B)).view(nb, 1, B, 1)).to(
        w.k_pool.dtype)
    Lp, mcl = nb * B, w.max_context_len
    ws = P.workspace_tensor(P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, 8, mcl, Lp), DEV)
    out = torch.full((w.num_seqs, 8, 64), float("nan"), dtype=torch.float32, device=DEV)
    P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, dev_i32(w.block_tables),
                                         dev_i32(w.context_lens), w.scale, out, mcl, Lp, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_decode("f16", host(w.k_pool), host(w.v_pool), host(w.q), w.block_tables,
                              w.context_lens, w.scale)
    assert max_abs(out, ref) <= TOL["f16"]
    assert_no_device_error(P)


def test_cascade_on_the_system_prompt_batch_matches_oracle(P):
    """The long-shared-prompt batch through bench.py's cascade step, against the oracle."""
    import bench
    w = workloads.make("system_prompt", seed=0, device=DEV, num_seqs=64)
    st = bench.Step(P, w, torch.device(DEV), fused=True, cascade=True)
    assert st.prefix_len == 2048
    st.pre_decode()
    st.decode()
    torch.cuda.synchronize()
    ref = oracle.paged_decode(w.dtype, host(w.k_pool), host(w.v_pool), host(w.q),
                              w.block_tables, w.context_lens, w.scale)
    _assert_16bit_close(st.out, ref, w.dtype)
    assert_no_device_error(P)


# ------------------------------------------------------------------ sizes at the edges

@pytest.mark.parametrize("engine", [1, 2], ids=["cuda_cores", "tensor_cores"], indirect=True)
def test_many_short_ragged_sequences(P, engine):
    """4096 sequences of 1..80 tokens (a large grid of mostly one-chunk CTAs)."""
    rng = np.random.default_rng(61)
    ctx = rng.integers(1, 81, size=4096)
    w = workloads.build("many", dtype="bf16", num_q_heads=8, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=ctx, seed=61, device=DEV)
    got = run_decode(P, w, partition_size=0)
    assert max_abs(got, oracle_decode(w)) <= TOL["bf16"]
    assert_no_device_error(P)


@pytest.mark.parametrize("psize", [0, 64, 1024])
def test_contexts_that_fill_their_table_rows_exactly(P, psize):
    """Every context = max_blocks_per_seq * B (no partial last block, no spare table entry),
    including one exactly one partition long."""
    B, M = 32, 32
    w = workloads.build("full", dtype="f16", num_q_heads=16, num_kv_heads=4, head_dim=128,
                        block_size=B, context_lens=[B * M, B * 2, 1024], seed=62, device=DEV,
                        table_width=M)
    assert w.block_tables.shape[1] == M and int(w.context_lens[0]) == B * M
    got = run_decode(P, w, partition_size=psize)
    assert max_abs(got, oracle_decode(w)) <= TOL["f16"]
    assert_no_device_error(P)


def test_empty_batch_launches_nothing(P):
    k = torch.zeros((4, 2, 16, 128), dtype=torch.float16, device=DEV)
    q = torch.zeros((0, 2, 128), dtype=torch.float16, device=DEV)
    out = torch.zeros((0, 2, 128), dtype=torch.float32, device=DEV)
    bt = torch.zeros((0, 1), dtype=torch.int32, device=DEV)
    ctx = torch.zeros((0,), dtype=torch.int32, device=DEV)
    P.pkv_paged_attention_decode(q, k, k, bt.reshape(0, 1), ctx, 0.1, out, 0)
    torch.cuda.synchronize()
    assert_no_device_error(P)
