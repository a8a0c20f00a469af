"""Seeded synthetic inputs for paged KV-cache decode.

This module draws inputs only: context lengths, the placement of each
sequence's blocks in the physical pool, and the q / K / V / new-token values.
It holds none of the attention, slot-mapping, write or copy arithmetic, so
both the CUDA path and the CPU oracle can be fed from it without sharing any
of the method.

The shapes follow the workloads the pages describe: blocks of 16 tokens
("Serving models with vLLM", "How it works: PagedAttention"; 16-32 tokens in
"What Is vLLM", "How does PagedAttention work?"), blocks placed anywhere in
the pool ("vLLM in Production", "PagedAttention - Virtual Memory for the KV
Cache"), LLaMA-7B / 13B-sized heads, mixed generation lengths, sequences
sharing the physical blocks of a common prefix, and long contexts.

Recipe: structure (lengths, placement, copy-on-write choices) from
``numpy.random.default_rng(seed)``; values ~ N(0, 1) drawn in fp32 by a
seeded ``torch.Generator`` on the target device and rounded to the KV dtype
(round-to-nearest-even).  Pool blocks that no sequence uses are zero; rows
past the end of a sequence in its last block hold random values too.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def blocks_for(num_tokens, block_size):
    """Blocks a sequence of num_tokens holds when blocks are given out one at a time."""
    n = np.asarray(num_tokens, dtype=np.int64)
    return -(-n // int(block_size))


def allocated_slots(num_tokens, block_size):
    """Token slots held by the blocks of every sequence together."""
    return int(np.sum(blocks_for(num_tokens, block_size) * int(block_size)))


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    context_lens: np.ndarray          # int32 [S], includes the token appended this step
    block_tables: np.ndarray          # int32 [S][M], -1 past each sequence's blocks
    positions: np.ndarray             # int32 [S], position of the appended token (ctx - 1)
    partition_size: int               # 0 = let the library choose
    q: torch.Tensor                   # [S][Hq][D]
    k_pool: torch.Tensor              # [N][Hkv][B][D]
    v_pool: torch.Tensor
    k_new: torch.Tensor               # [S][Hkv][D]
    v_new: torch.Tensor
    shared_blocks: np.ndarray         # physical ids referenced by more than one sequence
    cow_pairs: np.ndarray             # int32 [n][2] (src, dst) for copy-on-write, may be empty
    cow_seqs: np.ndarray              # sequences whose table entry is redirected to dst
    cow_logical_block: int            # which logical block those sequences copy
    seed: int = 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max(initial=0))

    @property
    def device(self) -> torch.device:
        return self.k_pool.device

    def block_tables_after_cow(self) -> np.ndarray:
        bt = self.block_tables.copy()
        for s, (_, dst) in zip(self.cow_seqs, self.cow_pairs):
            bt[s, self.cow_logical_block] = dst
        return bt


def _fill_blocks(pool: torch.Tensor, ids: np.ndarray, gen: torch.Generator, chunk: int = 4096):
    """pool[ids] <- N(0,1) rounded to the pool dtype, in chunks to bound scratch memory."""
    dev = pool.device
    shape = pool.shape[1:]
    for i in range(0, len(ids), chunk):
        sel = torch.as_tensor(ids[i:i + chunk], dtype=torch.long, device=dev)
        vals = torch.randn((len(sel),) + tuple(shape), generator=gen, device=dev,
                           dtype=torch.float32)
        pool.index_copy_(0, sel, vals.to(pool.dtype))


def _randn(shape, gen, device, dtype):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def build(name: str, *, dtype: str, num_q_heads: int, num_kv_heads: int, head_dim: int,
          block_size: int, context_lens, seed: int = 0, device="cpu",
          num_blocks: Optional[int] = None, pool_slack: float = 0.10, placement=None,
          shared_prefix_blocks: int = 0, cow_fraction: float = 0.0, partition_size: int = 0,
          scale: Optional[float] = None, table_width: Optional[int] = None) -> Workload:
    """Draw one batch.

    context_lens: per-sequence lengths, each including the token appended this
    step.  With shared_prefix_blocks = k > 0, the first k logical blocks of
    every sequence are the same physical blocks (the lengths must cover them).
    placement: optional explicit physical ids, consumed in order for every
    block that is allocated; by default a seeded random draw without
    replacement from the pool.
    """
    rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32)
    S = int(ctx.shape[0])
    B = int(block_size)
    nblk = blocks_for(ctx, B).astype(np.int64)
    k_sh = int(shared_prefix_blocks)
    if k_sh and np.any(nblk < k_sh):
        raise ValueError("context shorter than the shared prefix")
    private = nblk - k_sh
    n_cow = int(math.floor(cow_fraction * S)) if k_sh else 0
    needed = k_sh + int(private.sum()) + n_cow
    if num_blocks is None:
        num_blocks = max(1, int(math.ceil((1.0 + pool_slack) * needed)))
    if needed > num_blocks:
        raise ValueError("pool too small: need %d blocks, have %d" % (needed, num_blocks))
    if placement is None:
        if num_blocks <= 4 * needed:
            ids = rng.permutation(num_blocks)[:needed]
        else:
            ids = rng.choice(num_blocks, size=needed, replace=False)
    else:
        ids = np.asarray(placement, dtype=np.int64)[:needed]
        if len(ids) < needed:
            raise ValueError("placement too short")
    ids = ids.astype(np.int32)

    M = int(table_width) if table_width else max(1, int(nblk.max(initial=1)))
    bt = np.full((S, M), -1, dtype=np.int32)
    cursor = 0
    prefix = ids[cursor:cursor + k_sh]
    cursor += k_sh
    for s in range(S):
        bt[s, :k_sh] = prefix
        n = int(private[s])
        bt[s, k_sh:k_sh + n] = ids[cursor:cursor + n]
        cursor += n
    cow_dst = ids[cursor:cursor + n_cow]
    cursor += n_cow
    cow_seqs = np.sort(rng.choice(S, size=n_cow, replace=False)).astype(np.int32) if n_cow else \
        np.zeros((0,), np.int32)
    cow_logical = k_sh - 1 if k_sh else -1
    cow_pairs = np.stack([np.full(n_cow, prefix[cow_logical] if k_sh else 0, np.int32),
                          cow_dst], axis=1).astype(np.int32) if n_cow else np.zeros((0, 2), np.int32)

    tdt = TORCH_DTYPE[dtype]
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(int(seed) * 1000003 + 17)
    Hq, Hkv, D = int(num_q_heads), int(num_kv_heads), int(head_dim)
    k_pool = torch.zeros((num_blocks, Hkv, B, D), dtype=tdt, device=dev)
    v_pool = torch.zeros_like(k_pool)
    used = ids[:cursor - n_cow]
    _fill_blocks(k_pool, used, gen)
    _fill_blocks(v_pool, used, gen)
    q = _randn((S, Hq, D), gen, dev, tdt)
    k_new = _randn((S, Hkv, D), gen, dev, tdt)
    v_new = _randn((S, Hkv, D), gen, dev, tdt)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return Workload(name=name, dtype=dtype, num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv,
                    head_dim=D, block_size=B, num_blocks=int(num_blocks),
                    scale=float(np.float32(scale)), context_lens=ctx, block_tables=bt,
                    positions=(ctx - 1).astype(np.int32), partition_size=int(partition_size),
                    q=q, k_pool=k_pool, v_pool=v_pool, k_new=k_new, v_new=v_new,
                    shared_blocks=prefix.copy(), cow_pairs=cow_pairs, cow_seqs=cow_seqs,
                    cow_logical_block=cow_logical, seed=int(seed))


# --------------------------------------------------------------------------------------------
# The five batches.  Sizes: S sequences, Hq / Hkv heads, head_dim D, block size B.
# --------------------------------------------------------------------------------------------

def tiny(seed=0, device="cpu"):
    """4 sequences, MHA 4 x 64, fp32, B = 16, lengths {1, 17, 50, 100}, 32-block pool whose
    first 14 entries of a seeded permutation are the sequences' blocks, scale 1/8."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(32)
    return build("tiny_mha_f32", dtype="f32", num_q_heads=4, num_kv_heads=4, head_dim=64,
                 block_size=16, context_lens=[1, 17, 50, 100], seed=seed, device=device,
                 num_blocks=32, placement=perm, scale=0.125)


def llama7b(seed=0, device="cpu", num_seqs=64):
    """LLaMA-7B-shaped layer: 32 heads x 128, fp16, B = 16, lengths U[128, 2048]."""
    rng = np.random.default_rng(seed + 7)
    ctx = rng.integers(128, 2048, size=num_seqs, endpoint=True)
    return build("llama7b_f16_b16", dtype="f16", num_q_heads=32, num_kv_heads=32, head_dim=128,
                 block_size=16, context_lens=ctx, seed=seed, device=device)


def lognormal_lengths(rng, n, median=512.0, sigma=1.0, lo=16, hi=4096):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def llama13b(seed=0, device="cpu", block_size=16, num_seqs=128):
    """LLaMA-13B-shaped layer: 40 heads x 128, fp16, lengths lognormal (median 512,
    sigma 1) clipped to [16, 4096], B = 16 or 32."""
    rng = np.random.default_rng(seed + 13)
    ctx = lognormal_lengths(rng, num_seqs)
    return build("llama13b_f16_b%d" % block_size, dtype="f16", num_q_heads=40, num_kv_heads=40,
                 head_dim=128, block_size=block_size, context_lens=ctx, seed=seed, device=device)


def gqa_prefix(seed=0, device="cpu", num_seqs=256):
    """GQA 32 q / 8 kv heads x 128, bf16, B = 16; every sequence = a shared 512-token prefix
    (32 physical blocks referenced by all sequences) + a private suffix U[64, 2048];
    copy-on-write of the last shared block for 10% of the sequences."""
    rng = np.random.default_rng(seed + 4)
    ctx = 512 + rng.integers(64, 2048, size=num_seqs, endpoint=True)
    return build("gqa_prefix_bf16_b16", dtype="bf16", num_q_heads=32, num_kv_heads=8,
                 head_dim=128, block_size=16, context_lens=ctx, seed=seed, device=device,
                 shared_prefix_blocks=32, cow_fraction=0.10)


def system_prompt(seed=0, device="cpu", num_seqs=256):
    """A long shared system prompt with short replies, after the example in "Serving models
    with vLLM" ("A real example": prefix caching for a 2,000-token system prompt): GQA
    32 q / 8 kv heads x 128, bf16, B = 16; every sequence = the same 2048-token prefix
    (128 shared blocks) + a private suffix U[16, 256]."""
    rng = np.random.default_rng(seed + 6)
    ctx = 2048 + rng.integers(16, 256, size=num_seqs, endpoint=True)
    return build("system_prompt_bf16_b16", dtype="bf16", num_q_heads=32, num_kv_heads=8,
                 head_dim=128, block_size=16, context_lens=ctx, seed=seed, device=device,
                 shared_prefix_blocks=128)


LONG_POOL_BYTES = 20 * 10 ** 9


def long_splitk(seed=0, device="cpu", num_seqs=8, pool_bytes=LONG_POOL_BYTES):
    """Long contexts: 32 q / 8 kv heads x 128, bf16, B = 16, lengths U[32768, 131072],
    partitions of 512 tokens, blocks scattered over a pool of about 20 GB (K and V)."""
    rng = np.random.default_rng(seed + 5)
    ctx = rng.integers(32768, 131072, size=num_seqs, endpoint=True)
    per_block = 2 * 8 * 16 * 128 * 2
    return build("long_splitk_bf16_b16", dtype="bf16", num_q_heads=32, num_kv_heads=8,
                 head_dim=128, block_size=16, context_lens=ctx, seed=seed, device=device,
                 num_blocks=int(pool_bytes // per_block), partition_size=512)


CONFIGS = {
    "tiny": tiny,
    "llama7b": llama7b,
    "llama13b_b16": lambda seed=0, device="cpu", **kw: llama13b(seed, device, 16, **kw),
    "llama13b_b32": lambda seed=0, device="cpu", **kw: llama13b(seed, device, 32, **kw),
    "gqa_prefix": gqa_prefix,
    "long_splitk": long_splitk,
    "system_prompt": system_prompt,
}


def make(name, seed=0, device="cpu", **kw) -> Workload:
    return CONFIGS[name](seed=seed, device=device, **kw)


def shortest_last_order(context_lens, fraction=0.2) -> np.ndarray:
    """A batch order a serving engine can pick on the host, where it knows every
    sequence's length: the shortest `fraction` of the sequences last (longest of them
    first), the others in their given order.  GPUs launch a decode grid's CTAs in
    sequence order, so the CTAs still running when the grid drains are then short ones
    rather than whatever long sequences happened to come last.  (Fully longest-first is
    slower: CTAs of equal length finish, and restart, in waves.)"""
    ctx = np.asarray(context_lens)
    S = ctx.size
    k = int(round(fraction * S))
    by_len = np.argsort(-ctx, kind="stable")           # longest first, ties by index
    short = by_len[S - k:] if k else np.zeros(0, np.int64)
    is_short = np.zeros(S, bool)
    is_short[short] = True
    return np.concatenate([np.flatnonzero(~is_short), short]).astype(np.int64)


def reorder(w: Workload, order) -> Workload:
    """The same batch with its sequences in `order` (row i = old sequence order[i]); the
    pools and every sequence's blocks are untouched."""
    order = np.asarray(order, np.int64)
    idx = torch.as_tensor(order, device=w.q.device)
    old_to_new = np.empty_like(order)
    old_to_new[order] = np.arange(order.size)
    return dataclasses.replace(
        w, context_lens=w.context_lens[order].astype(np.int32),
        block_tables=w.block_tables[order], positions=w.positions[order],
        q=w.q.index_select(0, idx).contiguous(), k_new=w.k_new.index_select(0, idx).contiguous(),
        v_new=w.v_new.index_select(0, idx).contiguous(),
        cow_seqs=old_to_new[w.cow_seqs].astype(np.int32))


def storage_numpy(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's element storage (fp16 / bf16 as uint16 bits)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
