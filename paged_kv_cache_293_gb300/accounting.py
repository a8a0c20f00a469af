"""Algorithmic byte and flop counts of the paged decode path (for rooflines).

The per-token KV footprint is 2 (K and V) x kv heads x head_dim x element
bytes per layer; for LLaMA-13B (40 layers, 40 heads of 128, fp16) and 2048
tokens this is the "up to 1.7 GB per sequence" figure quoted in "vLLM in
Production", section "The KV Cache and the 60-80% Memory Tax".
"""
import numpy as np


def kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes):
    """K plus V bytes one cached token holds in one layer."""
    return 2 * int(num_kv_heads) * int(head_dim) * int(elem_bytes)


def decode_bytes(context_lens, num_kv_heads, num_q_heads, head_dim, elem_bytes, out_bytes,
                 block_size, partition_size=0, unique_tokens=None):
    """Bytes one decode call must move at least once.

    KV: every cached position of every sequence, once per kv head (or, with
    unique_tokens, each shared position once).  Plus q in, out, the block table
    entries the lengths need, the lengths themselves and, for partitioned
    calls, the fp32 partial results written and read back.
    """
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = ctx.size
    toks = int(ctx.sum()) if unique_tokens is None else int(unique_tokens)
    kv = toks * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes)
    qo = S * num_q_heads * head_dim * (elem_bytes + out_bytes)
    table = int((-(-ctx // block_size)).sum()) * 4 + S * 4
    ws = 0
    if partition_size:
        parts = -(-ctx // partition_size)
        multi = parts[parts > 1]
        ws = 2 * int(multi.sum()) * num_q_heads * (head_dim + 2) * 4
    return kv + qo + table + ws


def decode_flops(context_lens, num_q_heads, head_dim):
    """q.K and p.V multiply-adds: 4 * D flops per (position, q head)."""
    return int(np.asarray(context_lens, dtype=np.int64).sum()) * num_q_heads * 4 * head_dim


def write_bytes(num_tokens, num_kv_heads, head_dim, elem_bytes):
    """New K and V rows read, the same bytes written, plus the int64 slots."""
    return 2 * num_tokens * kv_bytes_per_token(num_kv_heads, head_dim, elem_bytes) + 8 * num_tokens


def copy_bytes(num_pairs, num_kv_heads, block_size, head_dim, elem_bytes):
    """Each pair reads and writes one whole block of both pools."""
    blk = num_kv_heads * block_size * head_dim * elem_bytes
    return num_pairs * (2 * 2 * blk + 8)


def cascade_workspace_bytes(context_lens, prefix_len, partition_size, num_q_heads, head_dim):
    """fp32 partials a cascade call writes and reads back: one prefix slot per (sequence,
    q head) row plus one per partition of each sequence's own suffix."""
    ctx = np.asarray(context_lens, dtype=np.int64)
    rest = np.maximum(ctx - int(prefix_len), 0)
    parts = 1 + (-(-rest // int(partition_size)))
    return 2 * int(parts.sum()) * num_q_heads * (head_dim + 2) * 4
