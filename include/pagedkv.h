/*
 * pagedkv.h -- C ABI of libpagedkv.so, paged KV-cache decode for GB300 (sm_103a).
 *
 * The method: the KV cache of each sequence is cut into fixed-size blocks that
 * can sit anywhere in GPU memory; a per-sequence block table maps logical
 * blocks to physical blocks; attention for the new token of a sequence reads
 * every cached position through that table ("What Is vLLM: The Fast Inference
 * Engine for Large Language Models", section "How does PagedAttention work?";
 * "vLLM in Production", section "PagedAttention - Virtual Memory for the KV
 * Cache"; "Serving models with vLLM", section "How it works: PagedAttention").
 *
 * Conventions shared by every entry point:
 *  - All array arguments are DEVICE pointers to caller-owned memory.  The
 *    library allocates nothing and keeps no handle to caller memory.
 *  - stream is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Every call is asynchronous on that stream and returns after
 *    enqueueing its kernels; nothing synchronises inside a call (except
 *    pkv_get_device_error, which says so).
 *  - Host-checkable argument errors are returned before anything is launched.
 *    A failed launch returns PKV_ERR_CUDA.  Index errors only the device can
 *    see (a table entry outside the pool, a slot past the pool, a context
 *    longer than its table row) skip the offending work and set bits in a
 *    device error word that pkv_get_device_error() reads back; kernels never
 *    trap, assert or wait without a limit.
 *  - Element types: PKV_F32, PKV_F16, PKV_BF16.  q, k_new and v_new have the
 *    pool's element type.  Decode output is fp32 or the pool's type.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,      /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0 ... */
    PKV_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, block size, group size, dtype */
    PKV_ERR_WORKSPACE = 3,    /* partitioned decode without a large enough workspace */
    PKV_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE = 5        /* pkv_get_device_error found error bits set */
} pkv_status;

typedef enum pkv_dtype { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2 } pkv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_BLOCK_ID 0x1u  /* a block-table entry that a position needs is outside [0, num_blocks) */
#define PKV_DEVERR_SLOT     0x2u  /* a slot at or past num_blocks * block_size */
#define PKV_DEVERR_CONTEXT  0x4u  /* context_len < 0, > max_blocks_per_seq * B or > max_context_len */
#define PKV_DEVERR_TIMEOUT  0x8u  /* a copy pipeline wait ran out of time (about 2 s) */
#define PKV_DEVERR_POSITION 0x10u /* slot mapping: position past the table row, or bad sequence index */
#define PKV_DEVERR_PAIR     0x20u /* copy_blocks: a src or dst outside [0, num_blocks) */
#define PKV_DEVERR_PREFIX   0x40u /* cascade decode: a sequence's prefix blocks differ from sequence 0's */

/*
 * The physical block pool: two caller-owned device arrays, K and V, each laid
 * out [num_blocks][num_kv_heads][block_size][head_dim], row-major, head_dim
 * innermost.  One (block, kv head) page is block_size * head_dim contiguous
 * elements; one physical block across all kv heads is
 * num_kv_heads * block_size * head_dim contiguous elements.  k and v must be
 * 16-byte aligned.  Built: block_size in {16, 32}, head_dim in {64, 128}.
 */
typedef struct pkv_pool {
    void* k;
    void* v;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t dtype; /* pkv_dtype */
} pkv_pool;

/*
 * Slot of each token to append: slot_mapping[t] = block_tables[s][p / B] * B + p % B,
 * with s = token_seq[t] (or t when token_seq is NULL) and p = positions[t].
 * "What Is vLLM", section "How does PagedAttention work?": the engine looks up
 * which physical block holds a position and indexes into it.
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]
 *   positions     int32 [num_tokens]; p < 0 gives slot -1 (padding)
 *   token_seq     int32 [num_tokens] or NULL
 *   slot_mapping  int64 [num_tokens] (output)
 * Device errors: p / B >= max_blocks_per_seq or s outside [0, num_seqs)
 * (PKV_DEVERR_POSITION), a negative table entry (PKV_DEVERR_BLOCK_ID); the
 * slot is then -1.
 */
pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            int32_t num_seqs, const int32_t* positions, const int32_t* token_seq,
                            int32_t num_tokens, int32_t block_size, int64_t* slot_mapping,
                            void* stream);

/*
 * Append new tokens: for each t with slot_mapping[t] >= 0 and every kv head h,
 * k_pool[slot / B][h][slot % B][:] = k_new[t][h][:] and the same for V (bit
 * copy).  "vLLM in Production", section "PagedAttention - Virtual Memory for
 * the KV Cache": a sequence grows one block at a time as tokens arrive.
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim] in the pool type, 16-byte aligned
 *   slot_mapping   int64 [num_tokens]; negative = skip
 * Slots within one call must be distinct.  A slot >= num_blocks * B is
 * skipped and sets PKV_DEVERR_SLOT.
 */
pkv_status pkv_kv_cache_write(const pkv_pool* pool, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, int32_t num_tokens, void* stream);

/*
 * Partition size (tokens) that pkv_paged_attention_decode uses when it is
 * given partition_size = 0: a multiple of the block size; a value >=
 * max_context_len means one pass with no workspace.  Returns 0 on bad input.
 */
int32_t pkv_choose_partition_size(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len);

/*
 * Workspace bytes a decode or partition call needs for these sizes
 * (partition_size 0 = the automatic choice).  0 when one pass suffices.
 * Layout, with P parts = ceil(max_context_len / partition_size) and
 * R = num_seqs * num_q_heads rows, all fp32:
 *   m [R][P]    at byte 0                    largest scaled score of the range
 *   l [R][P]    at byte A = align16(4 R P)   sum of exp(score - m)
 *   o [R][P][D] at byte 2 A                  sum of exp(score - m) * V, not divided by l
 */
size_t pkv_decode_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, int32_t partition_size);

/*
 * Workspace bytes pkv_paged_attention_partitions needs: the layout above with
 * ceil(max_context_len / partition_size) parts (at least one).  0 on bad input.
 */
size_t pkv_partition_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                     int32_t max_context_len, int32_t partition_size);

/*
 * Paged attention decode, one query row per sequence and q head:
 *   out[s][h] = softmax(scale * q[s][h] . K_s^T) V_s
 * over the context_lens[s] cached positions of sequence s, whose K and V rows
 * are read in logical order through block_tables[s] from kv head
 * h / (num_q_heads / num_kv_heads).  "vLLM in Production", section "The KV
 * Cache and the 60-80% Memory Tax": each new token attends to every previous
 * token through the cache.  context 0 gives a zero row.
 *   q             [num_seqs][num_q_heads][head_dim], pool type, 16-byte aligned
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(context_lens[s] / B) are never read
 *   context_lens  int32 [num_seqs]
 *   max_context_len  host-side upper bound of context_lens (sizes the grid)
 *   out           [num_seqs][num_q_heads][head_dim] of out_dtype (PKV_F32 or the pool type)
 *   partition_size   0 = automatic; otherwise a multiple of block_size.  When
 *                 ceil(max_context_len / partition_size) > 1 each partition of a
 *                 sequence is reduced separately into the workspace and a
 *                 log-sum-exp merge kernel writes out.
 *   workspace     device memory of at least pkv_decode_workspace_bytes(...)
 *                 bytes, 16-byte aligned, or NULL when none is needed.
 * Built group sizes num_q_heads / num_kv_heads: 1, 2, 4, 8.
 */
pkv_status pkv_paged_attention_decode(const pkv_pool* pool, const void* q, int32_t num_seqs,
                                      int32_t num_q_heads, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      int32_t max_context_len, float scale, void* out,
                                      int32_t out_dtype, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, void* stream);

/*
 * Append and decode in one launch: for every sequence s with
 * context_lens[s] >= 1, the new token sits at position p = context_lens[s] - 1
 * (the context includes it).  Its rows k_new[s][h], v_new[s][h] are written
 * into slot block_tables[s][p / B] * B + p % B of both pools, and the
 * attention over positions [0, context_lens[s]) uses them for position p.
 * The result (output and pools) is that of pkv_slot_mapping with positions =
 * context_lens - 1, then pkv_kv_cache_write, then pkv_paged_attention_decode,
 * with one launch instead of three ("vLLM in Production", section
 * "PagedAttention - Virtual Memory for the KV Cache": the cache grows as tokens
 * arrive; each new token then attends to all cached tokens).
 *   k_new, v_new   [num_seqs][num_kv_heads][head_dim], pool type, 16-byte aligned
 *   slot_mapping   optional int64 [num_seqs] output: the slot written (-1 for
 *                  an empty context or a bad table entry); NULL to skip
 * The block receiving a new token must belong to that sequence alone (copy it
 * on write first when it is shared).  Other arguments as in
 * pkv_paged_attention_decode.
 */
pkv_status pkv_paged_attention_decode_append(
    const pkv_pool* pool, const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, void* out,
    int32_t out_dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
    int64_t* slot_mapping, void* stream);

/*
 * Attention for several new tokens per sequence (the tail of a chunked prefill
 * or the draft tokens of speculative decoding: "Serving models with vLLM",
 * section "How it works: inference serving with vLLM", names both; "How it
 * works: continuous batching" describes chunked prefill).  The last
 * num_queries positions of sequence s are its new tokens, already written to
 * the cache (pkv_kv_cache_write with token_seq slots); query j (0-based)
 * attends causally to positions [0, context_lens[s] - num_queries + j]:
 *   out[s][j][h] = softmax(scale * q[s][j][h] . K_s[0..c_j)^T) V_s[0..c_j),
 *   c_j = context_lens[s] - num_queries + 1 + j   (a row with c_j <= 0 is zero).
 *   q, out   [num_seqs][num_queries][num_q_heads][head_dim]
 * fp16 / bf16 pools only (PKV_ERR_UNSUPPORTED for fp32); always the
 * tensor-core kernel, whose 8 columns hold (query, q head) pairs of one kv
 * head: 8 / G queries share one pass over the pages, and more queries take
 * further passes.  The workspace (when partitioned) is that of
 * pkv_decode_workspace_bytes(pool, num_seqs * num_queries, num_q_heads, ...),
 * its rows ordered [num_seqs][num_queries][num_q_heads].  Other arguments as
 * in pkv_paged_attention_decode.
 */
pkv_status pkv_paged_attention_decode_multi(
    const pkv_pool* pool, const void* q, int32_t num_queries, int32_t num_seqs,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, void* out,
    int32_t out_dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
    void* stream);

/*
 * pkv_paged_attention_decode_multi with the new tokens' K/V rows appended in the
 * same launch: position context_lens[s] - num_queries + j of sequence s receives
 * k_new[s][j], v_new[s][j] in slot block_tables[s][p / B] * B + p % B of both
 * pools, and the attention uses them for that position.  The result (output and
 * pools) is that of pkv_slot_mapping over those positions, pkv_kv_cache_write,
 * then pkv_paged_attention_decode_multi, in one launch instead of three
 * ("Serving models with vLLM", section "How it works: PagedAttention": the cache
 * grows block by block as tokens arrive).
 *   k_new, v_new   [num_seqs][num_queries][num_kv_heads][head_dim], pool type,
 *                  16-byte aligned
 *   slot_mapping   optional int64 [num_seqs][num_queries] output: the slot each
 *                  token went to (-1 for a position outside the context or a bad
 *                  table entry, which also sets PKV_DEVERR_BLOCK_ID); NULL to skip
 * The blocks receiving new tokens must belong to their sequence alone (copy them
 * on write first when shared).  Other arguments as in
 * pkv_paged_attention_decode_multi.
 */
pkv_status pkv_paged_attention_decode_multi_append(
    const pkv_pool* pool, const void* q, const void* k_new, const void* v_new,
    int32_t num_queries, int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
    float scale, void* out, int32_t out_dtype, int32_t partition_size, void* workspace,
    size_t workspace_bytes, int64_t* slot_mapping, void* stream);

/*
 * Decode for a batch whose sequences all begin with the same prefix_len tokens
 * held in the same physical blocks (a shared system prompt: "Serving models
 * with vLLM", section "How it works: PagedAttention": requests with the same
 * prefix point at the same physical blocks).  Same result as
 * pkv_paged_attention_decode (or, with k_new / v_new, as
 * pkv_paged_attention_decode_append), computed in three launches: the paged
 * decode of each sequence's own positions [prefix_len, context_lens[s]) in
 * partitions of partition_size (0 = automatic); the attention of all sequences'
 * queries over the shared prefix, read once per kv head and run on tensor cores
 * (launched so that it may start on the SMs the first launch's last CTAs leave
 * idle); and the log-sum-exp merge of the two.
 *   prefix_len   > 0, a multiple of 16 and of block_size, <= every context length;
 *                the first prefix_len / B table entries of every sequence must equal
 *                sequence 0's (checked on the device: PKV_DEVERR_PREFIX)
 *   k_new, v_new optional ([num_seqs][num_kv_heads][head_dim]): append each
 *                sequence's new token at position context_lens[s] - 1 (which must
 *                lie past the prefix) as the fused entry point does; NULL for none
 *   slot_mapping optional output as in pkv_paged_attention_decode_append
 *   workspace    pkv_cascade_workspace_bytes(...) bytes, always required
 * fp16 / bf16 pools only (PKV_ERR_UNSUPPORTED for fp32).  PKV_ERR_UNSUPPORTED also
 * for a pool of 2^31 or more (block, kv head, position) rows or more than
 * 65535 x 128 query rows (num_seqs x group size); every such error is returned
 * before anything is launched.
 */
size_t pkv_cascade_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_context_len, int32_t prefix_len,
                                   int32_t partition_size);
pkv_status pkv_paged_attention_decode_cascade(
    const pkv_pool* pool, const void* q, int32_t num_seqs, int32_t num_q_heads,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, float scale, int32_t prefix_len, void* out, int32_t out_dtype,
    int32_t partition_size, const void* k_new, const void* v_new, int64_t* slot_mapping,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The partition step alone: for every sequence s, q head h and partition
 * k < ceil(context_lens[s] / partition_size), writes (m, l, o) of tokens
 * [k P, min(ctx, (k+1) P)) to the workspace in the layout above (a context
 * of 0 writes m = -inf, l = 0, o = 0 at k = 0).  Lets a caller reduce token
 * ranges separately (for example on several devices) and combine them with
 * pkv_lse_merge.  partition_size > 0, a multiple of block_size.
 */
pkv_status pkv_paged_attention_partitions(const pkv_pool* pool, const void* q, int32_t num_seqs,
                                          int32_t num_q_heads, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t max_context_len,
                                          float scale, int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * Log-sum-exp merge of partition results (layout above):
 *   M = max_k m_k,  out = sum_k exp(m_k - M) o_k / sum_k exp(m_k - M) l_k
 * over k < ceil(context_lens[s] / partition_size); rows with no tokens give 0.
 */
pkv_status pkv_lse_merge(const void* workspace, size_t workspace_bytes, int32_t num_seqs,
                         int32_t num_q_heads, int32_t head_dim, const int32_t* context_lens,
                         int32_t max_context_len, int32_t partition_size, void* out,
                         int32_t out_dtype, void* stream);

/*
 * Decode without a caller-provided workspace.  The pages have no counterpart
 * to this: it exists for callers that cannot allocate device memory
 * themselves, for example a plugin whose host engine owns every device
 * allocation and forbids new ones while it enqueues work, or a caller reaching
 * this library through a foreign-function layer that has no device allocator.
 * Same arguments and result as pkv_paged_attention_decode, minus the
 * workspace.  When the call needs partition scratch (see
 * pkv_decode_workspace_bytes), it uses a fixed array inside libpagedkv.so of
 * PKV_STATIC_WORKSPACE_BYTES bytes; every GPU that loads the library holds that
 * array until the process exits.  A call that would need more returns
 * PKV_ERR_WORKSPACE without launching anything (a larger partition_size needs
 * less).  The call allocates nothing: no cudaMalloc, no cudaFree.
 * The first call on a device looks the array's device address up
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.
 * All calls share the one array and it keeps the last call's contents; the
 * kernels write every partial result before reading it, so nothing needs
 * clearing.  Calls whose kernels overlap on the GPU (different streams, or
 * different host threads without ordering) race on the array and give
 * undefined results: order them on one stream.
 */
#define PKV_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)

pkv_status pkv_paged_attention_decode_static_workspace(
    const pkv_pool* pool, const void* q, int32_t num_seqs, int32_t num_q_heads,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, float scale, void* out, int32_t out_dtype, int32_t partition_size,
    void* stream);

/*
 * Copy-on-write of shared blocks: for each pair i, physical block
 * src_dst_pairs[2i+1] of both pools becomes a bit copy of block
 * src_dst_pairs[2i] (all kv heads, all rows).  "What Is vLLM", section "How
 * does PagedAttention work?", step "Memory sharing": blocks shared by several
 * sequences are reference counted and copied on write.
 *   src_dst_pairs  int32 [num_pairs][2] on the device
 * dst blocks must be distinct and must not be sources in the same call.  A
 * pair with an id outside the pool is skipped and sets PKV_DEVERR_PAIR.
 */
pkv_status pkv_copy_blocks(const pkv_pool* pool, const int32_t* src_dst_pairs, int32_t num_pairs,
                           void* stream);

/*
 * Move whole blocks between two pools of the same geometry (dtype, block
 * size, kv heads, head_dim): for each pair i, block src_dst_pairs[2i+1] of dst
 * becomes a bit copy of block src_dst_pairs[2i] of src, K and V.  For
 * preemption, a sequence's blocks go from the GPU pool to a pool in host
 * memory and back later ("What Is vLLM", section "What is continuous batching
 * in vLLM?": low-priority sequences are preempted and their KV caches swapped
 * to CPU memory).  The copies run in a kernel that reads and writes both pools
 * directly, so either pool may be device memory or pinned host memory the GPU
 * can address (cudaHostAlloc / cudaMallocHost; with unified addressing its
 * host pointer is valid on the device); src_dst_pairs (int32 [num_pairs][2])
 * must be device-addressable too.  Every pointer is checked with
 * cudaPointerGetAttributes first: pinned host memory is used through its mapped
 * device address, and memory the runtime does not know (plain pageable host
 * memory) returns PKV_ERR_INVALID.  dst blocks must be distinct and must not
 * overlap the src blocks read in the same call.  Pairs outside either pool are
 * skipped and set PKV_DEVERR_PAIR.
 */
pkv_status pkv_swap_blocks(const pkv_pool* src, const pkv_pool* dst, const int32_t* src_dst_pairs,
                           int32_t num_pairs, void* stream);

/*
 * Block bookkeeping on the device.  "vLLM in Production", section
 * "PagedAttention - Virtual Memory for the KV Cache": a sequence grows one
 * block at a time as tokens arrive; "What Is vLLM", section "How does
 * PagedAttention work?": blocks are allocated on demand, and sequences sharing
 * a prefix share physical blocks through reference counting and copy-on-write.
 * The state is three caller-owned device arrays; every call below is one
 * launch on `stream` covering a whole batch of sequences, so a step's
 * allocation needs no round trip to the host.
 *   free_ids    int32 [num_blocks]: free physical ids; entries [0, *free_count) are valid
 *   free_count  int32 [1]
 *   refcount    int32 [num_blocks]: how many table entries point at each block
 * Which free id a request receives depends on the order the GPU serves
 * requests in; counts, statuses and the sequences' contents do not.
 */
typedef struct pkv_block_allocator {
    int32_t* free_ids;
    int32_t* free_count;
    int32_t* refcount;
    int32_t num_blocks;
} pkv_block_allocator;

/* Every block free, every count zero. */
pkv_status pkv_allocator_reset(const pkv_block_allocator* alloc, void* stream);

/*
 * Sequence s grows from old_lens[s] to new_lens[s] tokens (int32 [num_seqs]
 * each, device).  When old_lens[s] is not a multiple of B, the partly filled
 * last block receives tokens: if other references to it remain, it is first
 * copied to a fresh block (K and V, all kv heads) that replaces it in the
 * table, and the original loses one reference (copy-on-write; of several
 * holders appending in one call, the last reference keeps the original).  Then
 * each logical block ceil(old / B) .. ceil(new / B) - 1 gets a fresh block
 * with one reference.  seq_status[s] (int32, device, output): 0 done,
 * 1 out of free blocks (what was allocated for s stays; later table entries
 * are left as they were; the caller preempts or frees), 2 lengths invalid or
 * the table row too short (nothing done for s).  Table rows of different
 * sequences must be distinct memory.
 */
pkv_status pkv_allocate_for_append(const pkv_block_allocator* alloc, const pkv_pool* pool,
                                   int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* old_lens, const int32_t* new_lens,
                                   int32_t num_seqs, int32_t* seq_status, void* stream);

/*
 * Share blocks: for each pair i (src_dst_seqs int32 [num_pairs][2], device),
 * sequence dst's first ceil(lens[i] / B) table entries become those of src
 * and each of those blocks gains one reference (prefix sharing, or beam
 * candidates branching from one sequence).  dst rows must hold no references
 * (empty or freed) and must not be a src in the same call.
 */
pkv_status pkv_fork_sequences(const pkv_block_allocator* alloc, int32_t block_size,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* src_dst_seqs, const int32_t* lens,
                              int32_t num_pairs, void* stream);

/*
 * Release sequences (finished, or preempted after their blocks were swapped
 * out): each of the first ceil(lens[i] / B) blocks of sequence seqs[i] loses
 * one reference, a block left with none goes back to the free stack, and the
 * table entries become -1.  seqs must be distinct.
 */
pkv_status pkv_free_sequences(const pkv_block_allocator* alloc, int32_t block_size,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seqs, const int32_t* lens, int32_t num_seqs,
                              void* stream);

/*
 * Synchronises stream, then reads and clears the current device's error word
 * into *flags (host pointer).  Returns PKV_ERR_DEVICE when any bit was set.
 */
pkv_status pkv_get_device_error(uint32_t* flags, void* stream);

/*
 * Which decode kernel serves fp16 / bf16 pools (process-wide; fp32 pools always
 * use the CUDA-core kernel):
 *   PKV_ENGINE_AUTO          tensor cores (mma.sync, TMA-staged pages) when a kv
 *                            head serves >= 4 q heads, CUDA cores otherwise
 *   PKV_ENGINE_CUDA_CORES    always the CUDA-core kernel
 *   PKV_ENGINE_TENSOR_CORES  always the tensor-core kernel (q heads padded to 8)
 * Both give the same result within rounding; the choice is about speed.  A
 * pool of 2^31 or more rows (num_blocks * num_kv_heads * block_size) always
 * uses the CUDA-core kernel.  Returns PKV_ERR_INVALID for another value.
 */
#define PKV_ENGINE_AUTO 0
#define PKV_ENGINE_CUDA_CORES 1
#define PKV_ENGINE_TENSOR_CORES 2
pkv_status pkv_set_decode_engine(int32_t engine);
int32_t pkv_get_decode_engine(void);

/* Static text for a status code. */
const char* pkv_status_str(pkv_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
