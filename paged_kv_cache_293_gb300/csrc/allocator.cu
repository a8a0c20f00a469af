// allocator.cu -- the block pool's bookkeeping on the device: a stack of free
// physical block ids and a reference count per block, updated in batches (one
// launch per step) instead of by a host loop.
//
// "vLLM in Production", section "PagedAttention - Virtual Memory for the KV
// Cache": the engine grows a sequence one block at a time as tokens arrive.
// "What Is vLLM", section "How does PagedAttention work?": blocks are
// allocated on demand; sequences that share a prefix share physical blocks,
// with reference counting and copy-on-write.  "Serving models with vLLM",
// section "How it works: PagedAttention": requests with the same prefix point
// at the same physical blocks.
//
// Concurrency: a kernel either only takes ids from the stack (allocation) or
// only returns ids to it (free), never both, so a pop is one atomic decrement
// of the count (undone when the stack is empty) and a push one atomic
// increment.  A shared partly filled block receiving new tokens is copied by
// every appending holder except the last reference, decided by the value an
// atomic decrement of its count returns.
#include "pkv_common.cuh"

namespace pkv {

namespace {

// Take one id from the stack; -1 when it is empty.
__device__ __forceinline__ int pop_block(const AllocatorState& a) {
    const int idx = atomicSub(a.free_count, 1) - 1;
    if (idx < 0) {
        atomicAdd(a.free_count, 1);
        return -1;
    }
    return a.free_ids[idx];
}

__device__ __forceinline__ void push_block(const AllocatorState& a, int id) {
    const int idx = atomicAdd(a.free_count, 1);
    a.free_ids[idx] = id;
}

}  // namespace

// Every block free (the stack pops 0, 1, 2, ... first), every count zero.
__global__ void allocator_reset_kernel(AllocatorState a) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) *a.free_count = a.num_blocks;
    if (i < a.num_blocks) {
        a.free_ids[i] = a.num_blocks - 1 - i;
        a.refcount[i] = 0;
    }
}

// One CTA per sequence growing from old_lens[s] to new_lens[s] tokens.
// Thread 0 does the bookkeeping in order (copy-on-write of a shared last
// block, then one fresh block per new logical block); the CTA then copies the
// shared block's rows for every kv head of both pools.
__global__ void __launch_bounds__(256)
allocate_for_append_kernel(AllocatorState a, uint4* k_pool, uint4* v_pool, long long vec_per_block,
                           int32_t B, int32_t* block_tables, int32_t M,
                           const int32_t* old_lens, const int32_t* new_lens,
                           int32_t* seq_status, unsigned int* err) {
    const int s = blockIdx.x;
    __shared__ int copy_src, copy_dst;
    if (threadIdx.x == 0) {
        copy_src = copy_dst = -1;
        int status = 0;
        const int old_len = old_lens[s], new_len = new_lens[s];
        int32_t* row = block_tables + (size_t)s * M;
        if (old_len < 0 || new_len < old_len || (long long)new_len > (long long)M * B) {
            status = 2;
        } else if (new_len > old_len) {
            if (old_len % B != 0) {  // the last block is partly filled and will receive tokens
                const int j = (old_len - 1) / B;
                const int b = row[j];
                if ((unsigned)b >= (unsigned)a.num_blocks) {
                    set_error(err, PKV_DEVERR_BLOCK_ID);
                    status = 2;
                } else if (atomicSub(&a.refcount[b], 1) == 1) {
                    atomicAdd(&a.refcount[b], 1);  // the last reference keeps the block
                } else {
                    const int nb = pop_block(a);
                    if (nb < 0) {
                        atomicAdd(&a.refcount[b], 1);
                        status = 1;
                    } else {
                        a.refcount[nb] = 1;
                        row[j] = nb;
                        copy_src = b;
                        copy_dst = nb;
                    }
                }
            }
            const int first = (old_len + B - 1) / B, last = (new_len + B - 1) / B;
            for (int j = first; j < last && status == 0; ++j) {
                const int nb = pop_block(a);
                if (nb < 0) {
                    status = 1;
                    break;
                }
                a.refcount[nb] = 1;
                row[j] = nb;
            }
        }
        seq_status[s] = status;
    }
    __syncthreads();
    if (copy_src >= 0) {
        const uint4* ks = k_pool + (size_t)copy_src * vec_per_block;
        const uint4* vs = v_pool + (size_t)copy_src * vec_per_block;
        uint4* kd = k_pool + (size_t)copy_dst * vec_per_block;
        uint4* vd = v_pool + (size_t)copy_dst * vec_per_block;
        for (long long i = threadIdx.x; i < vec_per_block; i += blockDim.x) {
            kd[i] = ks[i];
            vd[i] = vs[i];
        }
    }
}

// pairs[i] = (src sequence, dst sequence): dst's first ceil(len / B) table
// entries become src's, and each of those blocks gains a reference.
__global__ void fork_sequences_kernel(AllocatorState a, int32_t B, int32_t* block_tables,
                                      int32_t M, const int32_t* pairs, const int32_t* lens,
                                      int32_t n, unsigned int* err) {
    const int i = blockIdx.x;
    const int src = pairs[2 * i], dst = pairs[2 * i + 1];
    const int len = lens[i];
    const int nb = (len + B - 1) / B;
    if (len < 0 || nb > M) {
        if (threadIdx.x == 0) set_error(err, PKV_DEVERR_CONTEXT);
        return;
    }
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        const int b = block_tables[(size_t)src * M + j];
        if ((unsigned)b >= (unsigned)a.num_blocks) {
            set_error(err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        block_tables[(size_t)dst * M + j] = b;
        atomicAdd(&a.refcount[b], 1);
    }
}

// Each listed sequence drops one reference from each of its blocks; a block
// whose count reaches zero goes back onto the stack.  Its table row is cleared.
__global__ void free_sequences_kernel(AllocatorState a, int32_t B, int32_t* block_tables,
                                      int32_t M, const int32_t* seqs, const int32_t* lens,
                                      int32_t n, unsigned int* err) {
    const int i = blockIdx.x;
    const int s = seqs[i];
    const int len = lens[i];
    const int nb = (len + B - 1) / B;
    if (len < 0 || nb > M) {
        if (threadIdx.x == 0) set_error(err, PKV_DEVERR_CONTEXT);
        return;
    }
    int32_t* row = block_tables + (size_t)s * M;
    for (int j = threadIdx.x; j < nb; j += blockDim.x) {
        const int b = row[j];
        row[j] = -1;
        if ((unsigned)b >= (unsigned)a.num_blocks) {
            set_error(err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        if (atomicSub(&a.refcount[b], 1) == 1) push_block(a, b);
    }
}

static int elem_bytes_of(int32_t dtype) { return dtype == PKV_F32 ? 4 : 2; }

cudaError_t launch_allocator_reset(const AllocatorState& a, cudaStream_t stream) {
    const int threads = 256;
    allocator_reset_kernel<<<(a.num_blocks + threads - 1) / threads, threads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_allocate_for_append(const AllocatorState& a, const pkv_pool& pool,
                                       int32_t* block_tables, int32_t M, const int32_t* old_lens,
                                       const int32_t* new_lens, int32_t num_seqs,
                                       int32_t* seq_status, unsigned int* err,
                                       cudaStream_t stream) {
    const long long vec = (long long)pool.num_kv_heads * pool.block_size * pool.head_dim *
                          elem_bytes_of(pool.dtype) / 16;
    allocate_for_append_kernel<<<num_seqs, 256, 0, stream>>>(
        a, static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v), vec, pool.block_size,
        block_tables, M, old_lens, new_lens, seq_status, err);
    return cudaGetLastError();
}

cudaError_t launch_fork_sequences(const AllocatorState& a, int32_t B, int32_t* block_tables,
                                  int32_t M, const int32_t* pairs, const int32_t* lens, int32_t n,
                                  unsigned int* err, cudaStream_t stream) {
    fork_sequences_kernel<<<n, 128, 0, stream>>>(a, B, block_tables, M, pairs, lens, n, err);
    return cudaGetLastError();
}

cudaError_t launch_free_sequences(const AllocatorState& a, int32_t B, int32_t* block_tables,
                                  int32_t M, const int32_t* seqs, const int32_t* lens, int32_t n,
                                  unsigned int* err, cudaStream_t stream) {
    free_sequences_kernel<<<n, 128, 0, stream>>>(a, B, block_tables, M, seqs, lens, n, err);
    return cudaGetLastError();
}

}  // namespace pkv
