// pkv_common.cuh -- device helpers shared by the paged KV-cache kernels (sm_103a).
//
// Inline PTX for the Blackwell bulk-copy engine (cp.async.bulk, 1-D, no tensor
// map, no multicast) and its mbarrier completion, bounded waits, element
// conversions to fp32, and the parameter blocks the host shim fills.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr unsigned FULL_MASK = 0xffffffffu;
constexpr int CHUNK_TOKENS = 16;  // tokens staged per pipeline stage
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;  // 2 s

// ------------------------------------------------------------------ parameter blocks

struct DecodeParams {
    const void* k_pool;
    const void* v_pool;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    const void* q;
    int32_t num_seqs;
    int32_t num_q_heads;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t max_context_len;
    float scale_log2;       // scale * log2(e): scores are kept in base 2
    int32_t partition_size; // tokens per partition, multiple of block_size
    int32_t max_parts;      // grid.z
    void* out;
    int32_t out_dtype;
    int32_t direct_single;  // 1: sequences with one partition write out directly
    int32_t skip_tokens;    // attend to positions >= skip_tokens only (0: the whole context)
    int32_t part_offset;    // partition k writes workspace slot k + part_offset
    int32_t num_queries;    // query rows per sequence (1 for decode)
    int32_t queries_per_cta;  // tensor-core kernel: queries sharing one CTA's 8 columns
    float* ws_m;
    float* ws_l;
    float* ws_o;
    // Fused append (null when off): the new token of sequence s sits at position
    // context_lens[s] - 1; its K/V rows k_new[s], v_new[s] ([S][Hkv][D]) are written
    // into that slot of the pools and used in place of the rows read from them.
    const void* k_new;
    const void* v_new;
    int64_t* slot_out;      // optional: the slot each new token went to (-1: none)
    unsigned int* err;
    // tensor-core kernel, 1: every CTA lets the next launch in the stream (programmatic
    // dependent launch) begin as soon as it starts, so that launch fills the SMs this
    // grid's last CTAs leave idle; it must not read what this grid writes
    int32_t trigger_dependents;
};

struct MergeParams {
    const float* ws_m;
    const float* ws_l;
    const float* ws_o;
    const int32_t* context_lens;
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t head_dim;
    int32_t max_parts;
    int32_t partition_size;
    int32_t skip_single;    // 1: rows with <= 1 partition were written by the decode kernel
    int32_t num_queries;    // rows are [num_seqs][num_queries][num_q_heads]
    int32_t prefix_parts;   // slots before the context's partitions (1: a shared-prefix partial)
    int32_t skip_tokens;    // the partitions cover positions >= skip_tokens
    void* out;
    int32_t out_dtype;
    unsigned int* err;
};

// Device-side block bookkeeping (allocator.cu): a stack of free ids and counts.
struct AllocatorState {
    int32_t* free_ids;
    int32_t* free_count;
    int32_t* refcount;
    int32_t num_blocks;
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of the barrier; false once limit_ns nanoseconds have passed
// without it completing (the caller then sets PKV_DEVERR_TIMEOUT and stops).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// L2 policy for data read once per call: evict first, so the block tables,
// queries and partial results stay resident.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// 16 bytes global -> shared through L1, asynchronously; both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Order this thread's generic-proxy global writes before later tensor-copy (async
// proxy) reads of the same addresses.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Order this thread's generic-proxy writes to shared memory (st.shared, cp.async) before a
// later bulk or tensor copy (async proxy) that overwrites the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Wait for this thread's cp.async copies.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_error(unsigned int* err, unsigned int bits) {
    atomicOr(err, bits);
}

// ------------------------------------------------------------------ chunk order

// Order in which a warp of the tensor-core decode kernel walks its n chunks (the warp's
// k-th chunk in position order is chunk warp + NW * k): alternately one from the front
// and one from the back of its list -- 0, n-1, 1, n-2, ...  When sequences share their
// first blocks (a common prefix, "Serving models with vLLM", section "How it works:
// PagedAttention"), the front chunks are mostly served from L2 and the back ones from
// DRAM; alternating keeps every warp's DRAM copies in flight while it works through the
// shared chunks, instead of a run of L2-only steps at the start of each CTA (measured
// 4-5 us faster on a 256-sequence batch sharing 512 tokens, neutral without sharing; the
// CUDA-core kernel, which serves MHA batches, measured about 1 % slower with it and keeps
// the plain order).  The order depends on logical positions only, so results still do
// not depend on where blocks sit in the pool.
__device__ __forceinline__ int alternating_chunk(int i, int n) {
    return (i & 1) ? n - 1 - (i >> 1) : (i >> 1);
}

// ------------------------------------------------------------------ element types

template <typename T> struct Elem;

template <> struct Elem<float> {
    static constexpr int PER_VEC = 4;  // elements per 16-byte vector
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
};

template <> struct Elem<__half> {
    static constexpr int PER_VEC = 8;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 v = __half22float2(h);
            f[2 * i] = v.x; f[2 * i + 1] = v.y;
        }
    }
};

template <> struct Elem<__nv_bfloat16> {
    static constexpr int PER_VEC = 8;
    __device__ __forceinline__ static void to_float(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

__device__ __forceinline__ void store_out(void* out, int32_t out_dtype, size_t i, float v) {
    if (out_dtype == PKV_F32)
        static_cast<float*>(out)[i] = v;
    else if (out_dtype == PKV_F16)
        static_cast<__half*>(out)[i] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
}

// ------------------------------------------------------------------ host launchers (internal)

// Which decode kernel serves a group of G q heads per kv head on 16-bit pools
// (set by pkv_set_decode_engine): tensor cores when G >= 4 by default.
bool use_tensor_cores(int group);

template <typename T>
cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, cudaStream_t stream);
// the tensor-core kernel alone (16-bit pools); cudaErrorNotSupported when the pool
// cannot be described by a tensor map
template <typename T>
cudaError_t launch_decode_mma(const DecodeParams& p, int head_dim, int group, cudaStream_t stream);

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
struct PrefixParams;
// attention over a shared prefix into workspace slot 0 (16-bit pools, prefix.cuh)
template <typename T>
cudaError_t launch_prefix(const PrefixParams& p, const void* k_pool, const void* v_pool,
                          int head_dim, cudaStream_t stream);
cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_seqs, const int32_t* positions,
                                const int32_t* token_seq, int32_t num_tokens, int32_t block_size,
                                int64_t* slot_mapping, unsigned int* err, cudaStream_t stream);
cudaError_t launch_cache_write(const pkv_pool& pool, const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, int32_t num_tokens, unsigned int* err,
                               cudaStream_t stream);
cudaError_t launch_allocator_reset(const AllocatorState& a, cudaStream_t stream);
cudaError_t launch_allocate_for_append(const AllocatorState& a, const pkv_pool& pool,
                                       int32_t* block_tables, int32_t M, const int32_t* old_lens,
                                       const int32_t* new_lens, int32_t num_seqs,
                                       int32_t* seq_status, unsigned int* err,
                                       cudaStream_t stream);
cudaError_t launch_fork_sequences(const AllocatorState& a, int32_t B, int32_t* block_tables,
                                  int32_t M, const int32_t* pairs, const int32_t* lens, int32_t n,
                                  unsigned int* err, cudaStream_t stream);
cudaError_t launch_free_sequences(const AllocatorState& a, int32_t B, int32_t* block_tables,
                                  int32_t M, const int32_t* seqs, const int32_t* lens, int32_t n,
                                  unsigned int* err, cudaStream_t stream);
cudaError_t launch_copy_blocks(const pkv_pool& src, const pkv_pool& dst, const int32_t* pairs,
                               int32_t num_pairs, unsigned int* err, cudaStream_t stream);

}  // namespace pkv
