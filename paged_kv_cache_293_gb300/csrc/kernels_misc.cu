// kernels_misc.cu -- slot mapping, cache write, copy-on-write block copy and the
// log-sum-exp merge of partitioned decode.
#include <cmath>

#include "pkv_common.cuh"

namespace pkv {

// ------------------------------------------------------------------ slot mapping
// "What Is vLLM", section "How does PagedAttention work?": the physical block
// that holds position p is the table entry of logical block p / B; the row is p % B.
__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_tables, int32_t M,
                                    int32_t S, const int32_t* __restrict__ positions,
                                    const int32_t* __restrict__ token_seq, int32_t T, int32_t B,
                                    int64_t* __restrict__ slots, unsigned int* err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int s = token_seq ? token_seq[t] : t;
    const int p = positions[t];
    if (p < 0) { slots[t] = -1; return; }
    const int j = p / B;
    if (s < 0 || s >= S || j >= M) {
        set_error(err, PKV_DEVERR_POSITION);
        slots[t] = -1;
        return;
    }
    const int phys = block_tables[(size_t)s * M + j];
    if (phys < 0) {
        set_error(err, PKV_DEVERR_BLOCK_ID);
        slots[t] = -1;
        return;
    }
    slots[t] = (int64_t)phys * B + (p - j * B);
}

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_seqs, const int32_t* positions,
                                const int32_t* token_seq, int32_t num_tokens, int32_t block_size,
                                int64_t* slot_mapping, unsigned int* err, cudaStream_t stream) {
    const int threads = 128;
    const int blocks = (num_tokens + threads - 1) / threads;
    slot_mapping_kernel<<<blocks, threads, 0, stream>>>(block_tables, max_blocks_per_seq, num_seqs,
                                                        positions, token_seq, num_tokens,
                                                        block_size, slot_mapping, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ cache write
// One thread per 16-byte vector of a (token, kv head) row, for K and V.
__global__ void cache_write_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                   const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                   const int64_t* __restrict__ slots, int32_t T, int32_t Hkv,
                                   int32_t B, int32_t vpr, long long num_slots,
                                   unsigned int* err) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long per_tok = (long long)Hkv * vpr;
    if (idx >= (long long)T * per_tok) return;
    const int t = int(idx / per_tok);
    const int rem = int(idx - (long long)t * per_tok);
    const int h = rem / vpr, v = rem - h * vpr;
    const long long slot = slots[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (rem == 0) set_error(err, PKV_DEVERR_SLOT);
        return;
    }
    const long long blk = slot / B, row = slot - blk * B;
    const size_t dst = (size_t)(((blk * Hkv + h) * B + row) * vpr + v);
    const uint4 kv = k_new[idx];
    const uint4 vv = v_new[idx];
    k_pool[dst] = kv;
    v_pool[dst] = vv;
}

static int elem_bytes(int32_t dtype) { return dtype == PKV_F32 ? 4 : 2; }

cudaError_t launch_cache_write(const pkv_pool& pool, const void* k_new, const void* v_new,
                               const int64_t* slot_mapping, int32_t num_tokens, unsigned int* err,
                               cudaStream_t stream) {
    const int vpr = pool.head_dim * elem_bytes(pool.dtype) / 16;
    const long long total = (long long)num_tokens * pool.num_kv_heads * vpr;
    const int threads = 256;
    const long long blocks = (total + threads - 1) / threads;
    cache_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<uint4*>(pool.k), static_cast<uint4*>(pool.v),
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping,
        num_tokens, pool.num_kv_heads, pool.block_size, vpr,
        (long long)pool.num_blocks * pool.block_size, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ block copy between pools
// Copy-on-write inside one pool ("What Is vLLM", section "How does PagedAttention
// work?", step "Memory sharing") and swapping between a device pool and a pool in
// pinned host memory (same page, "What is continuous batching in vLLM?": preempted
// sequences' KV caches move to the CPU).  grid = (pairs, slices of a block, 2 pools);
// 16-byte vectors.
__global__ void copy_blocks_kernel(const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                                   uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                                   int32_t src_blocks, int32_t dst_blocks, long long vec_per_block,
                                   const int32_t* __restrict__ pairs, unsigned int* err) {
    const int i = blockIdx.x;
    const int src = pairs[2 * i], dst = pairs[2 * i + 1];
    if ((unsigned)src >= (unsigned)src_blocks || (unsigned)dst >= (unsigned)dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, PKV_DEVERR_PAIR);
        return;
    }
    const uint4* from = (blockIdx.z == 0 ? src_k : src_v) + (size_t)src * vec_per_block;
    uint4* to = (blockIdx.z == 0 ? dst_k : dst_v) + (size_t)dst * vec_per_block;
    for (long long j = (long long)blockIdx.y * blockDim.x + threadIdx.x; j < vec_per_block;
         j += (long long)gridDim.y * blockDim.x)
        to[j] = from[j];
}

cudaError_t launch_copy_blocks(const pkv_pool& src, const pkv_pool& dst, const int32_t* pairs,
                               int32_t num_pairs, unsigned int* err, cudaStream_t stream) {
    const long long vec = (long long)src.num_kv_heads * src.block_size * src.head_dim *
                          elem_bytes(src.dtype) / 16;
    const int threads = 256;
    long long slices = (vec + threads * 4 - 1) / (threads * 4);
    if (slices > 65535) slices = 65535;
    dim3 grid((unsigned)num_pairs, (unsigned)slices, 2);
    copy_blocks_kernel<<<grid, threads, 0, stream>>>(
        static_cast<const uint4*>(src.k), static_cast<const uint4*>(src.v),
        static_cast<uint4*>(dst.k), static_cast<uint4*>(dst.v), src.num_blocks, dst.num_blocks,
        vec, pairs, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ log-sum-exp merge
// Row (s, h) with n = prefix_parts + ceil((ctx - skip_tokens) / P) partitions:
//   M = max_k m_k,  out = sum_k e^(m_k - M) o_k / sum_k e^(m_k - M) l_k.
// Both kernels are launched as programmatic dependents of the decode kernel: their
// launch overlaps the decode's last CTAs, and griddepcontrol.wait holds them until the
// decode grid's partials are complete and visible.

__device__ __forceinline__ int merge_parts(const MergeParams& p, long long row) {
    const int s = int(row / ((long long)p.num_q_heads * p.num_queries));
    int ctx = p.context_lens[s];
    const long long cap = (long long)p.skip_tokens +
                          (long long)(p.max_parts - p.prefix_parts) * p.partition_size;
    if (ctx < 0) ctx = 0;
    if (ctx > cap) ctx = int(cap);
    const int rest = ctx > p.skip_tokens ? ctx - p.skip_tokens : 0;
    return p.prefix_parts + (rest + p.partition_size - 1) / p.partition_size;
}

template <int D> struct MergeVec;
template <> struct MergeVec<128> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void load(const float* src, float (&v)[4]) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    }
};
template <> struct MergeVec<64> {
    static constexpr int N = 2;
    __device__ __forceinline__ static void load(const float* src, float (&v)[2]) {
        const float2 x = *reinterpret_cast<const float2*>(src);
        v[0] = x.x; v[1] = x.y;
    }
};

// Up to 8 partitions per row: one warp per row, 8 rows per CTA.  Lane k holds
// partition k's weight; lane j holds dims [j * V, (j + 1) * V) of the sum.
template <int D>
__global__ void __launch_bounds__(256) lse_merge_rows_kernel(const MergeParams p, long long rows) {
    constexpr int V = MergeVec<D>::N;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + warp;
    if (row >= rows) return;
    const float* mrow = p.ws_m + (size_t)row * p.max_parts;
    const float* lrow = p.ws_l + (size_t)row * p.max_parts;
    const float* orow = p.ws_o + (size_t)row * p.max_parts * D;
    // every load at once (all max_parts <= 8 slots of the row; the ones past this row's
    // partition count are read and then ignored), so the row costs one memory round trip
    float lk = 0.f, mk = -INFINITY;
    if (lane < p.max_parts) {
        lk = lrow[lane];
        mk = mrow[lane];
    }
    float v[8][V];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < p.max_parts) MergeVec<D>::load(orow + (size_t)k * D + lane * V, v[k]);
    const int n = merge_parts(p, row);
    if (p.skip_single && n <= 1) return;
    if (lane >= n || !(lk > 0.f)) {
        lk = 0.f;
        mk = -INFINITY;
    }
    float M = mk;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, o));
    const size_t out_base = (size_t)row * D + lane * V;
    if (M == -INFINITY) {
#pragma unroll
        for (int j = 0; j < V; ++j) store_out(p.out, p.out_dtype, out_base + j, 0.f);
        return;
    }
    const float w = lk > 0.f ? fast_exp2((mk - M) * 1.4426950408889634f) : 0.f;
    float L = w * lk;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(FULL_MASK, L, o);
    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float wk = __shfl_sync(FULL_MASK, w, k);
        if (k < n) {
#pragma unroll
            for (int j = 0; j < V; ++j) acc[j] = fmaf(wk, v[k][j], acc[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < V; ++j) store_out(p.out, p.out_dtype, out_base + j, acc[j] / L);
}

// Many partitions: one CTA of 16 warps per row; warp w takes partitions w, w + 16, ...
// with eight loads in flight, and the warps' sums meet in shared memory.
template <int D>
__global__ void __launch_bounds__(512) lse_merge_kernel(const MergeParams p) {
    constexpr int NWM = 16, V = MergeVec<D>::N;
    __shared__ float red[NWM][D + 1];
    __shared__ float smax[NWM];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = merge_parts(p, row);
    if (p.skip_single && n <= 1) return;
    const float* mrow = p.ws_m + (size_t)row * p.max_parts;
    const float* lrow = p.ws_l + (size_t)row * p.max_parts;
    const float* orow = p.ws_o + (size_t)row * p.max_parts * D;

    float M = -INFINITY;
    for (int k = threadIdx.x; k < n; k += NWM * 32)
        if (lrow[k] > 0.f) M = fmaxf(M, mrow[k]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL_MASK, M, o));
    if (lane == 0) smax[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NWM; ++w) M = fmaxf(M, smax[w]);
    const size_t out_base = (size_t)row * D;
    if (M == -INFINITY) {
        for (int d = threadIdx.x; d < D; d += NWM * 32) store_out(p.out, p.out_dtype, out_base + d, 0.f);
        return;
    }
    float L = 0.f, acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.f;
#pragma unroll 8
    for (int k = warp; k < n; k += NWM) {
        const float lk = lrow[k];
        const float wk = lk > 0.f ? fast_exp2((mrow[k] - M) * 1.4426950408889634f) : 0.f;
        float v[V];
        MergeVec<D>::load(orow + (size_t)k * D + lane * V, v);
        L = fmaf(wk, lk, L);
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = fmaf(wk, v[j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < V; ++j) red[warp][lane * V + j] = acc[j];
    if (lane == 0) red[warp][D] = L;
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += NWM * 32) {
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < NWM; ++w) { num += red[w][d]; den += red[w][D]; }
        store_out(p.out, p.out_dtype, out_base + d, num / den);
    }
}

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const long long rows = (long long)p.num_seqs * p.num_queries * p.num_q_heads;
    if (rows == 0) return cudaSuccess;
    if (p.head_dim != 64 && p.head_dim != 128) return cudaErrorInvalidValue;
    const bool few = p.max_parts <= 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(few ? (unsigned)((rows + 7) / 8) : (unsigned)rows);
    cfg.blockDim = dim3(few ? 256 : 512);  // 8 rows of one warp each, or 16 warps on one row
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (few)
        return p.head_dim == 64 ? cudaLaunchKernelEx(&cfg, lse_merge_rows_kernel<64>, p, rows)
                                : cudaLaunchKernelEx(&cfg, lse_merge_rows_kernel<128>, p, rows);
    return p.head_dim == 64 ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<64>, p)
                            : cudaLaunchKernelEx(&cfg, lse_merge_kernel<128>, p);
}

}  // namespace pkv
