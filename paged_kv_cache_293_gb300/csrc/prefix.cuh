// prefix.cuh -- attention of every sequence's queries over a prefix all of them share.
//
// "Serving models with vLLM", section "How it works: PagedAttention": requests with
// the same prefix (system prompt, documents) point at the same physical blocks;
// "What Is vLLM", section "How does PagedAttention work?": prefix sharing.  When
// every sequence of a batch starts with the same prefix_len tokens in the same
// physical blocks, their attention over those tokens is one dense contraction per
// kv head: (num_seqs * G) query rows against prefix_len keys.  This kernel reads
// the shared pages once per CTA and runs both contractions on mma.sync tensor
// cores; the per-row result (max score, sum of weights, weighted sum of V) of
// each split of the prefix goes to its own workspace slot, before the
// partitions of each sequence's own suffix, and
// the log-sum-exp merge combines them -- the same arithmetic as attending to the
// whole context at once, regrouped.
//
// CTA: 4 compute warps x 16 query rows of one kv head, plus one warp whose lane 0
// feeds a six-stage ring: the prefix's 16-token chunks are staged by TMA tensor
// copies (128-byte swizzle) and completed on a per-stage "full" mbarrier; each
// compute warp releases a stage on its "empty" mbarrier when done with it, so no
// CTA-wide barrier holds the warps together.  Per chunk and compute warp:
//   S [16 rows x 16 tokens] = Q [16 x D] . K^T        (2 D/16 MMAs, B = K via ldmatrix)
//   O [16 rows x D]        += P [16 x 16] . V          (4 D/16 MMAs: P as a 16-bit high
//                                                       part and remainder, B = V via
//                                                       ldmatrix.trans)
// with the online softmax of each row in registers (rows g and g + 8 of a lane).
#pragma once

#include "decode_mma.cuh"

namespace pkv {

constexpr int PREFIX_STAGES = 6;

struct PrefixParams {
    const void* q;             // [S][Hq][D]
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t num_blocks;
    int32_t block_size;
    const int32_t* block_tables;  // [S][M]; row 0 holds the shared prefix's blocks
    int32_t max_blocks_per_seq;
    int32_t prefix_len;        // tokens, a multiple of 16 and of the block size
    float scale_log2;
    int32_t max_parts;         // workspace rows hold max_parts slots
    int32_t chunks_per_split;  // grid.z splits the prefix: split z writes slot z
    float* ws_m;
    float* ws_l;
    float* ws_o;
    unsigned int* err;
};

template <typename T, int D>
__global__ void __launch_bounds__(160, 3)
prefix_attention_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const PrefixParams p) {
    using Geo = MmaGeometry<D>;
    constexpr int KS = Geo::KSTEPS, NS = PREFIX_STAGES, NT = D / 8;
    constexpr int CONSUMERS = 4;  // warps 0-3 compute; warp 4 feeds the ring
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t ring_s = smem_addr(smem);
    const uint32_t full0 = smem_addr(smem + NS * Geo::STAGE_BYTES);   // chunk landed
    const uint32_t empty0 = full0 + NS * 8;                              // chunk released

    const int kvh = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int B = p.block_size;
    // this CTA's share of the prefix: chunks [c0, c0 + n_chunks)
    const int c0 = blockIdx.z * p.chunks_per_split;
    const int n_chunks = min(p.prefix_len / CHUNK_TOKENS - c0, p.chunks_per_split);

    if (threadIdx.x == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(full0 + st * 8, 1);
            mbar_init(empty0 + st * 8, CONSUMERS);
        }
        mbar_init_fence();
    }
    // every sequence of this tile must hold the same prefix blocks as sequence 0
    if (kvh == 0 && blockIdx.z == 0) {
        const int nb = p.prefix_len / B;
        const int s_lo = blockIdx.y * 64 / G;
        const int s_hi = min(p.num_seqs, (blockIdx.y * 64 + 63) / G + 1);
        for (int i = threadIdx.x; i < (s_hi - s_lo) * nb; i += blockDim.x) {
            const int s = s_lo + i / nb, j = i % nb;
            if (p.block_tables[(size_t)s * p.max_blocks_per_seq + j] != p.block_tables[j])
                set_error(p.err, PKV_DEVERR_PREFIX);
        }
    }
    __syncthreads();

    if (warp == CONSUMERS) {
        // ---- producer: one lane hands each chunk to the copy engine once its stage is free
        if (lane != 0) return;
        const uint64_t policy = l2_evict_first_policy();
        int issued = 0;
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c % NS;
            if (c >= NS && !mbar_wait(empty0 + st * 8, ((c / NS) - 1) & 1)) {
                set_error(p.err, PKV_DEVERR_TIMEOUT);
                break;
            }
            const uint32_t bar = full0 + st * 8;
            const int t = (c0 + c) * CHUNK_TOKENS;
            const int phys = __ldg(p.block_tables + t / B);
            if ((unsigned)phys >= (unsigned)p.num_blocks) {
                set_error(p.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive(bar);  // the consumers see a zero-byte phase and skip nothing else
            } else {
                const int row = (phys * p.num_kv_heads + kvh) * B + (t % B);
                const uint32_t dst = ring_s + st * Geo::STAGE_BYTES;
                mbar_arrive_expect_tx(bar, Geo::STAGE_BYTES);
#pragma unroll
                for (int b = 0; b < Geo::BOXES; ++b) {
                    tma_load_2d(dst + b * Geo::BOX_BYTES, &tmap_k, b * 64, row, bar, policy);
                    tma_load_2d(dst + Geo::POOL_BYTES + b * Geo::BOX_BYTES, &tmap_v, b * 64, row,
                                bar, policy);
                }
            }
            issued = c + 1;
        }
        // the CTA must not end with copies still landing in its shared memory
        for (int c = issued > NS ? issued - NS : 0; c < issued; ++c)
            mbar_wait(full0 + (c % NS) * 8, (c / NS) & 1);
        return;
    }

    // ---- consumers: 16 query rows per warp
    const int g4 = lane >> 2, q4 = lane & 3;
    const int rows = p.num_seqs * G;
    const int row_lo = blockIdx.y * 64 + warp * 16 + g4;  // this lane's rows: row_lo, row_lo + 8
    auto q_row = [&](int r) -> long long {
        return r < rows ? ((long long)(r / G) * p.num_q_heads + kvh * G + r % G) : -1;
    };
    const long long qr0 = q_row(row_lo), qr1 = q_row(row_lo + 8);

    // Q as mma A fragments (rows g4 / g4 + 8, dims of k-step ks)
    uint32_t qa[KS][4];
    {
        const T* q = static_cast<const T*>(p.q);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d = ks * 16 + 2 * q4;
            qa[ks][0] = qr0 >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(q + qr0 * D + d)) : 0u;
            qa[ks][1] = qr1 >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(q + qr1 * D + d)) : 0u;
            qa[ks][2] = qr0 >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(q + qr0 * D + d + 8)) : 0u;
            qa[ks][3] = qr1 >= 0 ? __ldg(reinterpret_cast<const uint32_t*>(q + qr1 * D + d + 8)) : 0u;
        }
    }

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    const int mi = lane >> 3, mr = lane & 7;

    for (int c = 0; c < n_chunks; ++c) {
        const int st = c % NS;
        if (!__all_sync(FULL_MASK, mbar_wait(full0 + st * 8, (c / NS) & 1))) {
            if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
            break;
        }
        const int t = (c0 + c) * CHUNK_TOKENS;
        const bool ok = (unsigned)__ldg(p.block_tables + t / B) < (unsigned)p.num_blocks;
        if (ok) {
            const uint32_t ks_s = ring_s + st * Geo::STAGE_BYTES;
            const uint32_t vs_s = ks_s + Geo::POOL_BYTES;
            // S = Q . K^T for tokens 0-7 (s0) and 8-15 (s1)
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int row = ((mi >> 1) << 3) + mr;       // token
                const int col = 2 * ks + (mi & 1);            // 16-byte column of dims
                uint32_t b0, b1, b2, b3;
                ldsm_x4(ks_s + (col / 8) * Geo::BOX_BYTES + swz(row, col & 7), b0, b1, b2, b3);
                Mma<T>::run(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                Mma<T>::run(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
            // online softmax: row g4 holds s0[0..1], s1[0..1]; row g4 + 8 holds [2..3]
            float pr0[4], pr1[4], alpha[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float a = s0[2 * h] * p.scale_log2, b = s0[2 * h + 1] * p.scale_log2;
                const float c_ = s1[2 * h] * p.scale_log2, d_ = s1[2 * h + 1] * p.scale_log2;
                float bm = fmaxf(fmaxf(a, b), fmaxf(c_, d_));
                bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, 2));
                const float mn = fmaxf(m[h], bm);
                alpha[h] = fast_exp2(m[h] - mn);
                m[h] = mn;
                pr0[2 * h] = fast_exp2(a - mn);
                pr0[2 * h + 1] = fast_exp2(b - mn);
                pr1[2 * h] = fast_exp2(c_ - mn);
                pr1[2 * h + 1] = fast_exp2(d_ - mn);
                l[h] = l[h] * alpha[h] + pr0[2 * h] + pr0[2 * h + 1] + pr1[2 * h] + pr1[2 * h + 1];
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
            }
            // P as A fragments: a0 row g4 tokens 2q4.., a1 row g4+8, a2/a3 the same for tokens 8..
            const uint32_t ah0 = Mma<T>::pack(pr0[0], pr0[1]), ah1 = Mma<T>::pack(pr0[2], pr0[3]);
            const uint32_t ah2 = Mma<T>::pack(pr1[0], pr1[1]), ah3 = Mma<T>::pack(pr1[2], pr1[3]);
            const uint32_t al0 = Mma<T>::pack(pr0[0] - Mma<T>::round_trip(pr0[0]),
                                              pr0[1] - Mma<T>::round_trip(pr0[1]));
            const uint32_t al1 = Mma<T>::pack(pr0[2] - Mma<T>::round_trip(pr0[2]),
                                              pr0[3] - Mma<T>::round_trip(pr0[3]));
            const uint32_t al2 = Mma<T>::pack(pr1[0] - Mma<T>::round_trip(pr1[0]),
                                              pr1[1] - Mma<T>::round_trip(pr1[1]));
            const uint32_t al3 = Mma<T>::pack(pr1[2] - Mma<T>::round_trip(pr1[2]),
                                              pr1[3] - Mma<T>::round_trip(pr1[3]));
            // O += P . V, two 8-dim column tiles per ldmatrix.x4.trans
#pragma unroll
            for (int dn = 0; dn < D / 16; ++dn) {
                const int row = ((mi & 1) << 3) + mr;         // token
                const int col = 2 * dn + (mi >> 1);            // 16-byte column of dims
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vs_s + (col / 8) * Geo::BOX_BYTES + swz(row, col & 7), b0, b1, b2, b3);
                Mma<T>::run(o[2 * dn], ah0, ah1, ah2, ah3, b0, b1);
                Mma<T>::run(o[2 * dn], al0, al1, al2, al3, b0, b1);
                Mma<T>::run(o[2 * dn + 1], ah0, ah1, ah2, ah3, b2, b3);
                Mma<T>::run(o[2 * dn + 1], al0, al1, al2, al3, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + st * 8);  // this warp is done with the stage
    }

    // rows' totals over the four lanes of a row
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(FULL_MASK, l[h], 1);
        l[h] += __shfl_xor_sync(FULL_MASK, l[h], 2);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const long long qr = h ? qr1 : qr0;
        if (qr < 0) continue;
        const size_t r = (size_t)qr * p.max_parts + blockIdx.z;
        float* orow = p.ws_o + r * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            orow[nt * 8 + 2 * q4] = o[nt][2 * h];
            orow[nt * 8 + 2 * q4 + 1] = o[nt][2 * h + 1];
        }
        if (q4 == 0) {
            p.ws_m[r] = m[h] * 0.69314718055994530942f;  // natural-log units
            p.ws_l[r] = l[h];
        }
    }
}

template <typename T, int D>
cudaError_t launch_prefix_td(const PrefixParams& p, const void* k_pool, const void* v_pool,
                             cudaStream_t stream) {
    constexpr int SMEM = PREFIX_STAGES * MmaGeometry<D>::STAGE_BYTES + 2 * PREFIX_STAGES * 8 + 1024;
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    if (rows >= (1ll << 31)) return cudaErrorNotSupported;
    if (!encode_pool_map<T>(&tk, k_pool, rows, D) || !encode_pool_map<T>(&tv, v_pool, rows, D))
        return cudaErrorNotSupported;
    const int G = p.num_q_heads / p.num_kv_heads;
    const long long tiles = ((long long)p.num_seqs * G + 63) / 64;
    if (tiles > 65535) return cudaErrorNotSupported;
    const int splits = (p.prefix_len / CHUNK_TOKENS + p.chunks_per_split - 1) / p.chunks_per_split;
    dim3 grid(p.num_kv_heads, (unsigned)tiles, splits);
    auto kernel = prefix_attention_kernel<T, D>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {false};
    if (dev < 64 && !configured[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    kernel<<<grid, 160, SMEM, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_prefix_impl(const PrefixParams& p, const void* k_pool, const void* v_pool,
                               int head_dim, cudaStream_t stream) {
    if (head_dim == 64) return launch_prefix_td<T, 64>(p, k_pool, v_pool, stream);
    if (head_dim == 128) return launch_prefix_td<T, 128>(p, k_pool, v_pool, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
