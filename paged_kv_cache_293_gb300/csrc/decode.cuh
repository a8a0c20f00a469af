// decode.cuh -- paged attention decode kernel (one query row per sequence and q head).
//
// "What Is vLLM: The Fast Inference Engine for Large Language Models", section
// "How does PagedAttention work?": every cached position of a sequence is
// found through its block table and read from the physical block that holds
// it.  Here one CTA owns (kv head, sequence, partition of P tokens) and all G
// q heads of that kv head's group, so every staged page serves G queries.
//
// Data path per CTA:
//  * the partition is cut into 16-token chunks; chunk c goes to warp c % NW;
//  * each warp runs its own NS-stage ring in shared memory: lane 0 looks the
//    chunk's physical block up in the block table and issues two 1-D bulk
//    copies (K rows, V rows: 16 * D * sizeof(T) contiguous bytes each, since a
//    (block, kv head) page is [B][D] row-major) that complete on the stage's
//    mbarrier; the warp waits on the barrier, computes, and refills the stage;
//  * scores: lanes are laid over the 16 x D chunk so that CPR = D*sizeof(T)/16
//    consecutive lanes read one row as 16-byte vectors (bank-conflict free);
//    partial dot products are reduced with a butterfly reduce-scatter so that
//    each lane ends with one token's full score per q head;
//  * online softmax in base 2 (scale * log2 e folded into q), fp32 running
//    max / sum per warp, fp32 P.V accumulation in registers;
//  * the NW warp states are combined in shared memory; a sequence that fits in
//    one partition writes out directly, otherwise (m, l, o) go to the
//    workspace for the log-sum-exp merge kernel.
// The order of every floating-point operation depends only on logical
// positions, so results do not depend on where blocks sit in the pool.
#pragma once

#include <cmath>

#include "pkv_common.cuh"

namespace pkv {

template <typename T, int D>
struct Geometry {
    static constexpr int PER_VEC = Elem<T>::PER_VEC;          // elements per lane vector
    static constexpr int ROW_BYTES = D * int(sizeof(T));
    static constexpr int CPR = ROW_BYTES / 16;                 // lanes per row
    static constexpr int RPP = 32 / CPR;                       // rows per pass
    static constexpr int PASSES = CHUNK_TOKENS / RPP;          // = CPR / 2
    static constexpr int CHUNK_BYTES = CHUNK_TOKENS * ROW_BYTES;
    static_assert(CPR == 8 || CPR == 16 || CPR == 32, "row must be 128, 256 or 512 bytes");
    static_assert(PASSES * RPP == CHUNK_TOKENS, "geometry");
};

template <typename T, int D, int NW, int NS>
struct DecodeSmem {
    using Geo = Geometry<T, D>;
    static constexpr int STAGE_BYTES = 2 * Geo::CHUNK_BYTES;
    static constexpr int RING_BYTES = NW * NS * STAGE_BYTES;
    static constexpr int BAR_OFFSET = RING_BYTES;
    static constexpr int BYTES = RING_BYTES + NW * NS * 8;
};

// Butterfly reduce-scatter over the CPR lanes that share a row group: NV = CPR/2
// partial sums per lane in, lane l out with the full sum of value index
// (l % CPR) >> 1 (the last exchange duplicates it in lanes l and l ^ 1).
template <int CPR>
__device__ __forceinline__ float reduce_scatter(float (&v)[CPR / 2], int lane) {
#pragma unroll
    for (int o = CPR / 2, nv = CPR / 2; o >= 2; o >>= 1, nv >>= 1) {
        const bool upper = (lane & o) != 0;
        const int half = nv / 2;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float send = upper ? v[j] : v[j + half];
            const float keep = upper ? v[j + half] : v[j];
            v[j] = keep + __shfl_xor_sync(FULL_MASK, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(FULL_MASK, v[0], 1);
}

template <typename T, int D, int G, int NW, int NS>
__global__ void __launch_bounds__(NW * 32)
paged_decode_kernel(const DecodeParams p) {
    using Geo = Geometry<T, D>;
    using Smem = DecodeSmem<T, D, NW, NS>;
    constexpr int CPR = Geo::CPR, RPP = Geo::RPP, PASSES = Geo::PASSES, PV = Geo::PER_VEC;
    constexpr int ROWB = Geo::ROW_BYTES, CHB = Geo::CHUNK_BYTES;

    extern __shared__ __align__(128) unsigned char smem[];

    // partitions launch last-first: the highest ones exist only for the longest sequences,
    // so the CTAs left running at the end are first partitions, many of them short
    const int kvh = blockIdx.x, s = blockIdx.y, part = gridDim.z - 1 - blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.block_size, Hkv = p.num_kv_heads, Hq = p.num_q_heads, P = p.partition_size;

    int ctx = p.context_lens[s];
    bool ctx_bad = false;
    {
        const long long cap_table = (long long)p.max_blocks_per_seq * B;
        const long long cap_grid =
            (long long)p.skip_tokens + (long long)(p.max_parts - p.part_offset) * P;
        long long cap = cap_table < cap_grid ? cap_table : cap_grid;
        if (cap > p.max_context_len) cap = p.max_context_len;
        if (ctx < 0 || ctx > cap) {
            if (threadIdx.x == 0 && part == 0 && kvh == 0) set_error(p.err, PKV_DEVERR_CONTEXT);
            ctx = ctx < 0 ? 0 : int(cap);
            ctx_bad = true;
        }
    }
    const int skip = p.skip_tokens;
    const int n_parts = ctx > skip ? (ctx - skip + P - 1) / P : 0;
    const int tok0 = skip + part * P;
    if (part > 0 && tok0 >= ctx) return;
    const bool direct = p.direct_single && n_parts <= 1;

    if ((ctx == 0 || ctx_bad) && p.slot_out && kvh == 0 && part == 0 && threadIdx.x == 0)
        p.slot_out[s] = -1;
    if (ctx <= skip) {  // nothing to attend to here: zero output or an empty partial
        if (ctx < skip && threadIdx.x == 0 && blockIdx.x == 0) set_error(p.err, PKV_DEVERR_CONTEXT);
        for (int i = threadIdx.x; i < G * D; i += NW * 32) {
            const int h = kvh * G + i / D, d = i % D;
            const size_t row = (size_t)s * Hq + h;
            if (direct) {
                store_out(p.out, p.out_dtype, row * D + d, 0.f);
            } else {
                const size_t r = row * p.max_parts + p.part_offset;
                p.ws_o[r * D + d] = 0.f;
                if (d == 0) { p.ws_m[r] = -INFINITY; p.ws_l[r] = 0.f; }
            }
        }
        return;
    }

    const int tok_end = min(ctx, tok0 + P);
    const int n_chunks = (tok_end - tok0 + CHUNK_TOKENS - 1) / CHUNK_TOKENS;
    const int n_my = warp < n_chunks ? (n_chunks - warp + NW - 1) / NW : 0;

    // ---- queries of the group, scaled into base-2 score units
    float qf[G][PV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(
                              static_cast<const T*>(p.q) + ((size_t)s * Hq + kvh * G + g) * D) +
                          (lane % CPR));
        Elem<T>::to_float(raw, qf[g]);
#pragma unroll
        for (int e = 0; e < PV; ++e) qf[g][e] *= p.scale_log2;
    }

    // ---- per-warp ring
    unsigned char* ring = smem + warp * NS * Smem::STAGE_BYTES;
    const uint32_t ring_s = smem_addr(ring);
    const uint32_t bar0 = smem_addr(smem + Smem::BAR_OFFSET) + warp * NS * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NS; ++st) mbar_init(bar0 + st * 8, 1);
        mbar_init_fence();
    }
    __syncwarp();

    const int32_t* bt_row = p.block_tables + (size_t)s * p.max_blocks_per_seq;

    // ---- fused append: the partition holding position ctx - 1 writes the new K/V rows
    // of its kv head into their slot and splices them into the staged chunk.
    const int p_new = ctx - 1;
    const bool has_new = p.k_new != nullptr && !ctx_bad && p_new >= tok0 && p_new < tok_end;
    const int c_new = has_new ? (p_new - tok0) / CHUNK_TOKENS : -1;
    const bool warp_new = has_new && (c_new % NW) == warp;
    uint4 k_row = make_uint4(0, 0, 0, 0), v_row = make_uint4(0, 0, 0, 0);
    int phys_new = -1;
    if (warp_new) {
        phys_new = __ldg(bt_row + p_new / B);
        if (lane < CPR) {
            const size_t src = ((size_t)s * Hkv + kvh) * D;
            k_row = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src) + lane);
            v_row = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src) + lane);
        }
    }
    const T* kbase = static_cast<const T*>(p.k_pool);
    const T* vbase = static_cast<const T*>(p.v_pool);
    const uint64_t policy = l2_evict_first_policy();

    // Physical block of my i-th chunk, loaded 32 chunks at a time (lane j holds chunk base+j).
    auto table_entry = [&](int i) -> int {
        if (i >= n_my) return -1;
        const int t = tok0 + (warp + NW * i) * CHUNK_TOKENS;
        return __ldg(bt_row + t / B);
    };
    int ids = table_entry(lane);
    uint32_t bad_stages = 0;

    auto issue = [&](int i) {
        if ((i & 31) == 0 && i > 0) ids = table_entry(i + lane);
        const int phys = __shfl_sync(FULL_MASK, ids, i & 31);
        const int st = i % NS;
        const bool ok = (unsigned)phys < (unsigned)p.num_blocks;
        bad_stages = ok ? (bad_stages & ~(1u << st)) : (bad_stages | (1u << st));
        if (lane == 0) {
            const uint32_t bar = bar0 + st * 8;
            if (ok) {
                const int t = tok0 + (warp + NW * i) * CHUNK_TOKENS;
                const size_t off = (((size_t)phys * Hkv + kvh) * B + (t % B)) * D;
                const uint32_t dst = ring_s + st * Smem::STAGE_BYTES;
                mbar_arrive_expect_tx(bar, 2 * CHB);
                bulk_g2s(dst, kbase + off, CHB, bar, policy);
                bulk_g2s(dst + CHB, vbase + off, CHB, bar, policy);
            } else {
                set_error(p.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive(bar);
            }
        }
    };

    float m[G], l[G], acc[G][PV];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < PV; ++e) acc[g][e] = 0.f;
    }

    const int row_grp = lane / CPR;   // which row of a pass this lane reads
    const int col = lane % CPR;       // which 16-byte column
    const int my_tok = (col >> 1) * RPP + row_grp;  // token whose full score this lane ends with

    const int n_pro = n_my < NS ? n_my : NS;
    for (int i = 0; i < n_pro; ++i) issue(i);

    for (int i = 0; i < n_my; ++i) {
        const int st = i % NS;
        if (!mbar_wait(bar0 + st * 8, (i / NS) & 1)) {
            if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
            // give the copies still in flight a bounded chance to land, then stop
            for (int j = i + 1; j < n_my && j < i + NS; ++j) mbar_wait(bar0 + (j % NS) * 8, (j / NS) & 1);
            break;
        }
        const int c = warp + NW * i;
        const int valid = min(CHUNK_TOKENS, tok_end - (tok0 + c * CHUNK_TOKENS));
        if (warp_new && c == c_new) {
            const bool ok = (unsigned)phys_new < (unsigned)p.num_blocks;
            if (ok && lane < CPR) {
                unsigned char* Kw = ring + st * Smem::STAGE_BYTES;
                const int r = (p_new - tok0) & (CHUNK_TOKENS - 1);
                *reinterpret_cast<uint4*>(Kw + r * ROWB + lane * 16) = k_row;
                *reinterpret_cast<uint4*>(Kw + CHB + r * ROWB + lane * 16) = v_row;
                const size_t off = (((size_t)phys_new * Hkv + kvh) * B + (p_new % B)) * D;
                reinterpret_cast<uint4*>(const_cast<T*>(kbase) + off)[lane] = k_row;
                reinterpret_cast<uint4*>(const_cast<T*>(vbase) + off)[lane] = v_row;
            }
            if (p.slot_out && kvh == 0 && lane == 0)
                p.slot_out[s] = ok ? (int64_t)phys_new * B + (p_new % B) : -1;
            // the spliced rows are ordinary stores: order them before any later bulk copy
            // into this stage (none today: the new token's chunk is the warp's last)
            fence_proxy_async_shared();
            __syncwarp();
        }
        if (!((bad_stages >> st) & 1)) {
            const unsigned char* Ks = ring + st * Smem::STAGE_BYTES;
            const unsigned char* Vs = Ks + CHB;

            // scores
            float part_s[G][PASSES];
#pragma unroll
            for (int k = 0; k < PASSES; ++k) {
                const int t = k * RPP + row_grp;
                const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * ROWB + col * 16);
                float kf[PV];
                Elem<T>::to_float(raw, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < PV; ++e) a = fmaf(qf[g][e], kf[e], a);
                    part_s[g][k] = a;
                }
            }
            float pr[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float sc = reduce_scatter<CPR>(part_s[g], lane);
                if (my_tok >= valid) sc = -INFINITY;
                float bm = sc;
#pragma unroll
                for (int o = 16; o >= 2; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, o));
                const float mn = fmaxf(m[g], bm);
                const float alpha = fast_exp2(m[g] - mn);
                pr[g] = fast_exp2(sc - mn);
                l[g] = l[g] * alpha + ((lane & 1) ? 0.f : pr[g]);
                m[g] = mn;
#pragma unroll
                for (int e = 0; e < PV; ++e) acc[g][e] *= alpha;
            }
            // P.V
            const int src_base = lane & ~(CPR - 1);
#pragma unroll
            for (int k = 0; k < PASSES; ++k) {
                const int t = k * RPP + row_grp;
                const uint4 raw = *reinterpret_cast<const uint4*>(Vs + t * ROWB + col * 16);
                float vf[PV];
                Elem<T>::to_float(raw, vf);
                if (valid < CHUNK_TOKENS && t >= valid) {
#pragma unroll
                    for (int e = 0; e < PV; ++e) vf[e] = 0.f;
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float pt = __shfl_sync(FULL_MASK, pr[g], src_base | (2 * k));
#pragma unroll
                    for (int e = 0; e < PV; ++e) acc[g][e] = fmaf(pt, vf[e], acc[g][e]);
                }
            }
        }
        __syncwarp();
        if (i + NS < n_my) issue(i + NS);
    }

    // ---- warp totals: rows of a pass hold different tokens, lanes of a pair duplicate l
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int o = CPR; o < 32; o <<= 1)
#pragma unroll
            for (int e = 0; e < PV; ++e) acc[g][e] += __shfl_xor_sync(FULL_MASK, acc[g][e], o);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l[g] += __shfl_xor_sync(FULL_MASK, l[g], o);
    }

    // ---- combine the NW warps in shared memory (the ring is free now)
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem);  // [NW][G][D + 2]
    if (lane < CPR) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < PV; ++e) red[(warp * G + g) * (D + 2) + lane * PV + e] = acc[g][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            red[(warp * G + g) * (D + 2) + D] = m[g];
            red[(warp * G + g) * (D + 2) + D + 1] = l[g];
        }
    }
    __syncthreads();

    for (int i = threadIdx.x; i < G * D; i += NW * 32) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, red[(w * G + g) * (D + 2) + D]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* r = red + (w * G + g) * (D + 2);
            const float f = fast_exp2(r[D] - M);
            L = fmaf(r[D + 1], f, L);
            O = fmaf(r[d], f, O);
        }
        const size_t row = (size_t)s * Hq + kvh * G + g;
        if (direct) {
            store_out(p.out, p.out_dtype, row * D + d, O / L);
        } else {
            const size_t r = row * p.max_parts + part + p.part_offset;
            p.ws_o[r * D + d] = O;
            if (d == 0) {
                p.ws_m[r] = M * 0.69314718055994530942f;  // back to natural-log units
                p.ws_l[r] = L;
            }
        }
    }
}

// Ring shape: NW warps per CTA, NS stages per warp, sized so that a CTA holds
// 64 KB of ring and three CTAs (12 warps) fit on an SM.  Measured on the
// LLaMA-13B batch: 4 warps x 2 stages of 8 KB beat 3-4 stages or 2 / 8 warps.
template <typename T, int D> struct DecodeShape {
    static constexpr int STAGE = 2 * Geometry<T, D>::CHUNK_BYTES;
    static constexpr int NW = STAGE > 8192 ? 2 : 4;
    static constexpr int NS = (64 * 1024) / (NW * STAGE);
};

template <typename T, int D, int G>
cudaError_t launch_decode_tdg(const DecodeParams& p, cudaStream_t stream) {
    constexpr int NW = DecodeShape<T, D>::NW, NS = DecodeShape<T, D>::NS;
    constexpr int SMEM = DecodeSmem<T, D, NW, NS>::BYTES;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(NW * NS * 2 * Geometry<T, D>::CHUNK_BYTES >= NW * G * (D + 2) * 4,
                  "reduction scratch must fit in the ring");
    auto kernel = paged_decode_kernel<T, D, G, NW, NS>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> configured[64];  // per device; setting it twice is harmless
    if (dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    dim3 grid(p.num_kv_heads, p.num_seqs, p.max_parts - p.part_offset);
    kernel<<<grid, NW * 32, SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_decode_impl(const DecodeParams& p, int head_dim, int group, cudaStream_t stream) {
#define PKV_CASE(DV, GV) \
    if (head_dim == DV && group == GV) return launch_decode_tdg<T, DV, GV>(p, stream);
    PKV_CASE(64, 1) PKV_CASE(64, 2) PKV_CASE(64, 4) PKV_CASE(64, 8)
    PKV_CASE(128, 1) PKV_CASE(128, 2) PKV_CASE(128, 4) PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
