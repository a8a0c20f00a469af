// decode_mma.cuh -- paged attention decode for grouped-query heads on the tensor cores.
//
// Same method and result as decode.cuh ("What Is vLLM", section "How does
// PagedAttention work?": every cached position is found through the block table
// and read from the physical block holding it), for kv heads shared by G >= 4 q
// heads.  There the G query rows against a 16-token chunk form a small dense
// tile, so both contractions run on mma.sync.m16n8k16 (fp32 accumulate):
//
//   scores^T [16 tokens x 8 heads] = K_chunk [16 x D] . Q^T [D x 8]      (D/16 MMAs)
//   O^T      [D x 8 heads]        += V_chunk^T [D x 16] . P^T [16 x 8]    (2 D/16 MMAs)
//
// with the G query heads padded to the 8 columns of the N dimension.  P is
// split into a 16-bit high part and a 16-bit remainder (two MMAs), so the
// probabilities enter the P.V product with about 16 significant bits instead of
// the 8 of a single bf16 rounding.
//
// Pages are staged by TMA tensor copies (cp.async.bulk.tensor.3d) through a
// tensor map over the pool viewed as [rows = N*Hkv*B][D / 64][64]: one copy per
// pool brings a 16-token chunk of a page as D*2/128 boxes of [16 rows][64
// elements], landing in shared memory with the 128-byte swizzle, which makes the
// ldmatrix reads of both K (row-major) and V (transposed) free of bank conflicts.
// Each warp runs its own mbarrier ring as in decode.cuh, but walks its chunks
// alternately from the front and the back of its list (alternating_chunk); the
// NW warp states are combined in shared memory at the end.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "pkv_common.cuh"

namespace pkv {

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// One copy of a 3-D box: the D/64 column halves of a chunk's rows land as consecutive
// [16 rows][128 bytes] swizzled boxes, the same layout as D/64 2-D copies.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

template <typename T> struct Mma;

template <> struct Mma<__nv_bfloat16> {
    __device__ __forceinline__ static void run(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // (lo, hi) -> packed pair, low 16 bits = lo; also the rounding remainders.
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float round_trip(float x) {
        return __bfloat162float(__float2bfloat16_rn(x));
    }
    static constexpr CUtensorMapDataType TMA_TYPE = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};

template <> struct Mma<__half> {
    __device__ __forceinline__ static void run(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __device__ __forceinline__ static float round_trip(float x) {
        return __half2float(__float2half_rn(x));
    }
    static constexpr CUtensorMapDataType TMA_TYPE = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
};

// ------------------------------------------------------------------ shared-memory geometry

// A chunk of one pool: D / 64 boxes of [16 rows][128 bytes], 128-byte swizzled:
// the 16-byte column j of row r sits at r * 128 + ((j ^ (r & 7)) * 16).
template <int D>
struct MmaGeometry {
    static constexpr int BOXES = D / 64;             // 64 two-byte elements per box row
    static constexpr int BOX_BYTES = CHUNK_TOKENS * 128;
    static constexpr int POOL_BYTES = BOXES * BOX_BYTES;   // one pool's chunk
    static constexpr int STAGE_BYTES = 2 * POOL_BYTES;     // K then V
    static constexpr int KSTEPS = D / 16;
    static_assert(D == 64 || D == 128, "head_dim");
};

template <int D, int NW, int NS>
struct MmaSmem {
    using Geo = MmaGeometry<D>;
    static constexpr int RING_BYTES = NW * NS * Geo::STAGE_BYTES;
    static constexpr int RED_BYTES = NW * 8 * (D + 2) * 4;
    static constexpr int DATA_BYTES = RING_BYTES > RED_BYTES ? RING_BYTES : RED_BYTES;
    static constexpr int BAR_OFFSET = DATA_BYTES;
    static constexpr int BYTES = DATA_BYTES + NW * NS * 8 + 1024;  // + alignment slack
};

__device__ __forceinline__ uint32_t swz(int row, int col16) {
    return uint32_t(row * 128 + ((col16 ^ (row & 7)) << 4));
}

// Columns of the 8-wide N tile: n = (query j - j0) * G + g for the CTA's queries
// j0 .. j0 + nj - 1 and the G q heads g of kv head kvh.  With one query per
// sequence (decode) the columns are just the G heads of the group.
// Several appended tokens (the last num_queries positions of the context, rows of
// k_new / v_new [S][NQ][Hkv][D]).  Each warp writes the new rows of its own chunks to
// their pool slots (append_rows_to_pool) before it issues those chunks' tensor copies,
// which then bring them; a chunk whose copy was issued earlier (one of the first NS of
// the warp) gets them put into its staged rows after it lands (append_rows_into_chunk).
// Compiled only into the kernel variant for several appended tokens per sequence.
template <typename T, int D>
__device__ __forceinline__ void append_rows_to_pool(const DecodeParams& p, const int32_t* bt_row,
                                                    int s, int kvh, int ctx, int t_lo, int t_hi,
                                                    int lane) {
    constexpr int VPR = D * 2 / 16;  // 16-byte vectors per row
    constexpr int RPP = 32 / VPR;    // rows per warp-wide pass
    constexpr int BATCH = 4;         // passes whose loads are in flight together
    const int NQ = p.num_queries, Hkv = p.num_kv_heads, B = p.block_size;
    const int sub = lane / VPR, col = lane % VPR;
    for (int base = t_lo; base < t_hi; base += RPP * BATCH) {
        uint4 kr[BATCH], vr[BATCH];
        int phys[BATCH];
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int pj = base + b * RPP + sub;
            phys[b] = -1;
            if (pj < t_hi) {
                const size_t src = (((size_t)s * NQ + pj - (ctx - NQ)) * Hkv + kvh) * D;
                phys[b] = __ldg(bt_row + pj / B);
                kr[b] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src) + col);
                vr[b] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src) + col);
            }
        }
#pragma unroll
        for (int b = 0; b < BATCH; ++b) {
            const int pj = base + b * RPP + sub;
            if (pj < t_hi && (unsigned)phys[b] < (unsigned)p.num_blocks) {
                const size_t dst = (((size_t)phys[b] * Hkv + kvh) * B + (pj % B)) * D;
                reinterpret_cast<uint4*>(const_cast<T*>(static_cast<const T*>(p.k_pool)) + dst)[col] = kr[b];
                reinterpret_cast<uint4*>(const_cast<T*>(static_cast<const T*>(p.v_pool)) + dst)[col] = vr[b];
            }
        }
    }
    for (int pj = t_lo + lane; pj < t_hi; pj += 32) {
        const int ph = __ldg(bt_row + pj / B);
        const bool ok = (unsigned)ph < (unsigned)p.num_blocks;
        if (!ok) set_error(p.err, PKV_DEVERR_BLOCK_ID);
        if (p.slot_out && kvh == 0)
            p.slot_out[(size_t)s * NQ + pj - (ctx - NQ)] = ok ? (int64_t)ph * B + (pj % B) : -1;
    }
}

template <typename T, int D>
__device__ __forceinline__ void append_rows_into_chunk(const DecodeParams& p, unsigned char* Ks,
                                                    unsigned char* Vs, int s, int kvh, int ctx,
                                                    int t_c, int lane) {
    using Geo = MmaGeometry<D>;
    constexpr int VPR = D * 2 / 16;
    constexpr int RPP = 32 / VPR;
    const int NQ = p.num_queries, Hkv = p.num_kv_heads;
    const int sub = lane / VPR, col = lane % VPR;
    const int first = max(ctx - NQ, t_c), last = min(ctx, t_c + CHUNK_TOKENS);
    const uint32_t ks = smem_addr(Ks), vs = smem_addr(Vs);
    for (int pj = first + sub; pj < last; pj += RPP) {
        const size_t src = (((size_t)s * NQ + pj - (ctx - NQ)) * Hkv + kvh) * D + col * 8;
        const uint32_t o16 = (col / 8) * Geo::BOX_BYTES + swz(pj - t_c, col & 7);
        cp_async16(ks + o16, static_cast<const T*>(p.k_new) + src);
        cp_async16(vs + o16, static_cast<const T*>(p.v_new) + src);
    }
    cp_async_wait_all();
    __syncwarp();
}

// One staged 16-token chunk (K rows at ks_s, V rows at vs_s, 128-byte swizzled boxes)
// into the running state of the 8 columns of the N tile held by this lane (columns
// 2 q4 and 2 q4 + 1; the o fragments cover tokens g4 and g4 + 8 of each m16 tile):
//   scores^T = K . Q^T on D/16 MMAs; token t of the chunk counts for column h when
//   t < valid and chunk0 + t < lim[h] (else its score is -inf); online softmax per
//   column in base 2; O^T += V^T . P^T with P as a 16-bit high part plus remainder.
// V rows >= valid must hold zeros.  A column whose tokens are all masked is left exactly
// as it was (alpha = 1, p = 0).
template <typename T, int D>
__device__ __forceinline__ void mma_chunk_update(uint32_t ks_s, uint32_t vs_s,
                                                 const uint32_t (&qb)[D / 16][2], int chunk0,
                                                 int valid, const int (&lim)[2], float scale_log2,
                                                 float (&m)[2], float (&l)[2],
                                                 float (&o)[D / 16][4], int lane) {
    using Geo = MmaGeometry<D>;
    constexpr int KS = Geo::KSTEPS;
    const int g4 = lane >> 2, q4 = lane & 3;
    // ldmatrix row addresses: matrix mi = lane / 8, row lane % 8
    const int mi = lane >> 3, mr = lane & 7;
    // P^T fragment sources: tokens 2 q4 + e come from lane 8 q4 + 4 e + lane / 8
    const int src0 = 8 * q4 + (lane >> 3), src1 = src0 + 4;
    const uint32_t sel = ((lane >> 2) & 1) ? 0x7632u : 0x5410u;
    // scores^T = K . Q^T
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int col = 2 * ks + (mi >> 1);            // 16-byte column of dims
        const int r = ((mi & 1) << 3) + mr;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks_s + (col / 8) * Geo::BOX_BYTES + swz(r, col & 7), a0, a1, a2, a3);
        Mma<T>::run(sc, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
    }
    // online softmax per head column (tokens g4 and g4 + 8 of this lane)
    float pr[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int tok = g4 + ((j >> 1) << 3);
        pr[j] = (tok < valid && chunk0 + tok < lim[j & 1]) ? sc[j] * scale_log2 : -INFINITY;
    }
    float alpha[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float bm = fmaxf(pr[h], pr[h + 2]);
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) bm = fmaxf(bm, __shfl_xor_sync(FULL_MASK, bm, o_));
        const float mn = fmaxf(m[h], bm);
        const float mref = mn == -INFINITY ? 0.f : mn;   // column fully masked so far
        alpha[h] = fast_exp2(m[h] - mref);
        m[h] = mn;
        pr[h] = fast_exp2(pr[h] - mref);
        pr[h + 2] = fast_exp2(pr[h + 2] - mref);
        l[h] = l[h] * alpha[h] + pr[h] + pr[h + 2];
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= alpha[0]; o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0]; o[mt][3] *= alpha[1];
    }
    // P^T as B fragments, high part and remainder
    float rem[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) rem[j] = pr[j] - Mma<T>::round_trip(pr[j]);
    const uint32_t lo_hi = Mma<T>::pack(pr[0], pr[1]), hi_hi = Mma<T>::pack(pr[2], pr[3]);
    const uint32_t lo_lo = Mma<T>::pack(rem[0], rem[1]), hi_lo = Mma<T>::pack(rem[2], rem[3]);
    const uint32_t bh0 = __byte_perm(__shfl_sync(FULL_MASK, lo_hi, src0),
                                     __shfl_sync(FULL_MASK, lo_hi, src1), sel);
    const uint32_t bh1 = __byte_perm(__shfl_sync(FULL_MASK, hi_hi, src0),
                                     __shfl_sync(FULL_MASK, hi_hi, src1), sel);
    const uint32_t bl0 = __byte_perm(__shfl_sync(FULL_MASK, lo_lo, src0),
                                     __shfl_sync(FULL_MASK, lo_lo, src1), sel);
    const uint32_t bl1 = __byte_perm(__shfl_sync(FULL_MASK, hi_lo, src0),
                                     __shfl_sync(FULL_MASK, hi_lo, src1), sel);
    // O^T += V^T . P^T
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        const int col = 2 * mt + (mi & 1);
        const int r = ((mi >> 1) << 3) + mr;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vs_s + (col / 8) * Geo::BOX_BYTES + swz(r, col & 7), a0, a1, a2, a3);
        Mma<T>::run(o[mt], a0, a1, a2, a3, bh0, bh1);
        Mma<T>::run(o[mt], a0, a1, a2, a3, bl0, bl1);
    }
}

template <typename T, int D, int NW, int NS, bool MULTI_APPEND = false>
__global__ void __launch_bounds__(NW * 32)
paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const DecodeParams p) {
    using Geo = MmaGeometry<D>;
    using Smem = MmaSmem<D, NW, NS>;
    constexpr int KS = Geo::KSTEPS;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the 128-byte swizzle repeats every 1024 bytes: align the ring to that
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    if (p.trigger_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int Hkv = p.num_kv_heads;
    // partitions launch last-first, as in decode.cuh
    const int kvh = blockIdx.x % Hkv, qgrp = blockIdx.x / Hkv, s = blockIdx.y;
    const int part = gridDim.z - 1 - blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.block_size, Hq = p.num_q_heads, P = p.partition_size;
    const int G = Hq / Hkv, NQ = p.num_queries;
    const int j0 = qgrp * p.queries_per_cta;
    const int ncols = G * min(p.queries_per_cta, NQ - j0);   // live columns, <= 8
    const int g4 = lane >> 2, q4 = lane & 3;   // mma fragment row / column pair
    // output / workspace row of column n
    auto col_row = [&](int n) -> size_t {
        return ((size_t)s * NQ + j0 + n / G) * Hq + kvh * G + n % G;
    };

    int ctx = p.context_lens[s];
    bool ctx_bad = false;
    {
        const long long cap_table = (long long)p.max_blocks_per_seq * B;
        const long long cap_grid =
            (long long)p.skip_tokens + (long long)(p.max_parts - p.part_offset) * P;
        long long cap = cap_table < cap_grid ? cap_table : cap_grid;
        if (cap > p.max_context_len) cap = p.max_context_len;
        if (ctx < 0 || ctx > cap) {
            if (threadIdx.x == 0 && part == 0 && blockIdx.x == 0) set_error(p.err, PKV_DEVERR_CONTEXT);
            ctx = ctx < 0 ? 0 : int(cap);
            ctx_bad = true;
        }
    }
    const int skip = p.skip_tokens;
    const int n_parts = ctx > skip ? (ctx - skip + P - 1) / P : 0;
    const int tok0 = skip + part * P;
    if (part > 0 && tok0 >= ctx) return;
    const bool direct = p.direct_single && n_parts <= 1;
    // appended tokens (when k_new is set): the last num_queries positions of the context;
    // the slots of those with no position in it are -1 (one CTA of the sequence writes them)
    const int NQn = NQ;
    if (p.slot_out && kvh == 0 && qgrp == 0 && part == 0)
        for (int j = threadIdx.x; j < NQn; j += NW * 32)
            if (ctx == 0 || ctx_bad || ctx - NQn + j < 0) p.slot_out[(size_t)s * NQn + j] = -1;
    if (ctx <= skip) {  // nothing to attend to here: zero output or an empty partial
        if (ctx < skip && threadIdx.x == 0 && blockIdx.x == 0) set_error(p.err, PKV_DEVERR_CONTEXT);
        for (int i = threadIdx.x; i < ncols * D; i += NW * 32) {
            const size_t row = col_row(i / D);
            const int d = i % D;
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
    // the chunk of this warp's i-th step (chunks are dealt round-robin, each warp walks its
    // own alternately from the front and the back), and the owner of chunk c
    auto chunk_of = [&](int i) -> int { return warp + NW * alternating_chunk(i, n_my); };
    auto owner = [&](int c) -> int { return c % NW; };

    // ---- Q^T as mma B fragments: column n = g4 (zero past the live columns), rows = dims
    uint32_t qb[KS][2];
    {
        const int n = g4;
        const T* qrow = static_cast<const T*>(p.q) + col_row(n < ncols ? n : 0) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if (n < ncols) {
                qb[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * q4));
                qb[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * q4));
            } else {
                qb[ks][0] = qb[ks][1] = 0u;
            }
        }
    }

    // ---- per-warp ring
    unsigned char* ring = smem + warp * NS * Geo::STAGE_BYTES;
    const uint32_t ring_s = smem_addr(ring);
    const uint32_t bar0 = smem_addr(smem + Smem::BAR_OFFSET) + warp * NS * 8;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < NS; ++st) mbar_init(bar0 + st * 8, 1);
        mbar_init_fence();
    }
    __syncwarp();

    const int32_t* bt_row = p.block_tables + (size_t)s * p.max_blocks_per_seq;
    const uint64_t policy = l2_evict_first_policy();

    // fused append (see decode.cuh)
    const int p_new = ctx - 1;
    const bool has_new =
        p.k_new != nullptr && NQn == 1 && !ctx_bad && p_new >= tok0 && p_new < tok_end;
    const bool multi_new = MULTI_APPEND && p.k_new != nullptr && NQn > 1 && !ctx_bad;
    const int c_new = has_new ? (p_new - tok0) / CHUNK_TOKENS : -1;
    const bool warp_new = has_new && owner(c_new) == warp;
    constexpr int VPR = D * 2 / 16;  // 16-byte vectors per row
    uint4 k_row = make_uint4(0, 0, 0, 0), v_row = make_uint4(0, 0, 0, 0);
    int phys_new = -1;
    if (warp_new) {
        phys_new = __ldg(bt_row + p_new / B);
        if (lane < VPR) {
            const size_t src = ((size_t)s * Hkv + kvh) * D;
            k_row = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src) + lane);
            v_row = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src) + lane);
        }
    }

    auto table_entry = [&](int i) -> int {
        if (i >= n_my) return -1;
        const int t = tok0 + chunk_of(i) * CHUNK_TOKENS;
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
                const int t = tok0 + chunk_of(i) * CHUNK_TOKENS;
                const int row = (phys * Hkv + kvh) * B + (t % B);
                const uint32_t dst = ring_s + st * Geo::STAGE_BYTES;
                mbar_arrive_expect_tx(bar, Geo::STAGE_BYTES);
                // one copy per pool: every 128-byte column box of the chunk's 16 rows
                tma_load_3d(dst, &tmap_k, 0, row, 0, bar, policy);
                tma_load_3d(dst + Geo::POOL_BYTES, &tmap_v, 0, row, 0, bar, policy);
            } else {
                set_error(p.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive(bar);
            }
        }
    };

    // state: columns 2 q4 and 2 q4 + 1 of the accumulator fragments.  Query j sees
    // positions below ctx - NQ + 1 + j (the causal limit of a multi-token tail).
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    int lim[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int n = 2 * q4 + h;
        lim[h] = n < ncols ? ctx - NQ + 1 + j0 + n / G : ctx;
    }
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    const int n_pro = n_my < NS ? n_my : NS;
    for (int i = 0; i < n_pro; ++i) issue(i);
    if constexpr (MULTI_APPEND) {
        // this warp's new rows into the pool while its first copies fly; the fence and the
        // warp barrier put them ahead of the copies lane 0 issues from here on
        if (multi_new && ctx - NQn < tok_end) {
            const int c_lo = max(ctx - NQn - tok0, 0) / CHUNK_TOKENS;
            for (int i = 0; i < n_my; ++i) {
                const int c = chunk_of(i);
                if (c < c_lo) continue;
                const int t_c = tok0 + c * CHUNK_TOKENS;
                append_rows_to_pool<T, D>(p, bt_row, s, kvh, ctx, max(ctx - NQn, t_c),
                                          min(tok_end, t_c + CHUNK_TOKENS), lane);
            }
            fence_proxy_async_global();
            __syncwarp();
        }
    }

    for (int i = 0; i < n_my; ++i) {
        const int st = i % NS;
        if (!mbar_wait(bar0 + st * 8, (i / NS) & 1)) {
            if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
            for (int j = i + 1; j < n_my && j < i + NS; ++j) mbar_wait(bar0 + (j % NS) * 8, (j / NS) & 1);
            break;
        }
        const int c = chunk_of(i);
        const int valid = min(CHUNK_TOKENS, tok_end - (tok0 + c * CHUNK_TOKENS));
        unsigned char* Ks = ring + st * Geo::STAGE_BYTES;
        unsigned char* Vs = Ks + Geo::POOL_BYTES;
        // ordinary stores into this stage below (spliced rows, zeroed rows) must be ordered
        // before the tensor copy that refills it
        bool dirty = false;
        if (warp_new && c == c_new) {
            dirty = true;
            const bool ok = (unsigned)phys_new < (unsigned)p.num_blocks;
            if (ok && lane < VPR) {
                const int r = (p_new - tok0) & (CHUNK_TOKENS - 1);
                const uint32_t o16 = (lane / 8) * Geo::BOX_BYTES + swz(r, lane & 7);
                *reinterpret_cast<uint4*>(Ks + o16) = k_row;
                *reinterpret_cast<uint4*>(Vs + o16) = v_row;
                const size_t off = (((size_t)phys_new * Hkv + kvh) * B + (p_new % B)) * D;
                reinterpret_cast<uint4*>(const_cast<T*>(static_cast<const T*>(p.k_pool)) + off)[lane] = k_row;
                reinterpret_cast<uint4*>(const_cast<T*>(static_cast<const T*>(p.v_pool)) + off)[lane] = v_row;
            }
            if (p.slot_out && kvh == 0 && lane == 0)
                p.slot_out[s] = ok ? (int64_t)phys_new * B + (p_new % B) : -1;
            __syncwarp();
        }
        if constexpr (MULTI_APPEND) {
            const int t_c = tok0 + c * CHUNK_TOKENS;
            if (multi_new && i < NS && t_c + CHUNK_TOKENS > ctx - NQn) {
                append_rows_into_chunk<T, D>(p, Ks, Vs, s, kvh, ctx, t_c, lane);
                dirty = true;
            }
        }
        if (!((bad_stages >> st) & 1)) {
            if (valid < CHUNK_TOKENS) {
                dirty = true;
                // rows past the context may hold anything: zero them so 0 * row stays 0
                for (int v = lane; v < (CHUNK_TOKENS - valid) * VPR; v += 32) {
                    const int r = valid + v / VPR, col = v % VPR;
                    *reinterpret_cast<uint4*>(Vs + (col / 8) * Geo::BOX_BYTES + swz(r, col & 7)) =
                        make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            mma_chunk_update<T, D>(smem_addr(Ks), smem_addr(Vs), qb, tok0 + c * CHUNK_TOKENS, valid,
                                   lim, p.scale_log2, m, l, o, lane);
        }
        if (dirty) fence_proxy_async_shared();
        __syncwarp();
        if (i + NS < n_my) issue(i + NS);
    }

    // ---- warp totals: sum l over the 8 lanes of each head column
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) l[h] += __shfl_xor_sync(FULL_MASK, l[h], o_);

    // ---- combine the warps in shared memory
    __syncthreads();
    float* red = reinterpret_cast<float*>(smem);  // [NW][8][D + 2]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int n = 2 * q4 + h;
        if (n < ncols) {
            float* r = red + (warp * 8 + n) * (D + 2);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                r[mt * 16 + g4] = o[mt][h];
                r[mt * 16 + g4 + 8] = o[mt][h + 2];
            }
            if (g4 == 0) { r[D] = m[h]; r[D + 1] = l[h]; }
        }
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < ncols * D; idx += NW * 32) {
        const int n = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, red[(w * 8 + n) * (D + 2) + D]);
        const float Mref = M == -INFINITY ? 0.f : M;
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* r = red + (w * 8 + n) * (D + 2);
            const float f = fast_exp2(r[D] - Mref);
            L = fmaf(r[D + 1], f, L);
            O = fmaf(r[d], f, O);
        }
        const size_t row = col_row(n);
        if (direct) {
            store_out(p.out, p.out_dtype, row * D + d, L > 0.f ? O / L : 0.f);
        } else {
            const size_t rr = row * p.max_parts + part + p.part_offset;
            p.ws_o[rr * D + d] = O;
            if (d == 0) {
                p.ws_m[rr] = M * 0.69314718055994530942f;
                p.ws_l[rr] = L;
            }
        }
    }
}

// ------------------------------------------------------------------ host side

// cuTensorMapEncodeTiled, looked up once through the runtime (no libcuda link).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// The pool seen as a 2-D tensor [num_blocks * Hkv * B rows][D], boxes of
// [16 rows][64 elements] with the 128-byte swizzle (the shared-prefix pass in
// prefix.cuh copies its chunks through this map).
template <typename T>
inline bool encode_pool_map(CUtensorMap* map, const void* base, long long rows, int D) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * sizeof(T)};
    const cuuint32_t box[2] = {64, (cuuint32_t)CHUNK_TOKENS};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, Mma<T>::TMA_TYPE, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// The pool seen as a 3-D tensor for the decode kernel: x = 64 elements of a 128-byte
// column box, y = rows (N * Hkv * B), z = which 128-byte column of the row (D / 64 of
// them); strides D * 2 bytes (y) and 128 bytes (z).  A box of {64, 16, D / 64} is a whole
// 16-token chunk of one pool, landing as D / 64 consecutive [16][128-byte] boxes with the
// 128-byte swizzle: one copy per pool and chunk instead of D / 64.
template <typename T>
inline bool encode_pool_map_3d(CUtensorMap* map, const void* base, long long rows, int D) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)D * sizeof(T), 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)CHUNK_TOKENS, (cuuint32_t)(D / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, Mma<T>::TMA_TYPE, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int D> struct MmaShape { static constexpr int NW = 4, NS = (64 * 1024) / (4 * MmaGeometry<D>::STAGE_BYTES); };

template <typename T, int D, bool MULTI_APPEND>
cudaError_t launch_decode_mma_tdv(const DecodeParams& p, cudaStream_t stream) {
    constexpr int NW = MmaShape<D>::NW, NS = MmaShape<D>::NS;
    constexpr int SMEM = MmaSmem<D, NW, NS>::BYTES;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    if (rows >= (1ll << 31)) return cudaErrorNotSupported;  // TMA row coordinates are int32
    if (!encode_pool_map_3d<T>(&tk, p.k_pool, rows, D) ||
        !encode_pool_map_3d<T>(&tv, p.v_pool, rows, D))
        return cudaErrorNotSupported;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kernel = paged_decode_mma_kernel<T, D, NW, NS, MULTI_APPEND>;
    static std::atomic<bool> configured[64];  // per device; setting it twice is harmless
    if (dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    const int groups = (p.num_queries + p.queries_per_cta - 1) / p.queries_per_cta;
    dim3 grid(p.num_kv_heads * groups, p.num_seqs, p.max_parts - p.part_offset);
    kernel<<<grid, NW * 32, SMEM, stream>>>(tk, tv, p);
    return cudaGetLastError();
}

// the kernel variant appending several tokens per sequence only where it is asked for
template <typename T, int D>
cudaError_t launch_decode_mma_td(const DecodeParams& p, cudaStream_t stream) {
    if (p.k_new != nullptr && p.num_queries > 1)
        return launch_decode_mma_tdv<T, D, true>(p, stream);
    return launch_decode_mma_tdv<T, D, false>(p, stream);
}

template <typename T>
cudaError_t launch_decode_mma_impl(const DecodeParams& p, int head_dim, int group,
                                   cudaStream_t stream) {
    if (group < 1 || group > 8 || p.queries_per_cta * group > 8) return cudaErrorInvalidValue;
    if (head_dim == 64) return launch_decode_mma_td<T, 64>(p, stream);
    if (head_dim == 128) return launch_decode_mma_td<T, 128>(p, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
