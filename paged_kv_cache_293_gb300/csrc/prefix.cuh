// prefix.cuh -- attention of every sequence's queries over a prefix all of them share,
// on the fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// "Serving models with vLLM", section "How it works: PagedAttention": requests with
// the same prefix (system prompt, documents) point at the same physical blocks;
// "What Is vLLM", section "How does PagedAttention work?": prefix sharing.  When
// every sequence of a batch starts with the same prefix_len tokens in the same
// physical blocks, their attention over those tokens is one dense contraction per
// kv head: (num_seqs * G) query rows against prefix_len keys.  The per-row result
// (reference max, sum of weights, weighted sum of V) of each split of the prefix
// goes to its own workspace slot, before the partitions of each sequence's own
// suffix, and the log-sum-exp merge combines them -- the same arithmetic as
// attending to the whole context at once, regrouped.
//
// CTA = 128 query rows of one kv head (the MMA's M) x one split of the prefix,
// taken in chunks of 64 tokens.  Eleven warps with fixed roles:
//   warps 8 and 10: TMA tensor copies of each chunk's K pages (warp 8) and V pages
//     (warp 10) -- 128-byte swizzle, 16-token boxes -- into a two-stage K ring and a
//     two-stage V ring (two CTAs per SM); a K stage is released as soon as its
//     Q.K^T is done, a V stage after its P.V;
//   warp 9, one lane: issues the MMAs --
//     S_j [128 rows x 64 tokens] = Q . K_j^T   (tensor memory, two buffers)
//     O   [128 rows x D]        += P_j . V_j   (tensor memory; P_j is written over
//                                               S_j as a 16-bit high part and its
//                                               remainder and read from there)
//     and learns of their completion through tcgen05.commit on mbarriers;
//   warps 0-7: the softmax.  Warp w reads lanes 32 (w % 4) .. + 31 (its rows) and
//     half w / 4 of each S tile's columns; the two warps of a row quarter agree on
//     the row's chunk maximum (and at the end its sum) through shared memory; at the
//     end they write O as whole rows, staged through the then idle Q tile and rings.
// The running maximum is kept lazily: P = 2^(s - m_ref) with the reference m_ref
// raised only when a chunk's maximum exceeds it by more than 8 (base-2 units), so
// the O accumulator in tensor memory is rescaled (read, scaled and written back
// by the row's own threads) only on those chunks.  Every term of a row uses the
// same m_ref, so the result is the same function of the inputs; P stays below 2^8.
// Every wait is bounded; a CTA that gives up sets PKV_DEVERR_TIMEOUT and still
// returns its tensor memory.
#pragma once

#include <type_traits>

#include "decode_mma.cuh"
#include "umma.cuh"

namespace pkv {

constexpr int PREFIX_K_STAGES = 2;
constexpr int PREFIX_V_STAGES = 2;
constexpr int PREFIX_CTAS_PER_SM = 2;
constexpr int PREFIX_ROWS = 128;     // query rows per CTA
constexpr int PREFIX_CHUNK = 64;     // prefix tokens per S tile
constexpr int PREFIX_THREADS = 352;  // 8 softmax warps, K copies, MMA issue, V copies
constexpr float PREFIX_RESCALE_LOG2 = 8.f;

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
    int32_t tokens_per_split;  // a multiple of 64; grid.z splits the prefix, split z -> slot z
    float* ws_m;
    float* ws_l;
    float* ws_o;
    unsigned int* err;
};

template <int D>
struct PrefixSmem {
    static constexpr int BOXES = D / 64;                        // 128-byte columns of a row
    static constexpr int Q_BOX = PREFIX_ROWS * 128;             // one 128-byte column of Q
    static constexpr int KV_BOX = PREFIX_CHUNK * 128;           // one of a chunk of K or V
    static constexpr int STAGE_BYTES = BOXES * KV_BOX;          // a chunk of one pool
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + BOXES * Q_BOX;
    static constexpr int V_OFF = K_OFF + PREFIX_K_STAGES * STAGE_BYTES;
    static constexpr int RED_OFF = V_OFF + PREFIX_V_STAGES * STAGE_BYTES;  // float [2][2][128]
    static constexpr int BAR_OFF = RED_OFF + 4 * PREFIX_ROWS * 4;
    static constexpr int NBARS = 2 * PREFIX_K_STAGES + 2 * PREFIX_V_STAGES + 6 + 8 + 2;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
    static constexpr int BYTES = TMEM_SLOT_OFF + 16 + 1024;             // + alignment slack
    // tensor memory: S_j / P_j in columns 64 (j % 2) .. + 63, O from column 128
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t O_COL = 2 * PREFIX_CHUNK;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(BYTES <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <typename T, int D>
__global__ void __launch_bounds__(PREFIX_THREADS, PREFIX_CTAS_PER_SM)
prefix_attention_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v, const PrefixParams p) {
    using L = PrefixSmem<D>;
    constexpr int NK = PREFIX_K_STAGES, NV = PREFIX_V_STAGES, KS = D / 16;
    constexpr int K_WARP = 8, MMA_WARP = 9, V_WARP = 10;
    constexpr uint32_t FMT = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t IDESC_S = umma::idesc_f16(FMT, false, PREFIX_ROWS, PREFIX_CHUNK);
    constexpr uint32_t IDESC_O = umma::idesc_f16(FMT, true, PREFIX_ROWS, D);

    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t q_s = sbase + L::Q_OFF, k_ring = sbase + L::K_OFF, v_ring = sbase + L::V_OFF;
    float* red = reinterpret_cast<float*>(smem + L::RED_OFF);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    // barriers: K / V chunk landed and stage free; S tile ready; S/P buffer free (the
    // P.V that read it is done); P tile written; row-quarter exchange; all MMAs done;
    // Q tile stored
    auto k_full = [&](int st) { return bar0 + 8 * st; };
    auto k_empty = [&](int st) { return bar0 + 8 * (NK + st); };
    auto v_full = [&](int st) { return bar0 + 8 * (2 * NK + st); };
    auto v_empty = [&](int st) { return bar0 + 8 * (2 * NK + NV + st); };
    constexpr int NB = 2 * NK + 2 * NV;
    auto s_full = [&](int b) { return bar0 + 8 * (NB + b); };
    auto s_free = [&](int b) { return bar0 + 8 * (NB + 2 + b); };
    auto p_full = [&](int b) { return bar0 + 8 * (NB + 4 + b); };
    auto xbar = [&](int qtr, int b) { return bar0 + 8 * (NB + 6 + 2 * qtr + b); };
    const uint32_t o_done = bar0 + 8 * (NB + 14);
    const uint32_t q_full = bar0 + 8 * (NB + 15);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

    const int kvh = blockIdx.x, tile = blockIdx.y, split = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.num_q_heads / p.num_kv_heads;
    const int B = p.block_size;
    const int rows = p.num_seqs * G;
    const int t_begin = split * p.tokens_per_split;
    const int t_end = min(p.prefix_len, t_begin + p.tokens_per_split);
    const int n_chunks = t_end > t_begin ? (t_end - t_begin + PREFIX_CHUNK - 1) / PREFIX_CHUNK : 0;

    if (threadIdx.x == 0) {
        for (int st = 0; st < NK; ++st) {
            mbar_init(k_full(st), 1);
            mbar_init(k_empty(st), 1);
        }
        for (int st = 0; st < NV; ++st) {
            mbar_init(v_full(st), 1);
            mbar_init(v_empty(st), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(s_free(b), 1);
            mbar_init(p_full(b), 8);
            for (int qtr = 0; qtr < 4; ++qtr) mbar_init(xbar(qtr, b), 2);
        }
        mbar_init(o_done, 1);
        mbar_init(q_full, 8);
        mbar_init_fence();
    }
    if (warp == MMA_WARP) umma::alloc(smem_addr(tmem_slot), L::TMEM_COLS);

    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == K_WARP || warp == V_WARP) {
        // ---- copies of one pool's pages, each chunk once its stage has been released.
        // The whole warp runs the loop: its lanes fetch the block ids of 32 boxes (8
        // chunks) at a time, one window ahead, and lane 0 issues the copies.
        const bool is_k = warp == K_WARP;
        const int NST = is_k ? NK : NV;
        const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
        const uint32_t ring = is_k ? k_ring : v_ring;
        const uint64_t policy = l2_evict_last_policy();  // every tile of the head re-reads them
        const int box0 = t_begin / CHUNK_TOKENS, nbox = (t_end - t_begin) / CHUNK_TOKENS;
        auto window_ids = [&](int win) -> int {
            const int b = win * 32 + lane;
            return b < nbox ? __ldg(p.block_tables + (box0 + b) * CHUNK_TOKENS / B) : -1;
        };
        int ids = window_ids(0), ids_next = window_ids(1);
        int issued = 0;
        for (int j = 0; j < n_chunks; ++j) {
            const int st = j % NST;
            if (j >= NST) {
                bool free_ = true;
                if (lane == 0) free_ = mbar_wait(is_k ? k_empty(st) : v_empty(st), ((j / NST) - 1) & 1);
                if (!__shfl_sync(FULL_MASK, free_, 0)) {
                    if (lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
                    break;
                }
            }
            if (j > 0 && j % 8 == 0) {
                ids = ids_next;
                ids_next = window_ids(j / 8 + 1);
            }
            const int t0 = t_begin + j * PREFIX_CHUNK;
            const int boxes = min(PREFIX_CHUNK, t_end - t0) / CHUNK_TOKENS;
            int row[PREFIX_CHUNK / CHUNK_TOKENS];
            int good = 0;
#pragma unroll
            for (int b = 0; b < PREFIX_CHUNK / CHUNK_TOKENS; ++b) {
                const int phys = __shfl_sync(FULL_MASK, ids, (j % 8) * 4 + b);
                row[b] = -1;
                if (b >= boxes) continue;
                if ((unsigned)phys >= (unsigned)p.num_blocks) {
                    if (is_k && lane == 0) set_error(p.err, PKV_DEVERR_BLOCK_ID);  // not loaded
                } else {
                    row[b] = (phys * p.num_kv_heads + kvh) * B + (t0 + b * CHUNK_TOKENS) % B;
                    ++good;
                }
            }
            if (lane == 0) {
                const uint32_t bar = is_k ? k_full(st) : v_full(st);
                mbar_arrive_expect_tx(bar, (uint32_t)good * L::BOXES * CHUNK_TOKENS * 128);
                const uint32_t dst = ring + st * L::STAGE_BYTES;
#pragma unroll
                for (int b = 0; b < PREFIX_CHUNK / CHUNK_TOKENS; ++b) {
                    if (row[b] < 0) continue;
#pragma unroll
                    for (int x = 0; x < L::BOXES; ++x)
                        tma_load_2d(dst + x * L::KV_BOX + b * CHUNK_TOKENS * 128, map, x * 64,
                                    row[b], bar, policy);
                }
            }
            issued = j + 1;
        }
        // the CTA must not end with copies still landing in its shared memory
        if (lane == 0)
            for (int j = issued > NST ? issued - NST : 0; j < issued; ++j)
                mbar_wait(is_k ? k_full(j % NST) : v_full(j % NST), (j / NST) & 1);
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ---- MMA issue: S_j as soon as K_j is in, then the P.V of chunk j - 1
        if (lane == 0) {
            auto issue_pv = [&](int i) -> bool {
                if (!mbar_wait(v_full(i % NV), (i / NV) & 1) ||
                    !mbar_wait(p_full(i & 1), (i >> 1) & 1))
                    return false;
                umma::fence_after_sync();
                const int vt = min(PREFIX_CHUNK, t_end - (t_begin + i * PREFIX_CHUNK));
                const uint32_t v_s = v_ring + (i % NV) * L::STAGE_BYTES;
                const uint32_t p_t = tmem + (i & 1) * PREFIX_CHUNK;
                for (int kk = 0; kk < vt / 16; ++kk) {
                    // V is N-major: 64-dim blocks KV_BOX apart, 8-token groups 1024 apart.
                    // P's 16 tokens of step kk: half kk / 2, its columns 8 (kk % 2) .. + 7
                    // (high part) and 16 further (remainder)
                    const uint64_t bv = umma::sw128_desc(v_s + kk * 16 * 128, L::KV_BOX, 1024);
                    const uint32_t a = p_t + (kk >> 1) * 32 + (kk & 1) * 8;
                    umma::mma_f16_tmem_a(tmem + L::O_COL, a, bv, IDESC_O,
                                         (i > 0 || kk > 0) ? 1u : 0u);
                    umma::mma_f16_tmem_a(tmem + L::O_COL, a + 16, bv, IDESC_O, 1u);
                }
                umma::commit(s_free(i & 1));
                umma::commit(v_empty(i % NV));
                return true;
            };
            bool ok = mbar_wait(q_full, 0);
            for (int j = 0; j < n_chunks && ok; ++j) {
                const int st = j % NK;
                ok = mbar_wait(k_full(st), (j / NK) & 1) &&
                     (j < 2 || mbar_wait(s_free(j & 1), ((j - 2) >> 1) & 1));
                if (!ok) break;
                umma::fence_after_sync();
                const uint32_t k_s = k_ring + st * L::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint64_t a =
                        umma::sw128_desc(q_s + (kk >> 2) * L::Q_BOX + (kk & 3) * 32, 16, 1024);
                    const uint64_t b =
                        umma::sw128_desc(k_s + (kk >> 2) * L::KV_BOX + (kk & 3) * 32, 16, 1024);
                    umma::mma_f16(tmem + (j & 1) * PREFIX_CHUNK, a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
                umma::commit(s_full(j & 1));
                umma::commit(k_empty(st));
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok && n_chunks > 0) ok = issue_pv(n_chunks - 1);
            if (!ok) set_error(p.err, PKV_DEVERR_TIMEOUT);
            umma::commit(o_done);  // arrives once every MMA above has completed
            if (!mbar_wait(o_done, 0)) set_error(p.err, PKV_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ---- softmax warps.  First the Q tile, as the first MMA's A operand (rows past
        // the batch are zero): warp w copies rows 16 w .. 16 w + 15, whole rows per load.
        const int qtr = warp & 3, h = warp >> 2;
        const int i = qtr * 32 + lane;
        auto q_index = [&](int r) -> long long {  // tile row -> q row, -1 past the batch
            const int gr = tile * PREFIX_ROWS + r;
            return gr < rows ? (long long)(gr / G) * p.num_q_heads + (long long)kvh * G + gr % G
                             : -1;
        };
        {
            constexpr int CPR = D / 8;                // 16-byte columns per row
            constexpr int RPL = 32 / CPR;             // rows per warp load
            constexpr int LOADS = 16 / RPL;
            const int c = lane % CPR;
            uint4 v[LOADS];
#pragma unroll
            for (int k = 0; k < LOADS; ++k) {
                const long long qr = q_index(warp * 16 + k * RPL + lane / CPR);
                v[k] = qr >= 0 ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                                      qr * D) + c)
                               : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int k = 0; k < LOADS; ++k) {
                const int r = warp * 16 + k * RPL + lane / CPR;
                *reinterpret_cast<uint4*>(smem + L::Q_OFF + (c / 8) * L::Q_BOX + swz(r, c % 8)) = v[k];
            }
            umma::fence_smem_to_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_full);
        }
        // Every sequence must hold sequence 0's prefix blocks: this CTA checks the blocks
        // of its split for the sequences of its tile numbered kvh modulo num_kv_heads.
        {
            const int s_lo = tile * PREFIX_ROWS / G;
            const int s_hi = min(p.num_seqs, (tile * PREFIX_ROWS + PREFIX_ROWS - 1) / G + 1);
            const int j_lo = t_begin / B, nb = (t_end - t_begin) / B;
            const int ns = (s_hi - s_lo - kvh + p.num_kv_heads - 1) / p.num_kv_heads;
            for (int e = threadIdx.x; e < ns * nb; e += 8 * 32) {
                const int s = s_lo + kvh + (e / nb) * p.num_kv_heads, j = j_lo + e % nb;
                if (__ldg(p.block_tables + (size_t)s * p.max_blocks_per_seq + j) !=
                    __ldg(p.block_tables + j))
                    set_error(p.err, PKV_DEVERR_PREFIX);
            }
        }
        // ---- softmax: this thread's row i, columns of half h of each S tile
        const uint32_t lane_tmem = tmem + ((uint32_t)(qtr * 32) << 16);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        // the two warps of a row quarter swap one float per row through shared memory
        auto exchange = [&](int j, float v) -> float {
            red[((j & 1) * 2 + h) * PREFIX_ROWS + i] = v;
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar(qtr, j & 1));
            if (!__all_sync(FULL_MASK, mbar_wait(xbar(qtr, j & 1), (j >> 1) & 1))) {
                ok = false;
                return v;
            }
            return red[((j & 1) * 2 + (h ^ 1)) * PREFIX_ROWS + i];
        };
        for (int j = 0; j < n_chunks; ++j) {
            const int vt = min(PREFIX_CHUNK, t_end - (t_begin + j * PREFIX_CHUNK));
            if (!__all_sync(FULL_MASK, mbar_wait(s_full(j & 1), (j >> 1) & 1))) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
            const uint32_t sp = lane_tmem + (j & 1) * PREFIX_CHUNK + h * 32;  // S, then P
            float s[32];
            umma::ld32(sp, s);
            // columns past the chunk's last token hold no key: they take no part
            const int nvalid = vt - h * 32;
            float cm = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                s[k] *= p.scale_log2;
                if (k < nvalid) cm = fmaxf(cm, s[k]);
            }
            cm = fmaxf(cm, exchange(j, cm));
            if (!ok) break;
            const bool need = cm > m_ref + PREFIX_RESCALE_LOG2;
            float alpha = 1.f;
            if (need) {
                alpha = fast_exp2(m_ref - cm);
                m_ref = cm;
                l *= alpha;
            }
            // P over this half's 32 columns of S: 16 columns of high parts, then 16 of
            // remainders, two tokens per column
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
                const float a = k < nvalid ? fast_exp2(s[k] - m_ref) : 0.f;
                const float b = k + 1 < nvalid ? fast_exp2(s[k + 1] - m_ref) : 0.f;
                l += a + b;
                hi[k / 2] = Mma<T>::pack(a, b);
                lo[k / 2] = Mma<T>::pack(a - Mma<T>::round_trip(a), b - Mma<T>::round_trip(b));
            }
            umma::st16(sp, hi);
            umma::st16(sp + 16, lo);
            // rows whose reference rose: scale their O (complete through chunk j - 1)
            if (j >= 1 && __any_sync(FULL_MASK, need)) {
                if (!__all_sync(FULL_MASK, mbar_wait(s_free((j - 1) & 1), ((j - 1) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 2; c += 32) {
                    float o[32];
                    umma::ld32(lane_tmem + L::O_COL + h * (D / 2) + c, o);
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] *= alpha;
                    umma::st32(lane_tmem + L::O_COL + h * (D / 2) + c, o);
                }
            }
            umma::wait_st();
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(j & 1));
        }
        if (ok && n_chunks > 0) {
            ok = __all_sync(FULL_MASK, mbar_wait(o_done, 0));
            if (ok) l += exchange(n_chunks, l);
        }
        // O leaves through shared memory so that each warp then writes whole rows: row r
        // of the staging area holds D floats at a stride of D + 4 (no bank conflicts
        // between the rows of a warp's store).  The area spans the Q tile and the K and V
        // rings, all idle once every MMA is done, and ends before the exchange area, which
        // the other warp of a row quarter may still be reading.
        constexpr int SROW = D + 4;
        static_assert(L::Q_OFF + PREFIX_ROWS * SROW * 4 <= L::RED_OFF, "O staging area");
        float* stage = reinterpret_cast<float*>(smem + L::Q_OFF);
        if (ok && n_chunks > 0) {
            umma::fence_after_sync();
#pragma unroll
            for (int c = 0; c < D / 2; c += 32) {
                float o[32];
                umma::ld32(lane_tmem + L::O_COL + h * (D / 2) + c, o);
#pragma unroll
                for (int k = 0; k < 32; k += 4)
                    *reinterpret_cast<float4*>(stage + i * SROW + h * (D / 2) + c + k) =
                        make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
            }
        }
        // every softmax warp reaches this barrier, whatever happened above
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const bool all_ok = ok && n_chunks > 0;
        if (!ok && lane == 0) set_error(p.err, PKV_DEVERR_TIMEOUT);
        {
            const long long qr = q_index(i);
            const size_t slot = (size_t)(qr < 0 ? 0 : qr) * p.max_parts + split;
            if (qr >= 0 && h == 0 && ok) {
                p.ws_m[slot] = n_chunks > 0 ? m_ref * 0.69314718055994530942f : -INFINITY;
                p.ws_l[slot] = l;
            }
        }
        if (ok) {
            constexpr int F4 = D / 4;  // float4 per row
#pragma unroll 4
            for (int rr = 0; rr < 16; ++rr) {
                const int r = warp * 16 + rr;
                const long long qr = q_index(r);
                if (qr < 0 || lane >= F4) continue;
                const float4 v = all_ok ? *reinterpret_cast<const float4*>(stage + r * SROW + lane * 4)
                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4*>(p.ws_o + ((size_t)qr * p.max_parts + split) * D)[lane] = v;
            }
        }
    }

    // tensor memory goes back only after every warp is done with it
    umma::fence_before_sync();
    __syncthreads();
    if (warp == MMA_WARP) {
        umma::fence_after_sync();
        umma::dealloc(tmem, L::TMEM_COLS);
    }
    // launched early behind the suffix decode (programmatic dependent launch): finish only
    // after it, so that the merge launched behind this grid sees both grids' partials
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <typename T, int D>
cudaError_t launch_prefix_td(const PrefixParams& p, const void* k_pool, const void* v_pool,
                             cudaStream_t stream) {
    constexpr int SMEM = PrefixSmem<D>::BYTES;
    if (p.tokens_per_split <= 0 || p.tokens_per_split % PREFIX_CHUNK != 0)
        return cudaErrorInvalidValue;
    CUtensorMap tk, tv;
    const long long rows = (long long)p.num_blocks * p.num_kv_heads * p.block_size;
    if (rows >= (1ll << 31)) return cudaErrorNotSupported;
    if (!encode_pool_map<T>(&tk, k_pool, rows, D) || !encode_pool_map<T>(&tv, v_pool, rows, D))
        return cudaErrorNotSupported;
    const int G = p.num_q_heads / p.num_kv_heads;
    const long long tiles = ((long long)p.num_seqs * G + PREFIX_ROWS - 1) / PREFIX_ROWS;
    if (tiles > 65535) return cudaErrorNotSupported;
    const int splits = (p.prefix_len + p.tokens_per_split - 1) / p.tokens_per_split;
    dim3 grid(p.num_kv_heads, (unsigned)tiles, splits);
    auto kernel = prefix_attention_kernel<T, D>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> configured[64];  // per device; setting it twice is harmless
    if (dev < 64 && !configured[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured[dev].store(true, std::memory_order_release);
    }
    // programmatic dependent launch: the CTAs may start while the grid before this one in
    // the stream (the suffix decode, which triggers at its start) still runs; nothing here
    // reads what that grid writes
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(PREFIX_THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tk, tv, p);
}

template <typename T>
cudaError_t launch_prefix_impl(const PrefixParams& p, const void* k_pool, const void* v_pool,
                               int head_dim, cudaStream_t stream) {
    if (head_dim == 64) return launch_prefix_td<T, 64>(p, k_pool, v_pool, stream);
    if (head_dim == 128) return launch_prefix_td<T, 128>(p, k_pool, v_pool, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
