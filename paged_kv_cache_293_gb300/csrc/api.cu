// api.cu -- the C ABI of libpagedkv.so (declared in include/pagedkv.h).
//
// Host-side argument checks, the choice of partition size, workspace layout,
// dispatch to the typed kernels, and the device error word.  Nothing here
// allocates device memory or synchronises, except pkv_get_device_error.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pkv_common.cuh"
#include "prefix.cuh"

namespace {

// One word per device: kernels OR error bits into it instead of trapping.
__device__ unsigned int g_error_word;

constexpr int MAX_DEVICES = 64;
std::atomic<unsigned int*> g_error_ptr[MAX_DEVICES];  // looked up once per device

pkv_status error_word(unsigned int** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PKV_ERR_CUDA;
    unsigned int* w = g_error_ptr[dev].load(std::memory_order_acquire);
    if (!w) {  // callers racing here all find the same address
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_error_word) != cudaSuccess) return PKV_ERR_CUDA;
        w = static_cast<unsigned int*>(ptr);
        g_error_ptr[dev].store(w, std::memory_order_release);
    }
    *out = w;
    return PKV_OK;
}

std::atomic<int> g_engine{PKV_ENGINE_AUTO};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pkv_status check_pool(const pkv_pool* pool) {
    if (!pool || !pool->k || !pool->v) return PKV_ERR_INVALID;
    if (!aligned16(pool->k) || !aligned16(pool->v)) return PKV_ERR_INVALID;
    if (pool->num_blocks <= 0 || pool->block_size <= 0 || pool->num_kv_heads <= 0 ||
        pool->head_dim <= 0)
        return PKV_ERR_INVALID;
    if (pool->dtype != PKV_F32 && pool->dtype != PKV_F16 && pool->dtype != PKV_BF16)
        return PKV_ERR_INVALID;
    if (pool->block_size != 16 && pool->block_size != 32) return PKV_ERR_UNSUPPORTED;
    if (pool->head_dim != 64 && pool->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

int32_t ceil_div(int64_t a, int64_t b) { return int32_t((a + b - 1) / b); }

struct WsLayout {
    size_t l_off, o_off, bytes;
};

WsLayout ws_layout(int32_t S, int32_t Hq, int32_t D, int32_t parts) {
    const size_t rows = (size_t)S * Hq * parts;
    const size_t a = (rows * 4 + 15) & ~size_t(15);
    return WsLayout{a, 2 * a, 2 * a + rows * D * 4};
}

// One pass while the longest context is at most 3072 tokens; beyond that,
// 1024-token partitions (a multiple of 16 and 32), or 2048 with several query rows
// per sequence, whose partial results and merge cost num_queries times as much.
// Measured on the batches here: one pass was best for the LLaMA-7B (max 2048) and
// shared-prefix GQA (max 2560) batches, 1024-token partitions for LLaMA-13B (max
// 4096, a long lognormal tail) and the 32k-128k contexts; on the LLaMA-13B batch
// with 4 / 8 new tokens per sequence 2048-token partitions took 346.0 / 362.9 us
// against 348.6 / 371.8 us with 1024.
int32_t auto_partition(const pkv_pool* pool, int32_t max_context_len, int32_t num_queries = 1) {
    const int32_t B = pool->block_size;
    const int32_t one_pass_limit = 3072, split = num_queries > 1 ? 2048 : 1024;
    if (max_context_len <= one_pass_limit)
        return max_context_len <= 0 ? B : ceil_div(max_context_len, B) * B;
    return split;
}

struct DecodeArgs {
    const pkv_pool* pool;
    const void* q;
    int32_t S, Hq;
    const int32_t* bt;
    int32_t M;
    const int32_t* ctx;
    int32_t max_ctx;
    float scale;
    int32_t P;  // 0 = auto
    int32_t NQ = 1;  // query rows per sequence
};

pkv_status check_decode(const DecodeArgs& a) {
    pkv_status st = check_pool(a.pool);
    if (st != PKV_OK) return st;
    if (a.S < 0 || a.Hq <= 0 || a.M <= 0 || a.max_ctx < 0) return PKV_ERR_INVALID;
    if (a.Hq % a.pool->num_kv_heads != 0) return PKV_ERR_INVALID;
    if (!std::isfinite(a.scale)) return PKV_ERR_INVALID;
    if (a.P < 0 || (a.P > 0 && a.P % a.pool->block_size != 0)) return PKV_ERR_INVALID;
    if (a.S > 0 && (!a.q || !a.bt || !a.ctx)) return PKV_ERR_INVALID;
    if (a.S > 0 && !aligned16(a.q)) return PKV_ERR_INVALID;
    const int32_t G = a.Hq / a.pool->num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PKV_ERR_UNSUPPORTED;
    if (a.S > 65535) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

cudaError_t launch_decode_typed(const pkv::DecodeParams& p, int32_t dtype, int D, int G,
                                cudaStream_t stream) {
    switch (dtype) {
        case PKV_F32: return pkv::launch_decode<float>(p, D, G, stream);
        case PKV_F16: return pkv::launch_decode<__half>(p, D, G, stream);
        default: return pkv::launch_decode<__nv_bfloat16>(p, D, G, stream);
    }
}

struct AppendArgs {
    const void* k_new;
    const void* v_new;
    int64_t* slot_out;
};

// Shared body of decode (direct = 1) and the partition step (direct = 0);
// `append` (may be null) turns on the fused write of each sequence's new token.
pkv_status run_decode(const DecodeArgs& a, void* out, int32_t out_dtype, int direct,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream,
                      const AppendArgs* append = nullptr) {
    const pkv_pool* pool = a.pool;
    const int32_t P = a.P > 0 ? a.P : auto_partition(pool, a.max_ctx, a.NQ);
    const int32_t parts = a.max_ctx > 0 ? ceil_div(a.max_ctx, P) : 1;
    if (parts > 65535) return PKV_ERR_UNSUPPORTED;
    const bool need_ws = !direct || parts > 1;
    const WsLayout lay = ws_layout(a.S * a.NQ, a.Hq, pool->head_dim, parts);
    if (need_ws && (!workspace || !aligned16(workspace) || workspace_bytes < lay.bytes))
        return PKV_ERR_WORKSPACE;
    if (a.S == 0) return PKV_OK;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;

    pkv::DecodeParams p{};
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.num_blocks = pool->num_blocks;
    p.block_size = pool->block_size;
    p.num_kv_heads = pool->num_kv_heads;
    p.q = a.q;
    p.num_seqs = a.S;
    p.num_q_heads = a.Hq;
    p.block_tables = a.bt;
    p.max_blocks_per_seq = a.M;
    p.context_lens = a.ctx;
    p.max_context_len = a.max_ctx;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.partition_size = P;
    p.max_parts = parts;
    p.out = out;
    p.out_dtype = out_dtype;
    p.direct_single = direct;
    const int G = a.Hq / pool->num_kv_heads;
    p.num_queries = a.NQ;
    p.queries_per_cta = 8 / G < a.NQ ? 8 / G : a.NQ;
    if (need_ws) {
        char* ws = static_cast<char*>(workspace);
        p.ws_m = reinterpret_cast<float*>(ws);
        p.ws_l = reinterpret_cast<float*>(ws + lay.l_off);
        p.ws_o = reinterpret_cast<float*>(ws + lay.o_off);
    }
    if (append) {
        p.k_new = append->k_new;
        p.v_new = append->v_new;
        p.slot_out = append->slot_out;
    }
    p.err = err;
    if (a.NQ > 1) {
        // several query rows per sequence: the tensor-core kernel only
        const cudaError_t e =
            pool->dtype == PKV_F16
                ? pkv::launch_decode_mma<__half>(p, pool->head_dim, G, stream)
                : pkv::launch_decode_mma<__nv_bfloat16>(p, pool->head_dim, G, stream);
        if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return PKV_ERR_CUDA;
    } else if (launch_decode_typed(p, pool->dtype, pool->head_dim, G, stream) != cudaSuccess) {
        return PKV_ERR_CUDA;
    }
    if (direct && parts > 1) {
        pkv::MergeParams mp{};
        mp.ws_m = p.ws_m;
        mp.ws_l = p.ws_l;
        mp.ws_o = p.ws_o;
        mp.context_lens = a.ctx;
        mp.num_seqs = a.S;
        mp.num_q_heads = a.Hq;
        mp.head_dim = pool->head_dim;
        mp.max_parts = parts;
        mp.partition_size = P;
        mp.skip_single = 1;
        mp.num_queries = a.NQ;
        mp.prefix_parts = 0;
        mp.skip_tokens = 0;
        mp.out = out;
        mp.out_dtype = out_dtype;
        mp.err = err;
        if (pkv::launch_merge(mp, stream) != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

}  // namespace

bool pkv::use_tensor_cores(int group) {
    const int e = g_engine.load(std::memory_order_relaxed);
    return e == PKV_ENGINE_TENSOR_CORES || (e == PKV_ENGINE_AUTO && group >= 4);
}

// Partition scratch of pkv_paged_attention_decode_static_workspace, for callers
// that cannot allocate device memory: one fixed array per device, held for the
// life of the process, shared by every call of that entry point.
static __device__ __align__(256) unsigned char pkv_static_workspace[PKV_STATIC_WORKSPACE_BYTES];

namespace {

void* g_static_ws_ptr[MAX_DEVICES] = {nullptr};
cudaError_t g_static_ws_status[MAX_DEVICES];
std::once_flag g_static_ws_once[MAX_DEVICES];

// Device address of the array on the current device, looked up once per
// device with that device current.  Host code only sees a stand-in for the
// array's name, never a usable device address, so the kernels get this one.
pkv_status static_workspace(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return PKV_ERR_CUDA;
    std::call_once(g_static_ws_once[dev], [dev] {
        void* ptr = nullptr;
        g_static_ws_status[dev] = cudaGetSymbolAddress(&ptr, pkv_static_workspace);
        g_static_ws_ptr[dev] = ptr;
    });
    if (g_static_ws_status[dev] != cudaSuccess || !g_static_ws_ptr[dev]) return PKV_ERR_CUDA;
    *out = g_static_ws_ptr[dev];
    return PKV_OK;
}

}  // namespace

extern "C" {

int32_t pkv_version(void) { return 100; }

pkv_status pkv_set_decode_engine(int32_t engine) {
    if (engine != PKV_ENGINE_AUTO && engine != PKV_ENGINE_CUDA_CORES &&
        engine != PKV_ENGINE_TENSOR_CORES)
        return PKV_ERR_INVALID;
    g_engine.store(engine, std::memory_order_relaxed);
    return PKV_OK;
}

int32_t pkv_get_decode_engine(void) { return g_engine.load(std::memory_order_relaxed); }

const char* pkv_status_str(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_DEVICE: return "device error flags set";
    }
    return "unknown status";
}

pkv_status pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                            int32_t num_seqs, const int32_t* positions, const int32_t* token_seq,
                            int32_t num_tokens, int32_t block_size, int64_t* slot_mapping,
                            void* stream) {
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq <= 0 || num_seqs < 0)
        return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!block_tables || !positions || !slot_mapping || num_seqs == 0) return PKV_ERR_INVALID;
    if (!token_seq && num_tokens > num_seqs) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_slot_mapping(block_tables, max_blocks_per_seq, num_seqs, positions,
                                    token_seq, num_tokens, block_size, slot_mapping, err,
                                    static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_kv_cache_write(const pkv_pool* pool, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, int32_t num_tokens, void* stream) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !slot_mapping || !aligned16(k_new) || !aligned16(v_new))
        return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_cache_write(*pool, k_new, v_new, slot_mapping, num_tokens, err,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

int32_t pkv_choose_partition_size(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len) {
    (void)num_seqs;
    (void)num_q_heads;
    if (!pool || pool->block_size <= 0 || max_context_len < 0) return 0;
    return auto_partition(pool, max_context_len);
}

size_t pkv_decode_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, int32_t partition_size) {
    if (!pool || pool->block_size <= 0 || pool->head_dim <= 0 || num_seqs < 0 ||
        num_q_heads <= 0 || max_context_len < 0 || partition_size < 0)
        return 0;
    const int32_t P = partition_size > 0 ? partition_size : auto_partition(pool, max_context_len);
    const int32_t parts = max_context_len > 0 ? ceil_div(max_context_len, P) : 1;
    if (parts <= 1) return 0;
    return ws_layout(num_seqs, num_q_heads, pool->head_dim, parts).bytes;
}

size_t pkv_partition_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                     int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
        partition_size <= 0)
        return 0;
    const int32_t parts = max_context_len > 0 ? ceil_div(max_context_len, partition_size) : 1;
    return ws_layout(num_seqs, num_q_heads, head_dim, parts).bytes;
}

pkv_status pkv_paged_attention_decode(const pkv_pool* pool, const void* q, int32_t num_seqs,
                                      int32_t num_q_heads, const int32_t* block_tables,
                                      int32_t max_blocks_per_seq, const int32_t* context_lens,
                                      int32_t max_context_len, float scale, void* out,
                                      int32_t out_dtype, int32_t partition_size, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && !out) return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    return run_decode(a, out, out_dtype, 1, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

pkv_status pkv_paged_attention_decode_static_workspace(
    const pkv_pool* pool, const void* q, int32_t num_seqs, int32_t num_q_heads,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, float scale, void* out, int32_t out_dtype, int32_t partition_size,
    void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && !out) return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv_decode_workspace_bytes(pool, num_seqs, num_q_heads, max_context_len,
                                                   partition_size);
    if (need > PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE;
    if (num_seqs == 0) return PKV_OK;
    void* ws = nullptr;
    st = static_workspace(&ws);
    if (st != PKV_OK) return st;
    return run_decode(a, out, out_dtype, 1, ws, PKV_STATIC_WORKSPACE_BYTES,
                      static_cast<cudaStream_t>(stream));
}

pkv_status pkv_paged_attention_decode_append(
    const pkv_pool* pool, const void* q, const void* k_new, const void* v_new, int32_t num_seqs,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, void* out,
    int32_t out_dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
    int64_t* slot_mapping, void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (num_seqs > 0 && (!out || !k_new || !v_new)) return PKV_ERR_INVALID;
    if (num_seqs > 0 && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    const AppendArgs app{k_new, v_new, slot_mapping};
    return run_decode(a, out, out_dtype, 1, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), &app);
}

pkv_status pkv_paged_attention_decode_multi(
    const pkv_pool* pool, const void* q, int32_t num_queries, int32_t num_seqs,
    int32_t num_q_heads, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* context_lens, int32_t max_context_len, float scale, void* out,
    int32_t out_dtype, int32_t partition_size, void* workspace, size_t workspace_bytes,
    void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (num_queries < 1 || (int64_t)num_seqs * num_queries > INT32_MAX) return PKV_ERR_INVALID;
    if (num_seqs > 0 && !out) return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    if (pool->dtype == PKV_F32) return PKV_ERR_UNSUPPORTED;
    a.NQ = num_queries;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    if ((int64_t)pool->num_kv_heads * ((num_queries + 8 / G - 1) / (8 / G)) > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    return run_decode(a, out, out_dtype, 1, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

pkv_status pkv_paged_attention_decode_multi_append(
    const pkv_pool* pool, const void* q, const void* k_new, const void* v_new,
    int32_t num_queries, int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t max_context_len,
    float scale, void* out, int32_t out_dtype, int32_t partition_size, void* workspace,
    size_t workspace_bytes, int64_t* slot_mapping, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)))
        return PKV_ERR_INVALID;
    if (num_queries == 1)
        return pkv_paged_attention_decode_append(pool, q, k_new, v_new, num_seqs, num_q_heads,
                                                 block_tables, max_blocks_per_seq, context_lens,
                                                 max_context_len, scale, out, out_dtype,
                                                 partition_size, workspace, workspace_bytes,
                                                 slot_mapping, stream);
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (num_queries < 1 || (int64_t)num_seqs * num_queries > INT32_MAX) return PKV_ERR_INVALID;
    if (num_seqs > 0 && !out) return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    if (pool->dtype == PKV_F32) return PKV_ERR_UNSUPPORTED;
    a.NQ = num_queries;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    if ((int64_t)pool->num_kv_heads * ((num_queries + 8 / G - 1) / (8 / G)) > INT32_MAX)
        return PKV_ERR_UNSUPPORTED;
    const AppendArgs app{k_new, v_new, slot_mapping};
    return run_decode(a, out, out_dtype, 1, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream), &app);
}

namespace {

struct CascadeShape {
    int32_t P, suffix_parts, prefix_splits, tokens_per_split, max_parts;
};

// Streaming multiprocessors of the current device (152 when it cannot be asked).
int32_t sm_count() {
    static std::atomic<int32_t> cached[64];  // 0 until asked; racing callers agree
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int32_t n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The prefix pass runs two CTAs per SM over (kv head, 128-row tile, split of the
// prefix); the split count minimises waves x (64-token chunks per split + 3), the 3
// standing for a CTA's fixed cost (query tile, pipeline fill, epilogue).  Each split
// writes one slot, followed by the suffix partitions.
CascadeShape cascade_shape(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                           int32_t max_ctx, int32_t prefix_len, int32_t partition_size) {
    const int32_t rest = max_ctx > prefix_len ? max_ctx - prefix_len : 0;
    const int32_t P = partition_size > 0 ? partition_size : auto_partition(pool, rest);
    const int32_t sp = rest > 0 ? ceil_div(rest, P) : 1;
    const int32_t G = num_q_heads / pool->num_kv_heads;
    const int64_t ctas = std::max<int64_t>(
        1, (int64_t)pool->num_kv_heads * (((int64_t)num_seqs * G + 127) / 128));
    const int64_t sms = sm_count();
    const int32_t chunks = std::max<int32_t>(1, ceil_div(prefix_len, 64));
    int32_t best_cps = chunks;
    int64_t best_cost = INT64_MAX;
    for (int32_t s = 1; s <= std::min<int32_t>(chunks, 64); ++s) {
        const int32_t cps = ceil_div(chunks, s);
        const int64_t splits = ceil_div(chunks, cps);
        const int64_t waves = (ctas * splits + 2 * sms - 1) / (2 * sms);  // two CTAs per SM
        const int64_t cost = waves * (cps + 3);
        if (cost < best_cost) {
            best_cost = cost;
            best_cps = cps;
        }
    }
    const int32_t splits = ceil_div(chunks, best_cps);
    return CascadeShape{P, sp, splits, best_cps * 64, splits + sp};
}

}  // namespace

size_t pkv_cascade_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                                   int32_t max_context_len, int32_t prefix_len,
                                   int32_t partition_size) {
    if (!pool || pool->block_size <= 0 || pool->head_dim <= 0 || num_seqs < 0 ||
        num_q_heads <= 0 || max_context_len < 0 || prefix_len <= 0 || partition_size < 0)
        return 0;
    if (num_q_heads % pool->num_kv_heads != 0) return 0;
    const CascadeShape c =
        cascade_shape(pool, num_seqs, num_q_heads, max_context_len, prefix_len, partition_size);
    return ws_layout(num_seqs, num_q_heads, pool->head_dim, c.max_parts).bytes;
}

pkv_status pkv_paged_attention_decode_cascade(
    const pkv_pool* pool, const void* q, int32_t num_seqs, int32_t num_q_heads,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t max_context_len, float scale, int32_t prefix_len, void* out, int32_t out_dtype,
    int32_t partition_size, const void* k_new, const void* v_new, int64_t* slot_mapping,
    void* workspace, size_t workspace_bytes, void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (pool->dtype == PKV_F32) return PKV_ERR_UNSUPPORTED;
    if (out_dtype != PKV_F32 && out_dtype != pool->dtype) return PKV_ERR_UNSUPPORTED;
    if (prefix_len <= 0 || prefix_len % 16 != 0 || prefix_len % pool->block_size != 0 ||
        prefix_len > max_context_len || (int64_t)prefix_len > (int64_t)max_blocks_per_seq * pool->block_size)
        return PKV_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;
    if (num_seqs > 0 && !out) return PKV_ERR_INVALID;
    const CascadeShape c =
        cascade_shape(pool, num_seqs, num_q_heads, max_context_len, prefix_len, partition_size);
    if (c.suffix_parts > 65535) return PKV_ERR_UNSUPPORTED;
    const WsLayout lay = ws_layout(num_seqs, num_q_heads, pool->head_dim, c.max_parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < lay.bytes) return PKV_ERR_WORKSPACE;
    // the prefix pass's limits (tensor-map rows, 128-row tiles in grid.y), checked before
    // anything is launched
    if ((int64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size >= (1ll << 31) ||
        ((int64_t)num_seqs * (num_q_heads / pool->num_kv_heads) + 127) / 128 > 65535)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    unsigned int* err = nullptr;
    st = error_word(&err);
    if (st != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* ws_m = reinterpret_cast<float*>(ws);
    float* ws_l = reinterpret_cast<float*>(ws + lay.l_off);
    float* ws_o = reinterpret_cast<float*>(ws + lay.o_off);
    const int G = num_q_heads / pool->num_kv_heads;

    pkv::DecodeParams p{};
    p.k_pool = pool->k;
    p.v_pool = pool->v;
    p.num_blocks = pool->num_blocks;
    p.block_size = pool->block_size;
    p.num_kv_heads = pool->num_kv_heads;
    p.q = q;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.block_tables = block_tables;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.max_context_len = max_context_len;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.partition_size = c.P;
    p.max_parts = c.max_parts;
    p.out = out;
    p.out_dtype = out_dtype;
    p.direct_single = 0;
    p.skip_tokens = prefix_len;
    p.part_offset = c.prefix_splits;
    p.num_queries = 1;
    p.queries_per_cta = 1;
    p.ws_m = ws_m;
    p.ws_l = ws_l;
    p.ws_o = ws_o;
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_out = slot_mapping;
    p.err = err;
    // the suffix decode's grid covers max_parts - part_offset = suffix partitions.  It goes
    // first and lets the prefix pass start on the SMs its last CTAs leave idle (the two
    // read and write disjoint data); the prefix pass ends only after it.
    p.trigger_dependents = 1;
    if (launch_decode_typed(p, pool->dtype, pool->head_dim, G, s) != cudaSuccess)
        return PKV_ERR_CUDA;

    pkv::PrefixParams pp{};
    pp.q = q;
    pp.num_seqs = num_seqs;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = pool->num_kv_heads;
    pp.num_blocks = pool->num_blocks;
    pp.block_size = pool->block_size;
    pp.block_tables = block_tables;
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.prefix_len = prefix_len;
    pp.scale_log2 = scale * 1.4426950408889634f;
    pp.max_parts = c.max_parts;
    pp.tokens_per_split = c.tokens_per_split;
    pp.ws_m = ws_m;
    pp.ws_l = ws_l;
    pp.ws_o = ws_o;
    pp.err = err;
    cudaError_t e = pool->dtype == PKV_F16
                        ? pkv::launch_prefix<__half>(pp, pool->k, pool->v, pool->head_dim, s)
                        : pkv::launch_prefix<__nv_bfloat16>(pp, pool->k, pool->v, pool->head_dim, s);
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PKV_ERR_CUDA;

    pkv::MergeParams mp{};
    mp.ws_m = ws_m;
    mp.ws_l = ws_l;
    mp.ws_o = ws_o;
    mp.context_lens = context_lens;
    mp.num_seqs = num_seqs;
    mp.num_q_heads = num_q_heads;
    mp.head_dim = pool->head_dim;
    mp.max_parts = c.max_parts;
    mp.partition_size = c.P;
    mp.skip_single = 0;
    mp.num_queries = 1;
    mp.prefix_parts = c.prefix_splits;
    mp.skip_tokens = prefix_len;
    mp.out = out;
    mp.out_dtype = out_dtype;
    mp.err = err;
    return pkv::launch_merge(mp, s) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_attention_partitions(const pkv_pool* pool, const void* q, int32_t num_seqs,
                                          int32_t num_q_heads, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t max_context_len,
                                          float scale, int32_t partition_size, void* workspace,
                                          size_t workspace_bytes, void* stream) {
    DecodeArgs a{pool, q, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                 context_lens, max_context_len, scale, partition_size};
    pkv_status st = check_decode(a);
    if (st != PKV_OK) return st;
    if (partition_size <= 0) return PKV_ERR_INVALID;
    return run_decode(a, nullptr, PKV_F32, 0, workspace, workspace_bytes,
                      static_cast<cudaStream_t>(stream));
}

pkv_status pkv_lse_merge(const void* workspace, size_t workspace_bytes, int32_t num_seqs,
                         int32_t num_q_heads, int32_t head_dim, const int32_t* context_lens,
                         int32_t max_context_len, int32_t partition_size, void* out,
                         int32_t out_dtype, void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0 || partition_size <= 0)
        return PKV_ERR_INVALID;
    if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16)
        return PKV_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!context_lens || !out) return PKV_ERR_INVALID;
    const int32_t parts = max_context_len > 0 ? ceil_div(max_context_len, partition_size) : 1;
    const WsLayout lay = ws_layout(num_seqs, num_q_heads, head_dim, parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < lay.bytes) return PKV_ERR_WORKSPACE;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;
    const char* ws = static_cast<const char*>(workspace);
    pkv::MergeParams mp{};
    mp.ws_m = reinterpret_cast<const float*>(ws);
    mp.ws_l = reinterpret_cast<const float*>(ws + lay.l_off);
    mp.ws_o = reinterpret_cast<const float*>(ws + lay.o_off);
    mp.context_lens = context_lens;
    mp.num_seqs = num_seqs;
    mp.num_q_heads = num_q_heads;
    mp.head_dim = head_dim;
    mp.max_parts = parts;
    mp.partition_size = partition_size;
    mp.skip_single = 0;
    mp.num_queries = 1;
    mp.prefix_parts = 0;
    mp.skip_tokens = 0;
    mp.out = out;
    mp.out_dtype = out_dtype;
    mp.err = err;
    return pkv::launch_merge(mp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PKV_OK
                                                                                 : PKV_ERR_CUDA;
}

pkv_status pkv_copy_blocks(const pkv_pool* pool, const int32_t* src_dst_pairs, int32_t num_pairs,
                           void* stream) {
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (!src_dst_pairs) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_copy_blocks(*pool, *pool, src_dst_pairs, num_pairs, err,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

namespace {

// Device address of a pointer the kernels will dereference: device and managed
// memory as they are, pinned host memory through its mapped device address.
// Pageable host memory the runtime does not know is refused rather than risked.
bool device_addressable(const void* p, const void** out) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged:
            *out = p;
            return true;
        case cudaMemoryTypeHost:
            *out = attr.devicePointer;
            return attr.devicePointer != nullptr;
        default:
            return false;
    }
}

}  // namespace

pkv_status pkv_swap_blocks(const pkv_pool* src, const pkv_pool* dst, const int32_t* src_dst_pairs,
                           int32_t num_pairs, void* stream) {
    pkv_status st = check_pool(src);
    if (st != PKV_OK) return st;
    st = check_pool(dst);
    if (st != PKV_OK) return st;
    if (src->dtype != dst->dtype || src->block_size != dst->block_size ||
        src->num_kv_heads != dst->num_kv_heads || src->head_dim != dst->head_dim)
        return PKV_ERR_INVALID;
    if (num_pairs < 0) return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (!src_dst_pairs) return PKV_ERR_INVALID;
    pkv_pool s2 = *src, d2 = *dst;
    const void* pairs = nullptr;
    const void *sk, *sv, *dk, *dv;
    if (!device_addressable(src->k, &sk) || !device_addressable(src->v, &sv) ||
        !device_addressable(dst->k, &dk) || !device_addressable(dst->v, &dv) ||
        !device_addressable(src_dst_pairs, &pairs))
        return PKV_ERR_INVALID;
    s2.k = const_cast<void*>(sk);
    s2.v = const_cast<void*>(sv);
    d2.k = const_cast<void*>(dk);
    d2.v = const_cast<void*>(dv);
    unsigned int* err = nullptr;
    st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_copy_blocks(s2, d2, static_cast<const int32_t*>(pairs), num_pairs, err,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

static bool allocator_ok(const pkv_block_allocator* a) {
    return a && a->free_ids && a->free_count && a->refcount && a->num_blocks > 0;
}

static pkv::AllocatorState allocator_state(const pkv_block_allocator* a) {
    return pkv::AllocatorState{a->free_ids, a->free_count, a->refcount, a->num_blocks};
}

pkv_status pkv_allocator_reset(const pkv_block_allocator* alloc, void* stream) {
    if (!allocator_ok(alloc)) return PKV_ERR_INVALID;
    return pkv::launch_allocator_reset(allocator_state(alloc), static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_allocate_for_append(const pkv_block_allocator* alloc, const pkv_pool* pool,
                                   int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* old_lens, const int32_t* new_lens,
                                   int32_t num_seqs, int32_t* seq_status, void* stream) {
    if (!allocator_ok(alloc)) return PKV_ERR_INVALID;
    pkv_status st = check_pool(pool);
    if (st != PKV_OK) return st;
    if (alloc->num_blocks != pool->num_blocks || max_blocks_per_seq <= 0 || num_seqs < 0)
        return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables || !old_lens || !new_lens || !seq_status) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_allocate_for_append(allocator_state(alloc), *pool, block_tables,
                                           max_blocks_per_seq, old_lens, new_lens, num_seqs,
                                           seq_status, err, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_fork_sequences(const pkv_block_allocator* alloc, int32_t block_size,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* src_dst_seqs, const int32_t* lens,
                              int32_t num_pairs, void* stream) {
    if (!allocator_ok(alloc) || block_size <= 0 || max_blocks_per_seq <= 0 || num_pairs < 0)
        return PKV_ERR_INVALID;
    if (num_pairs == 0) return PKV_OK;
    if (!block_tables || !src_dst_seqs || !lens) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_fork_sequences(allocator_state(alloc), block_size, block_tables,
                                      max_blocks_per_seq, src_dst_seqs, lens, num_pairs, err,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_free_sequences(const pkv_block_allocator* alloc, int32_t block_size,
                              int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seqs, const int32_t* lens, int32_t num_seqs,
                              void* stream) {
    if (!allocator_ok(alloc) || block_size <= 0 || max_blocks_per_seq <= 0 || num_seqs < 0)
        return PKV_ERR_INVALID;
    if (num_seqs == 0) return PKV_OK;
    if (!block_tables || !seqs || !lens) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;
    return pkv::launch_free_sequences(allocator_state(alloc), block_size, block_tables,
                                      max_blocks_per_seq, seqs, lens, num_seqs, err,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

pkv_status pkv_get_device_error(uint32_t* flags, void* stream) {
    if (!flags) return PKV_ERR_INVALID;
    unsigned int* err = nullptr;
    pkv_status st = error_word(&err);
    if (st != PKV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, err, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(err, 0, sizeof(unsigned int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return PKV_ERR_CUDA;
    *flags = host;
    return host ? PKV_ERR_DEVICE : PKV_OK;
}

}  // extern "C"
