// C ABI of the paged KV-cache decode library (declared in include/pkv.h):
// argument validation, split planning, workspace layout and dispatch.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>  // CUcontext; the two driver calls below are looked up at run time

#include "pkv_internal.h"

namespace pkv {

namespace {
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
std::once_flag g_ctx_once;
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
}  // namespace

uint64_t current_context_id()
{
    std::call_once(g_ctx_once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
    });
    if (!g_ctx_current || !g_ctx_id)
        return 0;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return 0;
    unsigned long long id = 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return static_cast<uint64_t>(id) + 1;  // never 0 for a real context
}

int device_sm_count()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 1;
    if (dev >= 64) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        return n > 0 ? n : 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0)
            n = 1;
        cache[dev] = n;
    }
    return cache[dev];
}

constexpr int kStreamK = -2;  // plan code of the stream-K schedule

// Schedule for these sizes: > 0 fixed partitions of that many tokens, 0 one
// pass per (sequence, KV head), kStreamK equal page ranges per CTA (the
// automatic choice), -1 invalid.  num_layers layers share the lengths.
static int resolve_partition(int num_layers, int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_dim, int block_size, int max_seq_len, int requested)
{
    if (num_layers <= 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size != kBlockSize || max_seq_len < 0 ||
        num_q_heads % num_kv_heads != 0)
        return -1;
    if (requested == -1)
        return 0;
    if (requested == kStreamK)
        return kStreamK;
    if (requested > 0)
        return (requested % kBlockSize == 0) ? requested : -1;
    if (requested != 0)
        return -1;
    // Automatic choice.  Many (sequence, KV head) units keep every CTA busy
    // with whole units: one pass each when contexts are short, else 4096-token
    // items scheduled dynamically, full partitions first and the remainders
    // by size class, largest first, so that the grid ends on short items.
    // Measured on GB300 on the 70B-shaped layers (bf16 / e4m3 / INT4, us):
    // 1536 tokens 237.8 / 134.3 / 150.2, 2048 235.8 / 130.1 / 147.6, 3072
    // 230.7 / 122.7 / 144.9, 4096 227.0 / 122.8 / 141.3, 6144 232.5 / 155.2
    // / 165.6: longer items mean fewer partials and item boundaries until the
    // items get too few for the resident CTAs.  Few units -- long contexts
    // on a small batch -- use stream-K, which splits them evenly across all
    // CTAs.  The threshold is twice the CTAs resident on a GB300 (two per
    // SM); a fixed number keeps the plan, and so the workspace size,
    // independent of the current device.
    const long units = static_cast<long>(num_layers) * num_seqs * num_kv_heads;
    const long many = 2L * 2 * 152;
    if (units >= many)
        return max_seq_len <= 2048 ? 0 : 4096;
    return kStreamK;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace: [256-byte header: status, work counter][arrive counters
// L*S*Hkv u32][partial outputs L*S*Hq*max_parts*D f32][partial (m, l) pairs]
// for L layers (stream-K: partial slots per CTA instead, whatever L).
struct Plan {
    int partition;  // 0 = no split
    int max_parts;
    size_t arrive_off, part_o_off, part_ml_off, bytes;
};

static bool make_plan(int NL, int S, int Hq, int Hkv, int D, int B, int max_len, int requested,
                      Plan *pl)
{
    const int P = resolve_partition(NL, S, Hq, Hkv, D, B, max_len, requested);
    if (P == -1)
        return false;
    pl->partition = P;
    pl->max_parts = 1;
    pl->arrive_off = pl->part_o_off = pl->part_ml_off = 0;
    pl->bytes = kWorkspaceHeader;
    if (P == kStreamK) {
        // Two partial slots per CTA, G rows each.
        const size_t rows = static_cast<size_t>(2) * kStreamKMaxCtas * (Hq / Hkv);
        pl->arrive_off = kWorkspaceHeader;
        pl->part_o_off =
            pl->arrive_off + align256(static_cast<size_t>(NL) * S * Hkv * sizeof(unsigned));
        pl->part_ml_off = pl->part_o_off + align256(rows * D * sizeof(float));
        pl->bytes = pl->part_ml_off + align256(rows * 2 * sizeof(float));
    } else if (P > 0) {
        pl->max_parts = max_len > P ? (max_len + P - 1) / P : 1;
        const size_t rows = static_cast<size_t>(NL) * S * Hq * pl->max_parts;
        pl->arrive_off = kWorkspaceHeader;
        pl->part_o_off =
            pl->arrive_off + align256(static_cast<size_t>(NL) * S * Hkv * sizeof(unsigned));
        pl->part_ml_off = pl->part_o_off + align256(rows * D * sizeof(float));
        pl->bytes = pl->part_ml_off + align256(rows * 2 * sizeof(float));
    }
    return true;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace pkv

using namespace pkv;

extern "C" {

size_t pkv_paged_attn_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_seq_len,
                                     int partition_tokens)
{
    return pkv_paged_attn_layers_workspace_size(1, num_seqs, num_q_heads, num_kv_heads,
                                                head_dim, block_size, max_seq_len,
                                                partition_tokens);
}

int pkv_paged_attn_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_seq_len,
                                    int partition_tokens)
{
    return resolve_partition(1, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_seq_len, partition_tokens);
}

size_t pkv_paged_attn_layers_workspace_size(int num_layers, int num_seqs, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int max_seq_len, int partition_tokens)
{
    Plan pl;
    if (!make_plan(num_layers, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                   max_seq_len, partition_tokens, &pl))
        return 0;
    return pl.bytes;
}

int pkv_paged_attn_layers_partition_tokens(int num_layers, int num_seqs, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int max_seq_len, int partition_tokens)
{
    return resolve_partition(num_layers, num_seqs, num_q_heads, num_kv_heads, head_dim,
                             block_size, max_seq_len, partition_tokens);
}

}  // extern "C"

namespace pkv {

// Decode of one layer (`layers` null: the tensors in `one`, checked here) or
// of num_layers layers whose tensors sit in a device table (checked by the
// kernels), optionally with the fused cache write of one new token per
// sequence (`append`: the layers' new_k rows, where non-null).
static pkv_status decode_impl(const LayerPtrs &one, const LayerPtrs *layers, int num_layers,
                              bool append, pkv_dtype q_dtype, pkv_dtype kv_dtype, float k_scale,
                              float v_scale, const int32_t *block_tables,
                              const int32_t *seq_lens, int num_seqs, int num_q_heads,
                              int num_kv_heads, int head_dim, int block_size, int num_blocks,
                              int max_blocks_per_seq, int max_seq_len, float scale,
                              pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
                              int partition_tokens, int flags, void *stream, pkv_dtype new_dtype,
                              const float *k_head_scales = nullptr,
                              const float *v_head_scales = nullptr)
{
    if (num_layers <= 0 || num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (static_cast<long>(max_seq_len) > static_cast<long>(max_blocks_per_seq) * kBlockSize)
        return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_F32 && q_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && !is_scaled(kv_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (block_size != kBlockSize)
        return PKV_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (group > 16)
        return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
        return PKV_ERR_INVALID_ARG;
    if ((flags & ~(PKV_FLAG_IMPL_MASK | PKV_FLAG_SEPARATE_MERGE | PKV_FLAG_TEST_DROP_FIRST_COPY)) !=
            0 ||
        (flags & PKV_FLAG_IMPL_MASK) == PKV_FLAG_IMPL_MASK)
        return PKV_ERR_INVALID_ARG;
    Plan pl;
    if (!make_plan(num_layers, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                   max_seq_len, partition_tokens, &pl))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.bytes)
        return PKV_ERR_WORKSPACE;
    if (num_seqs == 0)
        return PKV_OK;
    if (!block_tables || !seq_lens || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID_ARG;
    if (layers) {
        if (!aligned(layers, alignof(LayerPtrs)))
            return PKV_ERR_INVALID_ARG;
    } else {
        if (!one.q || !one.k_cache || !one.v_cache || !one.out)
            return PKV_ERR_INVALID_ARG;
        if (!aligned(one.q, 16) || !aligned(one.k_cache, 16) || !aligned(one.v_cache, 16) ||
            !aligned(one.out, 16))
            return PKV_ERR_INVALID_ARG;
        if (append && (!one.new_k || !one.new_v || !aligned(one.new_k, 16) ||
                       !aligned(one.new_v, 16)))
            return PKV_ERR_INVALID_ARG;
    }

    const int impl = flags & PKV_FLAG_IMPL_MASK;
    const bool mma_ok = mma_supports(kv_dtype, q_dtype, head_dim, group);
    if (impl == PKV_FLAG_IMPL_MMA && !mma_ok)
        return PKV_ERR_UNSUPPORTED;
    const bool use_mma = (impl == PKV_FLAG_IMPL_MMA) || (impl == PKV_FLAG_IMPL_AUTO && mma_ok);

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.one = one;
    if (!append)
        p.one.new_k = p.one.new_v = nullptr;
    p.layers = layers;
    p.num_layers = num_layers;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.status = reinterpret_cast<int *>(ws);
    p.counter = reinterpret_cast<unsigned *>(ws + 4);
    const bool partials = pl.partition != 0;
    p.arrive = partials ? reinterpret_cast<unsigned *>(ws + pl.arrive_off) : nullptr;
    p.part_o = partials ? reinterpret_cast<float *>(ws + pl.part_o_off) : nullptr;
    p.part_ml = partials ? reinterpret_cast<float *>(ws + pl.part_ml_off) : nullptr;
    p.q_dtype = q_dtype;
    p.out_dtype = out_dtype;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_len = max_seq_len;
    p.group = group;
    const float k_mul = is_scaled(kv_dtype) ? k_scale : 1.0f;
    p.score_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 * k_mul);
    p.out_scale = is_scaled(kv_dtype) ? v_scale : 1.0f;
    if (use_mma && kv_dtype == PKV_FP8_E4M3) {
        p.score_scale *= kE4m3Shift;
        p.out_scale *= kE4m3Shift;
    }
    p.partition = pl.partition > 0 ? pl.partition : max_blocks_per_seq * kBlockSize;
    p.max_parts = pl.max_parts;
    p.split = pl.partition > 0 ? 1 : 0;
    p.streamk = pl.partition == kStreamK ? 1 : 0;
    p.streamk_max_ctas = kStreamKMaxCtas;
    p.fused_merge = (flags & PKV_FLAG_SEPARATE_MERGE) ? 0 : 1;
    p.drop_first_copy = (flags & PKV_FLAG_TEST_DROP_FIRST_COPY) ? 1 : 0;
    p.append = append ? 1 : 0;
    p.new_dtype = new_dtype;
    p.kv_dtype = kv_dtype;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_head_scale = k_head_scales;
    p.v_head_scale = v_head_scales;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Status word, work counter and arrival counters start at zero.
    const size_t zero_bytes = partials ? pl.part_o_off : 16;
    if (cudaMemsetAsync(ws, 0, zero_bytes, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    pkv_status rc = use_mma ? launch_decode_mma(p, kv_dtype, st) : launch_decode_simt(p, kv_dtype, st);
    if (rc != PKV_OK)
        return rc;
    if (p.split && p.max_parts > 1 && !p.fused_merge)
        rc = launch_merge(p, st);
    return rc;
}

}  // namespace pkv

extern "C" {

pkv_status pkv_paged_attn_decode(const void *q, pkv_dtype q_dtype, const void *k_cache,
                                 const void *v_cache, pkv_dtype kv_dtype, float k_scale,
                                 float v_scale, const int32_t *block_tables,
                                 const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks,
                                 int max_blocks_per_seq, int max_seq_len, float scale, void *out,
                                 pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                 int partition_tokens, int flags, void *stream)
{
    const LayerPtrs one = {q, nullptr, nullptr, const_cast<void *>(k_cache),
                           const_cast<void *>(v_cache), out};
    return decode_impl(one, nullptr, 1, false, q_dtype, kv_dtype, k_scale, v_scale, block_tables,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_blocks_per_seq, max_seq_len, scale, out_dtype, workspace,
                       workspace_bytes, partition_tokens, flags, stream, PKV_F32);
}

pkv_status pkv_paged_attn_decode_append(const void *q, pkv_dtype q_dtype, const void *new_k,
                                        const void *new_v, pkv_dtype new_dtype, void *k_cache,
                                        void *v_cache, pkv_dtype kv_dtype, float k_scale,
                                        float v_scale, const int32_t *block_tables,
                                        const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, int max_blocks_per_seq, int max_seq_len,
                                        float scale, void *out, pkv_dtype out_dtype,
                                        void *workspace, size_t workspace_bytes,
                                        int partition_tokens, int flags, void *stream)
{
    if (new_dtype != PKV_F32 && new_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (is_scaled(kv_dtype) && (k_scale == 0.f || v_scale == 0.f))
        return PKV_ERR_INVALID_ARG;
    const LayerPtrs one = {q, new_k, new_v, k_cache, v_cache, out};
    return decode_impl(one, nullptr, 1, true, q_dtype, kv_dtype, k_scale, v_scale, block_tables,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_blocks_per_seq, max_seq_len, scale, out_dtype, workspace,
                       workspace_bytes, partition_tokens, flags, stream, new_dtype);
}

pkv_status pkv_paged_attn_decode_layers(const pkv_layer *layers, int num_layers,
                                        pkv_dtype q_dtype, pkv_dtype new_dtype,
                                        pkv_dtype kv_dtype, float k_scale, float v_scale,
                                        const int32_t *block_tables, const int32_t *seq_lens,
                                        int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int num_blocks,
                                        int max_blocks_per_seq, int max_seq_len, float scale,
                                        pkv_dtype out_dtype, void *workspace,
                                        size_t workspace_bytes, int partition_tokens, int flags,
                                        void *stream)
{
    static_assert(sizeof(pkv_layer) == sizeof(LayerPtrs), "pkv_layer layout");
    if (!layers)
        return PKV_ERR_INVALID_ARG;
    if (new_dtype != PKV_F32 && new_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (is_scaled(kv_dtype) && (k_scale == 0.f || v_scale == 0.f))
        return PKV_ERR_INVALID_ARG;
    const LayerPtrs none = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    return decode_impl(none, reinterpret_cast<const LayerPtrs *>(layers), num_layers, true,
                       q_dtype, kv_dtype, k_scale, v_scale, block_tables, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                       max_blocks_per_seq, max_seq_len, scale, out_dtype, workspace,
                       workspace_bytes, partition_tokens, flags, stream, new_dtype);
}

pkv_status pkv_paged_attn_decode_head_scaled(
    const void *q, pkv_dtype q_dtype, const void *k_cache, const void *v_cache, pkv_dtype kv_dtype,
    const float *k_head_scales, const float *v_head_scales, const int32_t *block_tables,
    const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_seq_len, float scale,
    void *out, pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
    int partition_tokens, int flags, void *stream)
{
    if (!is_scaled(kv_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 0 && (!k_head_scales || !v_head_scales || !aligned(k_head_scales, 4) ||
                         !aligned(v_head_scales, 4)))
        return PKV_ERR_INVALID_ARG;
    const LayerPtrs one = {q, nullptr, nullptr, const_cast<void *>(k_cache),
                           const_cast<void *>(v_cache), out};
    return decode_impl(one, nullptr, 1, false, q_dtype, kv_dtype, 1.0f, 1.0f, block_tables,
                       seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_blocks_per_seq, max_seq_len, scale, out_dtype, workspace,
                       workspace_bytes, partition_tokens, flags, stream, PKV_F32, k_head_scales,
                       v_head_scales);
}

static pkv_status reshape_impl(const void *k, const void *v, pkv_dtype in_dtype,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, void *k_cache,
                               void *v_cache, pkv_dtype kv_dtype, float k_scale, float v_scale,
                               const float *k_head_scales, const float *v_head_scales,
                               int32_t *status, void *stream);

pkv_status pkv_reshape_and_cache(const void *k, const void *v, pkv_dtype in_dtype,
                                 const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks, void *k_cache,
                                 void *v_cache, pkv_dtype kv_dtype, float k_scale, float v_scale,
                                 int32_t *status, void *stream)
{
    return reshape_impl(k, v, in_dtype, slot_mapping, num_tokens, num_kv_heads, head_dim,
                        block_size, num_blocks, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                        nullptr, nullptr, status, stream);
}

pkv_status pkv_reshape_and_cache_head_scaled(const void *k, const void *v, pkv_dtype in_dtype,
                                             const int64_t *slot_mapping, int num_tokens,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int num_blocks, void *k_cache, void *v_cache,
                                             pkv_dtype kv_dtype, const float *k_head_scales,
                                             const float *v_head_scales, int32_t *status,
                                             void *stream)
{
    if (!is_scaled(kv_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (num_tokens > 0 && (!k_head_scales || !v_head_scales || !aligned(k_head_scales, 4) ||
                           !aligned(v_head_scales, 4)))
        return PKV_ERR_INVALID_ARG;
    return reshape_impl(k, v, in_dtype, slot_mapping, num_tokens, num_kv_heads, head_dim,
                        block_size, num_blocks, k_cache, v_cache, kv_dtype, 1.0f, 1.0f,
                        k_head_scales, v_head_scales, status, stream);
}

static pkv_status reshape_impl(const void *k, const void *v, pkv_dtype in_dtype,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, void *k_cache,
                               void *v_cache, pkv_dtype kv_dtype, float k_scale, float v_scale,
                               const float *k_head_scales, const float *v_head_scales,
                               int32_t *status, void *stream)
{
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size != kBlockSize)
        return PKV_ERR_UNSUPPORTED;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && !is_scaled(kv_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (is_scaled(kv_dtype) &&
        (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f || v_scale == 0.f))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || (status && !aligned(status, 4)))
        return PKV_ERR_INVALID_ARG;
    return launch_reshape_and_cache(k, v, in_dtype, slot_mapping, num_tokens, num_kv_heads,
                                    head_dim, num_blocks, k_cache, v_cache, kv_dtype, k_scale,
                                    v_scale, k_head_scales, v_head_scales, status,
                                    static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace pkv {

// Split plan of the several-queries kernel.  Items are (sequence, KV head,
// partition, 64-row block); the host knows only T, S and the length bounds,
// so it estimates the unsplit item count from them.  Enough items keep every
// CTA busy without a split (contexts over 2048 tokens still use 4096-token
// partitions so long items do not dominate the tail); fewer are split so
// that about four items per resident CTA exist.
static int resolve_prefill_partition(int S, int T, int Hq, int Hkv, int B, int max_q_len,
                                     int max_len, int requested)
{
    if (S < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || B != kBlockSize ||
        max_len < 0 || max_q_len < 0)
        return -1;
    if (requested == -1)
        return 0;
    if (requested > 0)
        return requested % kBlockSize == 0 ? requested : -1;
    if (requested != 0)
        return -1;
    const long G = Hq / Hkv;
    const long blocks = (static_cast<long>(T) * G + 63) / 64;
    const long est = static_cast<long>(Hkv) * (blocks > S ? blocks : S);
    const long many = 2L * 2 * 152;
    // Two waves or more: 4096-token partitions (the tcgen05 kernel hands out
    // the last partitions largest first; verification layer, same box: 2048
    // tokens 324.8 us, 3072 317.5, 4096 315.2).
    if (est >= many)
        return max_len <= 2048 ? 0 : 4096;
    // One wave of items or more (two CTAs per SM): no split -- no partials
    // and no merge (measured on GB300, chunked prefill of the 8B layer,
    // 544 estimated items: no split 258 us, 2048-token partitions 275 us).
    if (2 * est >= many)
        return 0;
    const long parts = (many + est - 1) / (est > 0 ? est : 1);
    long P = (max_len + parts - 1) / parts;
    P = (P + 255) / 256 * 256;
    if (P < 256)
        P = 256;
    return max_len <= P ? 0 : static_cast<int>(P);
}

// Workspace of the several-queries call: [256-byte header: status word,
// work counter, the routed decode's work counter][partials of the
// several-queries kernels][the routed decode's arrival counters and
// partials, as its own plan lays them out after its header].
struct PrefillPlan {
    int partition;  // 0 = no split
    int max_parts;
    size_t part_o_off, part_ml_off, bytes;
    bool route;     // one-query sequences run on the decode kernels
    Plan dec;       // their decode plan
    size_t dec_off; // where the decode plan's bytes after its header start
};

// Mixed batches -- some sequences with one query, others with several, as
// chunked prefill schedules prompt chunks with decoding sequences -- and
// all-one-query batches send their one-query sequences to the decode
// kernels: on the several-queries kernels a one-query sequence is an item
// of G rows padded to the tensor-core tile (128 rows on tcgen05), while the
// decode kernels put the page's tokens on the MMA and stream it at the decode
// rate.  A batch whose every sequence has max_q_len queries (speculative
// verification) stays on the several-queries kernels.
static bool route_single(int S, int T, int max_q_len)
{
    return S > 0 && T > 0 && (max_q_len == 1 || static_cast<long>(T) < static_cast<long>(S) * max_q_len);
}

static bool make_prefill_plan(int S, int T, int Hq, int Hkv, int D, int B, int max_q_len,
                              int max_len, int requested, PrefillPlan *pl)
{
    const int P = resolve_prefill_partition(S, T, Hq, Hkv, B, max_q_len, max_len, requested);
    if (P < 0)
        return false;
    pl->partition = P;
    pl->max_parts = (P > 0 && max_len > P) ? (max_len + P - 1) / P : 1;
    pl->part_o_off = pl->part_ml_off = 0;
    pl->bytes = kWorkspaceHeader;
    if (pl->max_parts > 1) {
        const size_t rows = static_cast<size_t>(T) * Hq * pl->max_parts;
        pl->part_o_off = kWorkspaceHeader;
        pl->part_ml_off = pl->part_o_off + align256(rows * D * sizeof(float));
        pl->bytes = pl->part_ml_off + align256(rows * 2 * sizeof(float));
    }
    pl->route = route_single(S, T, max_q_len);
    pl->dec_off = 0;
    if (pl->route) {
        // The caller's partition request applies to both kernels.  The
        // automatic one gives the routed decode the item schedule once its
        // (sequence, KV head) units fill a wave of decode CTAs (three per
        // SM): measured after the several-queries kernel of the 8B chunked
        // prefill (512 units), stream-K 130 us, items 115 us.
        int dreq = requested;
        if (requested == 0 && static_cast<long>(S) * Hkv >= 3L * 152)
            dreq = max_len <= 2048 ? -1 : 4096;
        if (!make_plan(1, S, Hq, Hkv, D, B, max_len, dreq, &pl->dec))
            return false;
        pl->dec_off = align256(pl->bytes);
        pl->bytes = pl->dec_off + (pl->dec.bytes - kWorkspaceHeader);
    }
    return true;
}

}  // namespace pkv

extern "C" {

size_t pkv_paged_attn_prefill_workspace_size(int num_seqs, int num_tokens, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int max_q_len, int max_seq_len,
                                             int partition_tokens)
{
    PrefillPlan pl;
    if (!make_prefill_plan(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_q_len, max_seq_len, partition_tokens, &pl))
        return 0;
    return pl.bytes;
}

int pkv_paged_attn_prefill_partition_tokens(int num_seqs, int num_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int max_q_len, int max_seq_len,
                                            int partition_tokens)
{
    (void)head_dim;
    return resolve_prefill_partition(num_seqs, num_tokens, num_q_heads, num_kv_heads, block_size,
                                     max_q_len, max_seq_len, partition_tokens);
}

pkv_status pkv_paged_attn_prefill(const void *q, pkv_dtype q_dtype, const int32_t *q_start,
                                  const void *k_cache, const void *v_cache, pkv_dtype kv_dtype,
                                  float k_scale, float v_scale, const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs, int num_tokens,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                  int max_q_len, int max_seq_len, float scale, void *out,
                                  pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                  int partition_tokens, int flags, void *stream)
{
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 || max_q_len < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0)
        return PKV_ERR_INVALID_ARG;
    if (static_cast<long>(max_seq_len) > static_cast<long>(max_blocks_per_seq) * kBlockSize)
        return PKV_ERR_INVALID_ARG;
    if (q_dtype != PKV_BF16 || (kv_dtype != PKV_BF16 && !is_scaled(kv_dtype)))
        return PKV_ERR_UNSUPPORTED;
    // fp8 / INT4 caches run on the mma.sync kernel; the tcgen05 one is bf16 only.
    if (is_scaled(kv_dtype) && (flags & PKV_FLAG_IMPL_MASK) == PKV_FLAG_IMPL_TC)
        return PKV_ERR_UNSUPPORTED;
    if (is_scaled(kv_dtype) &&
        (!std::isfinite(k_scale) || !std::isfinite(v_scale) || k_scale == 0.f || v_scale == 0.f))
        return PKV_ERR_INVALID_ARG;
    if (out_dtype != PKV_F32 && out_dtype != PKV_BF16)
        return PKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128)
        return PKV_ERR_UNSUPPORTED;
    if (block_size != kBlockSize)
        return PKV_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (group > 16)
        return PKV_ERR_UNSUPPORTED;
    if (!std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if ((flags & ~(PKV_FLAG_IMPL_MASK | PKV_FLAG_TEST_DROP_FIRST_COPY)) != 0 ||
        (flags & PKV_FLAG_IMPL_MASK) == PKV_FLAG_IMPL_SIMT)
        return PKV_ERR_INVALID_ARG;
    PrefillPlan pl;
    if (!make_prefill_plan(num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_q_len, max_seq_len, partition_tokens, &pl))
        return PKV_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < pl.bytes)
        return PKV_ERR_WORKSPACE;
    if (num_seqs == 0 || num_tokens == 0)
        return PKV_OK;
    if (!q || !q_start || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
        return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(q_start, 4) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID_ARG;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    PrefillParams p;
    std::memset(&p, 0, sizeof p);
    p.q = q;
    p.q_start = q_start;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = out;
    p.status = reinterpret_cast<int *>(ws);
    p.counter = reinterpret_cast<unsigned *>(ws + 4);
    p.part_o = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.part_o_off) : nullptr;
    p.part_ml = pl.max_parts > 1 ? reinterpret_cast<float *>(ws + pl.part_ml_off) : nullptr;
    p.out_dtype = out_dtype;
    p.num_seqs = num_seqs;
    p.num_tokens = num_tokens;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.max_len = max_seq_len;
    p.max_q_len = max_q_len;
    p.group = group;
    p.kv_dtype = kv_dtype;
    const bool scaled = is_scaled(kv_dtype);
    p.score_scale = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 *
                                       (scaled ? k_scale : 1.0f));
    p.out_scale = scaled ? v_scale : 1.0f;
    if (kv_dtype == PKV_FP8_E4M3) {  // codes widened to 2^-8 times their value
        p.score_scale *= kE4m3Shift;
        p.out_scale *= kE4m3Shift;
    }
    p.partition = pl.partition > 0 ? pl.partition : max_blocks_per_seq * kBlockSize;
    p.max_parts = pl.max_parts;
    p.drop_first_copy = (flags & PKV_FLAG_TEST_DROP_FIRST_COPY) ? 1 : 0;
    // Automatic: the tcgen05 kernel for bf16 caches (faster on every measured
    // layer), the mma.sync kernel for fp8 / INT4 caches.
    p.impl = ((flags & PKV_FLAG_IMPL_MASK) == PKV_FLAG_IMPL_MMA || scaled) ? PKV_FLAG_IMPL_MMA
                                                                          : PKV_FLAG_IMPL_TC;
    p.skip_single = pl.route ? 1 : 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Status word and the two work counters.
    if (cudaMemsetAsync(ws, 0, 16, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    pkv_status rc = PKV_OK;
    if (max_q_len > 1 || !pl.route)
        rc = launch_prefill(p, kv_dtype, st);
    if (rc != PKV_OK || !pl.route)
        return rc;

    // The one-query sequences: decode, reading and writing row q_start[s].
    const Plan &dp = pl.dec;
    unsigned char *dws = ws + pl.dec_off - kWorkspaceHeader;  // the decode plan's offsets
    DecodeParams d;
    std::memset(&d, 0, sizeof d);
    d.one = {q, nullptr, nullptr, const_cast<void *>(k_cache), const_cast<void *>(v_cache), out};
    d.num_layers = 1;
    d.block_tables = block_tables;
    d.seq_lens = seq_lens;
    d.status = reinterpret_cast<int *>(ws);
    d.counter = reinterpret_cast<unsigned *>(ws + 8);
    const bool partials = dp.partition != 0;
    d.arrive = partials ? reinterpret_cast<unsigned *>(dws + dp.arrive_off) : nullptr;
    d.part_o = partials ? reinterpret_cast<float *>(dws + dp.part_o_off) : nullptr;
    d.part_ml = partials ? reinterpret_cast<float *>(dws + dp.part_ml_off) : nullptr;
    d.q_dtype = q_dtype;
    d.out_dtype = out_dtype;
    d.num_seqs = num_seqs;
    d.num_q_heads = num_q_heads;
    d.num_kv_heads = num_kv_heads;
    d.head_dim = head_dim;
    d.num_blocks = num_blocks;
    d.max_blocks = max_blocks_per_seq;
    d.max_len = max_seq_len;
    d.group = group;
    d.score_scale = p.score_scale;  // same folding (k_scale, the e4m3 shift) as the mma policies
    d.out_scale = p.out_scale;
    d.partition = dp.partition > 0 ? dp.partition : max_blocks_per_seq * kBlockSize;
    d.max_parts = dp.max_parts;
    d.split = dp.partition > 0 ? 1 : 0;
    d.streamk = dp.partition == kStreamK ? 1 : 0;
    d.streamk_max_ctas = kStreamKMaxCtas;
    d.fused_merge = 1;
    d.new_dtype = PKV_F32;
    d.kv_dtype = kv_dtype;
    d.k_scale = k_scale;
    d.v_scale = v_scale;
    d.q_rows = q_start;
    d.num_rows = num_tokens;
    if (partials && cudaMemsetAsync(dws + dp.arrive_off, 0, dp.part_o_off - dp.arrive_off, st) !=
                        cudaSuccess)
        return PKV_ERR_CUDA;
    return launch_decode_mma(d, kv_dtype, st);
}

pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, pkv_dtype kv_dtype, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, const int32_t *pairs,
                           int num_pairs, int32_t *status, void *stream)
{
    if (num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || num_pairs < 0)
        return PKV_ERR_INVALID_ARG;
    if (block_size != kBlockSize)
        return PKV_ERR_UNSUPPORTED;
    if (kv_dtype != PKV_F32 && kv_dtype != PKV_BF16 && !is_scaled(kv_dtype))
        return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0)
        return PKV_OK;
    if (!k_cache || !v_cache || !pairs)
        return PKV_ERR_INVALID_ARG;
    const size_t block_bytes =
        static_cast<size_t>(num_kv_heads) * static_cast<size_t>(tile_bytes(kv_dtype, head_dim));
    if (block_bytes % 16 != 0 || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(pairs, 4) || (status && !aligned(status, 4)))
        return PKV_ERR_INVALID_ARG;
    return launch_copy_blocks(k_cache, v_cache, block_bytes, pairs, num_pairs, num_blocks, status,
                              static_cast<cudaStream_t>(stream));
}

pkv_status pkv_read_status(void *workspace, int clear, int32_t *host_status, void *stream)
{
    if (!workspace || !host_status)
        return PKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (clear && cudaMemsetAsync(workspace, 0, sizeof v, st) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return PKV_ERR_CUDA;
    *host_status = v;
    return PKV_OK;
}

const char *pkv_status_string(pkv_status status)
{
    switch (status) {
    case PKV_OK:
        return "PKV_OK";
    case PKV_ERR_INVALID_ARG:
        return "PKV_ERR_INVALID_ARG: invalid argument";
    case PKV_ERR_UNSUPPORTED:
        return "PKV_ERR_UNSUPPORTED: unsupported dtype or shape";
    case PKV_ERR_CUDA:
        return "PKV_ERR_CUDA: CUDA runtime error";
    case PKV_ERR_OUT_OF_RANGE:
        return "PKV_ERR_OUT_OF_RANGE: block id, slot or seq_len outside the pool or table";
    case PKV_ERR_TIMEOUT:
        return "PKV_ERR_TIMEOUT: a bounded device wait gave up";
    case PKV_ERR_WORKSPACE:
        return "PKV_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case PKV_ERR_NO_BLOCKS:
        return "PKV_ERR_NO_BLOCKS: the block pool (or host memory) is exhausted";
    default:
        return "PKV_ERR_?: unknown status";
    }
}

int pkv_version(void) { return 100; }

}  // extern "C"
