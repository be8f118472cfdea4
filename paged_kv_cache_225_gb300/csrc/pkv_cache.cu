// Paged KV-cache write ("reshape_and_cache").
//
// The "Inference optimization" lesson (section "Caches de KV") computes K and
// V only for the new token and appends them to the cache; with paging
// (section "PagedAttention") the append lands in a 16-token page anywhere in
// the pool.  Token i goes to slot = slot_mapping[i] = block * 16 + offset of
// every KV head; element (h, d) is stored at [block, h, d, offset].
#include "pkv_convert.cuh"

namespace pkv {

// One CTA per new token; threads stride over (head, dim).
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const void *k, const void *v, int in_dtype,
                             const int64_t *slot_mapping, int num_kv_heads, int head_dim,
                             int num_blocks, void *k_cache, void *v_cache, int kv_dtype,
                             float k_scale, float v_scale, const float *k_head_scale,
                             const float *v_head_scale, int32_t *status)
{
    const int i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0)
        return;
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot - blk * kBlockSize);
    if (blk >= num_blocks) {
        if (threadIdx.x == 0)
            set_status(status, PKV_ERR_OUT_OF_RANGE);
        return;
    }
    const int n = num_kv_heads * head_dim;
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
        const size_t src = static_cast<size_t>(i) * n + e;
        const size_t dst = (static_cast<size_t>(blk) * n + e) * kBlockSize + off;
        const int h = e / head_dim;
        const float ks = k_head_scale ? k_scale * __ldg(k_head_scale + h) : k_scale;
        const float vs = v_head_scale ? v_scale * __ldg(v_head_scale + h) : v_scale;
        store_kv(k_cache, kv_dtype, dst, k, in_dtype, src, ks);
        store_kv(v_cache, kv_dtype, dst, v, in_dtype, src, vs);
    }
}

pkv_status launch_reshape_and_cache(const void *k, const void *v, int in_dtype,
                                    const int64_t *slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int num_blocks,
                                    void *k_cache, void *v_cache, int kv_dtype, float k_scale,
                                    float v_scale, const float *k_head_scale,
                                    const float *v_head_scale, int32_t *status,
                                    cudaStream_t stream)
{
    if (num_tokens <= 0)
        return PKV_OK;
    const int n = num_kv_heads * head_dim;
    const int threads = n >= 256 ? 256 : ((n + 31) / 32) * 32;
    reshape_and_cache_kernel<<<num_tokens, threads, 0, stream>>>(
        k, v, in_dtype, slot_mapping, num_kv_heads, head_dim, num_blocks, k_cache, v_cache,
        kv_dtype, k_scale, v_scale, k_head_scale, v_head_scale, status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Copy-on-write page copies ("Inference optimization" lesson, section
// "PagedAttention": a request that diverges from a shared prompt gets its own
// copy of the shared page).  pairs[i] = (src, dst) block ids; the whole block
// of K and of V (every KV head's [D x 16] tile, `block_bytes` each) is copied
// with 16-byte loads and stores.  Flattened grid: (pair, cache, chunk).
constexpr int kCopyThreads = 256;
constexpr int kCopyVecPerThread = 4;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(unsigned char *k_cache, unsigned char *v_cache, size_t block_bytes,
                       const int32_t *pairs, int num_blocks, int chunks, int32_t *status)
{
    const int chunk = blockIdx.x % chunks;
    const int which = (blockIdx.x / chunks) & 1;
    const int i = blockIdx.x / (2 * chunks);
    const int32_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
    if (src < 0 || dst < 0 || src >= num_blocks || dst >= num_blocks) {
        if (threadIdx.x == 0 && chunk == 0 && which == 0)
            set_status(status, PKV_ERR_OUT_OF_RANGE);
        return;
    }
    unsigned char *base = which ? v_cache : k_cache;
    const uint4 *s = reinterpret_cast<const uint4 *>(base + static_cast<size_t>(src) * block_bytes);
    uint4 *d = reinterpret_cast<uint4 *>(base + static_cast<size_t>(dst) * block_bytes);
    const size_t n16 = block_bytes / 16;
    const size_t per_chunk = static_cast<size_t>(kCopyThreads) * kCopyVecPerThread;
    const size_t lo = static_cast<size_t>(chunk) * per_chunk;
    uint4 v[kCopyVecPerThread];
#pragma unroll
    for (int j = 0; j < kCopyVecPerThread; ++j) {
        const size_t e = lo + static_cast<size_t>(j) * kCopyThreads + threadIdx.x;
        if (e < n16)
            v[j] = __ldcs(s + e);
    }
#pragma unroll
    for (int j = 0; j < kCopyVecPerThread; ++j) {
        const size_t e = lo + static_cast<size_t>(j) * kCopyThreads + threadIdx.x;
        if (e < n16)
            d[e] = v[j];
    }
}

pkv_status launch_copy_blocks(void *k_cache, void *v_cache, size_t block_bytes,
                              const int32_t *pairs, int num_pairs, int num_blocks,
                              int32_t *status, cudaStream_t stream)
{
    if (num_pairs <= 0)
        return PKV_OK;
    const size_t per_chunk = static_cast<size_t>(kCopyThreads) * kCopyVecPerThread;
    const size_t n16 = block_bytes / 16;
    const long chunks = static_cast<long>((n16 + per_chunk - 1) / per_chunk);
    const long grid = static_cast<long>(num_pairs) * 2 * chunks;
    if (grid > 0x7fffffffL)
        return PKV_ERR_INVALID_ARG;
    copy_blocks_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, stream>>>(
        static_cast<unsigned char *>(k_cache), static_cast<unsigned char *>(v_cache),
        block_bytes, pairs, num_blocks, static_cast<int>(chunks), status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
