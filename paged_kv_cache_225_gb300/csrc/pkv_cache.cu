// Paged KV-cache write ("reshape_and_cache").
//
// The "Inference optimization" lesson (section "Caches de KV") computes K and
// V only for the new token and appends them to the cache; with paging
// (section "PagedAttention") the append lands in a 16-token page anywhere in
// the pool.  Token i goes to slot = slot_mapping[i] = block * 16 + offset of
// every KV head; element (h, d) is stored at [block, h, d, offset].
#include "pkv_convert.cuh"

namespace pkv {

// A CTA takes 32 consecutive new tokens and 64 of their (head, dim)
// elements.  The rows are read coalesced (elements on the lanes) into a
// shared-memory tile of the raw input words; then, tokens on the lanes, one
// warp store writes element e of the 32 tokens: tokens in consecutive slots
// of a page land in consecutive cells of that page's [head_dim][16] row, so
// the store covers one or two 32-byte sectors where a token at a time wrote
// a partial sector per element.  Tile rows are padded to 65 words, so the
// token-strided reads hit distinct banks.
constexpr int kCacheTokens = 32;
constexpr int kCacheElems = 64;
constexpr int kTileWords = kCacheElems + 1;  // one tile row, in 32-bit words

__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const void *k, const void *v, int in_dtype,
                             const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                             int head_dim, int num_blocks, void *k_cache, void *v_cache,
                             int kv_dtype, float k_scale, float v_scale,
                             const float *k_head_scale, const float *v_head_scale,
                             int32_t *status)
{
    __shared__ uint32_t tk[kCacheTokens * kTileWords], tv[kCacheTokens * kTileWords];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int n = num_kv_heads * head_dim;
    const int t0 = blockIdx.x * kCacheTokens;
    const int e0 = blockIdx.y * kCacheElems;
    const int ne = min(kCacheElems, n - e0);
    // Raw words: element c of tile row r at word r * kTileWords + c (f32) or
    // half-word 2 r * kTileWords + c (bf16).
    const bool f32 = in_dtype == PKV_F32;
    const int rs = f32 ? kTileWords : 2 * kTileWords;  // row stride in elements
    for (int r = warp; r < kCacheTokens && t0 + r < num_tokens; r += 8) {
        const size_t row = static_cast<size_t>(t0 + r) * n + e0;
        for (int c = lane; c < ne; c += 32) {
            if (f32) {
                reinterpret_cast<float *>(tk)[r * rs + c] = static_cast<const float *>(k)[row + c];
                reinterpret_cast<float *>(tv)[r * rs + c] = static_cast<const float *>(v)[row + c];
            } else {
                reinterpret_cast<unsigned short *>(tk)[r * rs + c] =
                    static_cast<const unsigned short *>(k)[row + c];
                reinterpret_cast<unsigned short *>(tv)[r * rs + c] =
                    static_cast<const unsigned short *>(v)[row + c];
            }
        }
    }
    __syncthreads();
    const int i = t0 + lane;
    if (i >= num_tokens)
        return;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0)
        return;  // no slot: skipped
    const int64_t blk = slot / kBlockSize;
    const int off = static_cast<int>(slot - blk * kBlockSize);
    if (blk >= num_blocks) {
        if (blockIdx.y == 0 && warp == 0)
            set_status(status, PKV_ERR_OUT_OF_RANGE);
        return;
    }
    for (int c = warp; c < ne; c += 8) {
        const int e = e0 + c;
        const size_t dst = (static_cast<size_t>(blk) * n + e) * kBlockSize + off;
        const int h = e / head_dim;
        const float ks = k_head_scale ? k_scale * __ldg(k_head_scale + h) : k_scale;
        const float vs = v_head_scale ? v_scale * __ldg(v_head_scale + h) : v_scale;
        const size_t j = static_cast<size_t>(lane) * rs + c;
        store_kv(k_cache, kv_dtype, dst, tk, in_dtype, j, ks);
        store_kv(v_cache, kv_dtype, dst, tv, in_dtype, j, vs);
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
    const long n = static_cast<long>(num_kv_heads) * head_dim;
    const long gx = (static_cast<long>(num_tokens) + kCacheTokens - 1) / kCacheTokens;
    const long gy = (n + kCacheElems - 1) / kCacheElems;
    if (gy > 65535)
        return PKV_ERR_UNSUPPORTED;
    reshape_and_cache_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), 256,
                               0, stream>>>(k, v, in_dtype, slot_mapping, num_tokens,
                                            num_kv_heads, head_dim, num_blocks, k_cache, v_cache,
                                            kv_dtype, k_scale, v_scale, k_head_scale,
                                            v_head_scale, status);
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
