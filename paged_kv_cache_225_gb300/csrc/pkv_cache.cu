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
                             float k_scale, float v_scale, int32_t *status)
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
        store_kv(k_cache, kv_dtype, dst, k, in_dtype, src, k_scale);
        store_kv(v_cache, kv_dtype, dst, v, in_dtype, src, v_scale);
    }
}

pkv_status launch_reshape_and_cache(const void *k, const void *v, int in_dtype,
                                    const int64_t *slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int num_blocks,
                                    void *k_cache, void *v_cache, int kv_dtype, float k_scale,
                                    float v_scale, int32_t *status, cudaStream_t stream)
{
    if (num_tokens <= 0)
        return PKV_OK;
    const int n = num_kv_heads * head_dim;
    const int threads = n >= 256 ? 256 : ((n + 31) / 32) * 32;
    reshape_and_cache_kernel<<<num_tokens, threads, 0, stream>>>(
        k, v, in_dtype, slot_mapping, num_kv_heads, head_dim, num_blocks, k_cache, v_cache,
        kv_dtype, k_scale, v_scale, status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
