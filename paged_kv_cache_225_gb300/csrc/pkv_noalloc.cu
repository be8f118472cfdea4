// Decode entry point for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin running
// inside a host runtime that owns all device memory and exposes no allocator,
// or a latency-critical loop where cudaMalloc (which can synchronise the
// device) is not allowed once serving has started.  For them,
// pkv_paged_attn_decode_noalloc runs the same decode with its scratch taken
// from a fixed array compiled into this library instead of a caller buffer.
//
// The array is a file-scope __device__ variable, so every GPU on which the
// library's module is loaded holds PKV_NOALLOC_SCRATCH_BYTES of it until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it is only a stand-in symbol), so the entry point looks the
// address up with cudaGetSymbolAddress, with the caller's device current, and
// passes it on like any workspace pointer.  The address belongs to the CUDA
// context the module was loaded into: a plugin that pushes its own context on
// a device, or a caller that resets the device between calls, gets a new copy
// of the array at a new address.  The lookup is therefore remembered per
// context (keyed on the driver's unique context id), never per device ordinal.
#include <mutex>

#include "pkv_internal.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kSlots = 32;
std::mutex g_scratch_mu;
uint64_t g_scratch_ctx[kSlots];  // context id of each remembered address (0 = empty)
void *g_scratch_addr[kSlots];    // device address of g_noalloc_scratch in that context
int g_scratch_next = 0;

// Device address of the scratch array in the current context (looked up the
// first time this context calls).
pkv_status scratch_in_current_context(void **addr)
{
    const uint64_t ctx = pkv::current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (ctx != 0)
        for (int i = 0; i < kSlots; ++i)
            if (g_scratch_ctx[i] == ctx) {
                *addr = g_scratch_addr[i];
                return PKV_OK;
            }
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess || p == nullptr)
        return PKV_ERR_CUDA;
    // The lookup itself may have made the device's primary context current.
    const uint64_t now = ctx != 0 ? ctx : pkv::current_context_id();
    if (now != 0) {
        g_scratch_ctx[g_scratch_next] = now;
        g_scratch_addr[g_scratch_next] = p;
        g_scratch_next = (g_scratch_next + 1) % kSlots;
    }
    *addr = p;
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_attn_decode_noalloc(
    const void *q, pkv_dtype q_dtype, const void *k_cache, const void *v_cache,
    pkv_dtype kv_dtype, float k_scale, float v_scale, const int32_t *block_tables,
    const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_seq_len, float scale,
    void *out, pkv_dtype out_dtype, int partition_tokens, int flags, void *stream)
{
    const size_t need = pkv_paged_attn_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                      head_dim, block_size, max_seq_len,
                                                      partition_tokens);
    if (need == 0)
        return PKV_ERR_INVALID_ARG;
    if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES))
        return PKV_ERR_WORKSPACE;  // these sizes need more scratch than the fixed array
    void *scratch = nullptr;
    const pkv_status rc = scratch_in_current_context(&scratch);
    if (rc != PKV_OK)
        return rc;
    return pkv_paged_attn_decode(q, q_dtype, k_cache, v_cache, kv_dtype, k_scale, v_scale,
                                 block_tables, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                                 head_dim, block_size, num_blocks, max_blocks_per_seq,
                                 max_seq_len, scale, out, out_dtype, scratch,
                                 static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES), partition_tokens,
                                 flags, stream);
}
