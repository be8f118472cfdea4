// Internal interface between the C ABI (pkv_api.cu) and the kernel units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/pkv.h"

namespace pkv {

// The tensors of one decode layer (the layout of the public pkv_layer).
struct LayerPtrs {
    const void *q;      // [S, Hq, D]
    const void *new_k;  // [S, Hkv, D] rows of the fused cache write, or null
    const void *new_v;
    void *k_cache;      // [N, Hkv, D, 16]
    void *v_cache;
    void *out;          // [S, Hq, D]
};
static_assert(sizeof(LayerPtrs) == 6 * sizeof(void *), "pkv_layer layout");

// Everything a decode launch needs; passed by value as the kernel parameter.
// A launch covers num_layers layers that share the block tables and lengths:
// their tensors come from the device table `layers`, or from `one` when it is
// null (single-layer calls).  Work of layer l, sequence s is indexed as the
// global sequence l * S + s in the workspace (partials, arrival counters).
struct DecodeParams {
    LayerPtrs one;
    const LayerPtrs *layers;
    int num_layers;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *part_o;        // [L*S][Hq][max_parts][D] normalised partial outputs
    float *part_ml;       // [L*S][Hq][max_parts][2] (max of log2-scaled scores, sum)
    int *status;          // workspace word 0
    unsigned *counter;    // workspace word 1: next work item (split mode)
    unsigned *arrive;     // [L*S][Hkv] partials written so far (in-kernel merge)
    int q_dtype, out_dtype;
    int num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks;
    int max_len;          // caller's bound on seq_lens (<= max_blocks * 16)
    int group;            // query heads per KV head
    float score_scale;    // scale * log2(e) (* k_scale for fp8)
    float out_scale;      // v_scale for fp8, else 1
    int partition;        // tokens per work item (multiple of 16)
    int max_parts;        // partitions per sequence the workspace holds
    int split;            // 1: fixed partitions: persistent grid, work counter, partials
    int streamk;          // 1: stream-K schedule (equal page ranges per CTA)
    int streamk_max_ctas; // CTAs the stream-K partial slots are sized for
    int fused_merge;      // 1: the CTA finishing a sequence's last partial merges it
    int drop_first_copy;  // test hook: never issue the first copy of item 0
    // Fused cache write (layers whose new_k is null have none): the new token
    // of sequence s is its position seq_lens[s] - 1; its K/V rows [S][Hkv][D]
    // of new_dtype are converted to the cache dtype and written to the cache
    // and into the page tile the kernel is about to attend.  `append` is set
    // when any layer may carry new rows.
    int append;
    int new_dtype;
    int kv_dtype;
    float k_scale, v_scale;
    // Per-KV-head factors of fp8 caches ([num_kv_heads], device; null = 1):
    // a code of head h stands for code * k_scale * k_head_scale[h].
    const float *k_head_scale;
    const float *v_head_scale;
    // A several-queries call's one-query sequences served by the decode
    // kernels (null: plain decode): q_rows is its q_start [S + 1] over
    // num_rows rows of q and out; sequence s is attended only when it has
    // exactly one query, read from and written to row q_rows[s]; the others
    // count as empty and write nothing.
    const int32_t *q_rows;
    int num_rows;
};

// Paged attention of several query tokens per sequence (chunked prefill,
// speculative verification).  The queries of sequence s are rows
// q_start[s] .. q_start[s+1]-1 of q [T, Hq, D], its last n_s positions.
struct PrefillParams {
    const void *q;
    const int32_t *q_start;  // [S + 1]
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    void *out;               // [T, Hq, D]
    float *part_o;           // [T][Hq][max_parts][D] normalised partial outputs
    float *part_ml;          // [T][Hq][max_parts][2]
    int *status;             // workspace word 0
    unsigned *counter;       // workspace word 1: next work item
    int out_dtype;
    int num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks;
    int max_len;             // bound on seq_lens
    int max_q_len;           // bound on n_s
    int group;
    int kv_dtype;            // BF16, or an fp8 / INT4 cache (mma.sync kernel only)
    float score_scale;       // scale * log2(e) (* k_scale for fp8 / INT4 caches)
    float out_scale;         // v_scale for fp8 / INT4 caches, else 1
    int partition;           // tokens per partition (multiple of 16)
    int max_parts;           // 1: no split
    int drop_first_copy;     // test hook: never issue the first copy of item 0
    int impl;                // PKV_FLAG_IMPL_MMA (mma.sync) or PKV_FLAG_IMPL_TC (tcgen05)
    int skip_single;         // 1: one-query sequences are served by the decode kernels
};

constexpr int kBlockSize = 16;

// The 8-bit KV dtypes (value = code * scale).
constexpr bool is_fp8(int dtype) { return dtype == PKV_FP8_E5M2 || dtype == PKV_FP8_E4M3; }
// Every KV dtype whose stored codes are multiplied by a dequant scale.
constexpr bool is_scaled(int dtype) { return is_fp8(dtype) || dtype == PKV_INT4; }
// Bytes of one [head_dim x 16] page tile of a KV dtype.
constexpr int tile_bytes(int dtype, int head_dim)
{
    return dtype == PKV_F32 ? head_dim * 64
                            : dtype == PKV_BF16 ? head_dim * 32
                                                : dtype == PKV_INT4 ? head_dim * 8 : head_dim * 16;
}

// The tensor-core e4m3 policy widens a code to a binary16 holding 2^-8 times
// its value; the host multiplies the score and output scales by 2^8.
constexpr float kE4m3Shift = 256.0f;
constexpr size_t kWorkspaceHeader = 256;
constexpr int kStreamKMaxCtas = 1024;  // partial slots of the stream-K schedule

// Kernel-unit entry points.  Each launches on `stream` and returns a status
// (PKV_OK, PKV_ERR_UNSUPPORTED for a shape with no kernel, PKV_ERR_CUDA).
// `grid_items` is the number of CTAs to launch (0 = let the unit decide).
pkv_status launch_decode_simt(const DecodeParams &p, int kv_dtype, cudaStream_t stream);
pkv_status launch_decode_simt_fp8(const DecodeParams &p, int kv_dtype, cudaStream_t stream);
pkv_status launch_decode_mma(const DecodeParams &p, int kv_dtype, cudaStream_t stream);
pkv_status launch_merge(const DecodeParams &p, cudaStream_t stream);
bool mma_supports(int kv_dtype, int q_dtype, int head_dim, int group);
pkv_status launch_prefill(const PrefillParams &p, int kv_dtype, cudaStream_t stream);
// The tcgen05 form of the several-queries kernel (bf16, head_dim 64 / 128).
pkv_status launch_prefill_tc(const PrefillParams &p, cudaStream_t stream);

pkv_status launch_reshape_and_cache(const void *k, const void *v, int in_dtype,
                                    const int64_t *slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int num_blocks,
                                    void *k_cache, void *v_cache, int kv_dtype, float k_scale,
                                    float v_scale, const float *k_head_scale,
                                    const float *v_head_scale, int32_t *status,
                                    cudaStream_t stream);

pkv_status launch_copy_blocks(void *k_cache, void *v_cache, size_t block_bytes,
                              const int32_t *pairs, int num_pairs, int num_blocks,
                              int32_t *status, cudaStream_t stream);

int device_sm_count();

// A process-unique id of the CUDA context current on the calling thread (0 when
// there is none or the driver cannot tell).  Kernel attributes, module symbols
// and occupancy facts belong to a context, which a device reset or a second
// context on the same device replaces: caches of them are keyed on this id.
uint64_t current_context_id();

// One int per CUDA context, computed by make(&value) the first time a host
// thread asks with that context current (e.g. a kernel's resident CTAs per SM,
// after its shared-memory attribute is set).  Thread-safe; a few contexts are
// remembered at once, others are recomputed.
class ContextCache {
  public:
    template <class F> pkv_status get(int *value, F &&make)
    {
        const uint64_t ctx = current_context_id();
        if (ctx != 0) {
            std::lock_guard<std::mutex> lock(mu_);
            for (int i = 0; i < kSlots; ++i)
                if (id_[i] == ctx) {
                    *value = val_[i];
                    return PKV_OK;
                }
        }
        int v = 0;
        const pkv_status rc = make(&v);
        if (rc != PKV_OK)
            return rc;
        if (ctx != 0) {
            std::lock_guard<std::mutex> lock(mu_);
            id_[next_] = ctx;
            val_[next_] = v;
            next_ = (next_ + 1) % kSlots;
        }
        *value = v;
        return PKV_OK;
    }

  private:
    static constexpr int kSlots = 16;
    std::mutex mu_;
    uint64_t id_[kSlots] = {};
    int val_[kSlots] = {};
    int next_ = 0;
};

}  // namespace pkv
