/*
 * pkv.h - C ABI of the GB300 (sm_103a) paged KV-cache decode library.
 *
 * The operations, all from the pages' statement of the problem:
 *
 *  - pkv_paged_attn_decode: PagedAttention decode ("vLLM e PagedAttention:
 *    serving high-throughput", simplified PagedAttention CUDA-kernel
 *    pseudocode).  For every sequence s and query head h the kernel walks the
 *    sequence's logical blocks, looks up each block's physical id in
 *    block_tables[s], reads that block's K and V tile, and folds the scores
 *    into an online (running max / running sum) softmax; the result is
 *    softmax(scale * q K^T) V over the first seq_lens[s] logical rows, i.e.
 *    the dense single-query attention of the "Inference optimization" lesson
 *    (Step 2, scaled_dot_product_attention) on the gathered rows.
 *    Variants: with the cache write fused in (pkv_paged_attn_decode_append),
 *    several layers in one launch (pkv_paged_attn_decode_layers), with
 *    per-KV-head scales of quantised caches
 *    (pkv_paged_attn_decode_head_scaled), without a caller workspace
 *    (pkv_paged_attn_decode_noalloc).
 *
 *  - pkv_paged_attn_prefill: the same attention for several causal query
 *    tokens per sequence (chunked prefill, speculative verification).
 *
 *  - pkv_reshape_and_cache (and _head_scaled): the KV-cache update
 *    ("Inference optimization" lesson, section "Caches de KV": only the new
 *    token's K and V are computed and appended; section "PagedAttention":
 *    fixed-size pages anywhere in GPU memory, mapped by a per-request table).
 *    Each new token's K/V row is written into its slot of the paged pool.
 *
 *  - pkv_bm_* and pkv_copy_blocks: the page pool's bookkeeping on the host
 *    (per-sequence page tables, shared pages stored once, copy-on-write) and
 *    the page copies it asks for.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless a
 *    comment says "host".  The library allocates no device memory and keeps
 *    no device state between calls; scratch space is the caller's
 *    `workspace` (pkv_paged_attn_decode_noalloc uses one fixed array instead;
 *    the block manager keeps its tables in host memory).
 *  - All tensors are dense, row-major, with the shapes given below, and every
 *    device pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls only enqueue work on it; none synchronises, except
 *    pkv_read_status which copies a status word to the host.
 *  - Argument errors are returned before anything is enqueued.  Problems only
 *    the device can see (a block id or slot outside the pool, a seq_len
 *    longer than its table, a wait that timed out) are never trapped: the
 *    kernels skip the offending access, record a pkv_status in the status
 *    word, and carry on; pkv_read_status returns it.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or count      */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype, head_dim, ...) */
    PKV_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed             */
    PKV_ERR_OUT_OF_RANGE = 4,  /* device side: block id / slot / seq_len invalid   */
    PKV_ERR_TIMEOUT = 5,       /* device side: a bounded wait gave up              */
    PKV_ERR_WORKSPACE = 6,     /* workspace missing or smaller than required       */
    PKV_ERR_NO_BLOCKS = 7      /* block manager: the pool (or host memory) ran out */
} pkv_status;

typedef enum {
    PKV_F32 = 0,       /* IEEE binary32                                   */
    PKV_BF16 = 1,      /* bfloat16                                        */
    PKV_FP8_E5M2 = 2,  /* OCP fp8 E5M2 (KV cache only), value = code * scale */
    PKV_FP8_E4M3 = 3,  /* OCP fp8 E4M3, finite form: no infinities, +-448 max,
                          the all-ones code is NaN (KV cache only), value = code * scale.
                          The tensor-core decode reads a NaN code in a valid slot
                          as 480 (the cache write never stores one for finite
                          inputs). */
    PKV_INT4 = 4       /* signed 4-bit integers -8..7 (KV cache only), value =
                          code * scale; two tokens per byte: a cache is
                          [num_blocks, num_kv_heads, head_dim, block_size / 2]
                          bytes, token 2j of a row in the low nibble of byte j,
                          token 2j+1 in the high nibble. */
} pkv_dtype;

/* Flags of pkv_paged_attn_decode. */
#define PKV_FLAG_IMPL_AUTO 0x0      /* tensor-core path when it applies, else CUDA cores */
#define PKV_FLAG_IMPL_SIMT 0x1      /* force the CUDA-core (FFMA) kernel                 */
#define PKV_FLAG_IMPL_MMA  0x2      /* force the tensor-core (mma.sync) kernel           */
#define PKV_FLAG_IMPL_TC   0x3      /* pkv_paged_attn_prefill only: the tcgen05 kernel   */
#define PKV_FLAG_IMPL_MASK 0x3
/* Split sequences are merged by the decode kernel itself (the CTA finishing a
 * sequence's last partition merges it).  This flag merges them in a second
 * log-sum-exp kernel instead; the results are identical. */
#define PKV_FLAG_SEPARATE_MERGE 0x4
/* Test hook for the failure path: the first page copy of the first work item
 * is never issued, so its bounded wait runs out and the call records
 * PKV_ERR_TIMEOUT (after about one second) instead of hanging.  Output rows
 * are then undefined. */
#define PKV_FLAG_TEST_DROP_FIRST_COPY 0x100

/*
 * Workspace bytes pkv_paged_attn_decode needs for these sizes (always >= 256:
 * the first 256 bytes hold the status word and a work counter).
 *   partition_tokens:
 *     0  = automatic: with at least 608 (sequence, KV head) units, one pass
 *          per unit when max_seq_len <= 2048, else 4096-token partitions
 *          (full partitions first, then the remainders, largest first);
 *          with fewer units, the stream-K schedule (PKV_SCHEDULE_STREAMK):
 *          the flattened (sequence, KV head, page) space is cut into one
 *          equal contiguous range per CTA, and sequences cut by range
 *          boundaries are merged with log-sum-exp weights by the CTA that
 *          finishes their last piece (workspace independent of the lengths).
 *    -2  = (PKV_SCHEDULE_STREAMK) the stream-K schedule, whatever the sizes.
 *    -1  = never split: one CTA per (sequence, KV head), one pass.
 *    > 0 = split every sequence into partitions of this many tokens (a
 *          multiple of block_size), scheduled dynamically, merged with
 *          log-sum-exp weights.
 * Returns 0 for invalid sizes.  Host only; touches no device.
 */
size_t pkv_paged_attn_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_seq_len,
                                     int partition_tokens);

/*
 * The schedule pkv_paged_attn_decode will use for these sizes: > 0 tokens per
 * fixed partition, 0 one pass per (sequence, KV head), PKV_SCHEDULE_STREAMK
 * for the stream-K schedule, -1 for invalid sizes.  Host only.
 */
#define PKV_SCHEDULE_STREAMK (-2)
int pkv_paged_attn_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_seq_len,
                                    int partition_tokens);

/*
 * Paged decode attention.
 *
 *   q            [num_seqs, num_q_heads, head_dim], q_dtype in {F32, BF16}
 *   k_cache,
 *   v_cache      [num_blocks, num_kv_heads, head_dim, block_size], kv_dtype in
 *                {F32, BF16, FP8_E5M2, FP8_E4M3, INT4}: tokens of a page are contiguous for
 *                each (head, dim), as in the pages' K_cache layout.
 *   k_scale,
 *   v_scale      dequant scales of fp8 and INT4 caches (value = code * scale);
 *                ignored for F32/BF16.
 *   block_tables int32 [num_seqs, max_blocks_per_seq]; entry j of row s is the
 *                physical block holding logical tokens [16j, 16j+16) of
 *                sequence s.  Entries past ceil(seq_lens[s]/block_size) are
 *                never read.  Rows may share blocks (shared prefixes).
 *   seq_lens     int32 [num_seqs]; 0 gives a zero output row.
 *   num_q_heads  a multiple of num_kv_heads; query head h uses KV head
 *                h / (num_q_heads / num_kv_heads).  At most 16 query heads
 *                per KV head.
 *   head_dim     64 or 128.   block_size: 16.
 *   max_seq_len  an upper bound of every seq_lens[s] (<= max_blocks_per_seq *
 *                block_size), used to size the launch and the workspace (no
 *                device-to-host copy of seq_lens).  A seq_lens[s] outside
 *                [0, max_seq_len] is clamped and reported as
 *                PKV_ERR_OUT_OF_RANGE in the status word.
 *   scale        multiplies q.k (e.g. 1/sqrt(head_dim)).
 *   out          [num_seqs, num_q_heads, head_dim], out_dtype in {F32, BF16}.
 *   workspace    >= pkv_paged_attn_workspace_size(...) bytes of device memory,
 *                256-byte aligned.  Its content on entry does not matter; it
 *                is overwritten.  Concurrent calls need separate workspaces.
 *   partition_tokens  as for pkv_paged_attn_workspace_size.
 *   flags        PKV_FLAG_IMPL_* and test hooks.
 *
 * The status word in the workspace is cleared at the start of the call.
 * Returns PKV_OK when the work was enqueued.
 */
pkv_status pkv_paged_attn_decode(const void *q, pkv_dtype q_dtype,
                                 const void *k_cache, const void *v_cache, pkv_dtype kv_dtype,
                                 float k_scale, float v_scale,
                                 const int32_t *block_tables, const int32_t *seq_lens,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, int max_blocks_per_seq,
                                 int max_seq_len, float scale,
                                 void *out, pkv_dtype out_dtype,
                                 void *workspace, size_t workspace_bytes,
                                 int partition_tokens, int flags, void *stream);

/*
 * One decode step with the cache write fused in: for every sequence s with
 * seq_lens[s] > 0, its new token is logical position seq_lens[s] - 1; its
 * K/V rows new_k[s], new_v[s] ([num_seqs, num_kv_heads, head_dim] of
 * new_dtype, F32 or BF16) are converted and written into that position's
 * slot of k_cache / v_cache (block block_tables[s][(L-1)/16], offset
 * (L-1)%16), and the attention over the seq_lens[s] tokens includes them.
 * Bit-identical to pkv_reshape_and_cache of those slots followed by
 * pkv_paged_attn_decode, in one launch ("Inference optimization" lesson,
 * section "Caches de KV": compute K, V only for the new token, append, attend).
 * The block holding position L-1 must not be shared with another sequence.
 * Other arguments, errors and the workspace as for pkv_paged_attn_decode.
 */
pkv_status pkv_paged_attn_decode_append(const void *q, pkv_dtype q_dtype, const void *new_k,
                                        const void *new_v, pkv_dtype new_dtype, void *k_cache,
                                        void *v_cache, pkv_dtype kv_dtype, float k_scale,
                                        float v_scale, const int32_t *block_tables,
                                        const int32_t *seq_lens, int num_seqs, int num_q_heads,
                                        int num_kv_heads, int head_dim, int block_size,
                                        int num_blocks, int max_blocks_per_seq, int max_seq_len,
                                        float scale, void *out, pkv_dtype out_dtype,
                                        void *workspace, size_t workspace_bytes,
                                        int partition_tokens, int flags, void *stream);

/*
 * Several decode layers in one launch.  A decoder stack repeats the same
 * attention in every layer over the same sequences: the block tables and
 * lengths are shared, while each layer has its own caches, query, new rows
 * and output ("Inference optimization" lesson, section "Caches de KV": the
 * cache holds K and V of every layer, 2 * layers * KV heads * head_dim *
 * bytes per token).  Decode is bound by memory reads
 * (section "O framework de operacoes:byte"), so on small layers (a chat
 * batch of short sequences) the fixed cost of each launch -- grid fill and
 * drain -- is a large share of the time; this entry point runs the decode of
 * num_layers layers as one persistent grid, the work of all layers
 * scheduled together, with the fused cache write of
 * pkv_paged_attn_decode_append in every layer that has new rows.
 *
 *   layers       DEVICE array of num_layers pkv_layer entries (8-byte
 *                aligned), read by the kernels.  Per layer:
 *                  q        [num_seqs, num_q_heads, head_dim] of q_dtype
 *                  new_k,
 *                  new_v    [num_seqs, num_kv_heads, head_dim] of new_dtype
 *                           (F32 or BF16), or both NULL: no cache write in
 *                           that layer (then seq_lens[s] counts only cached
 *                           tokens, as for pkv_paged_attn_decode)
 *                  k_cache,
 *                  v_cache  [num_blocks, num_kv_heads, head_dim, block_size]
 *                           of kv_dtype
 *                  out      [num_seqs, num_q_heads, head_dim] of out_dtype
 *                Every pointer must be 16-byte aligned device memory.  An
 *                entry with a null or misaligned tensor is skipped (nothing
 *                is read through it or written to it) and reported as
 *                PKV_ERR_INVALID_ARG in the status word.
 *   block_tables, seq_lens, sizes, scales, scale: shared by every layer, as
 *                for pkv_paged_attn_decode_append.
 *   workspace    >= pkv_paged_attn_layers_workspace_size(num_layers, ...)
 *                bytes, 256-byte aligned.
 * Every layer's result is bit-identical to pkv_paged_attn_decode_append (or
 * pkv_paged_attn_decode for a layer without new rows) of that layer alone
 * with the partition size this call uses (pkv_paged_attn_layers_partition_
 * tokens; the automatic choice counts the (layer, sequence, KV head) units).
 * Other arguments and errors as for pkv_paged_attn_decode.
 */
typedef struct pkv_layer {
    const void *q;
    const void *new_k;
    const void *new_v;
    void *k_cache;
    void *v_cache;
    void *out;
} pkv_layer;
size_t pkv_paged_attn_layers_workspace_size(int num_layers, int num_seqs, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int max_seq_len, int partition_tokens);
int pkv_paged_attn_layers_partition_tokens(int num_layers, int num_seqs, int num_q_heads,
                                           int num_kv_heads, int head_dim, int block_size,
                                           int max_seq_len, int partition_tokens);
pkv_status pkv_paged_attn_decode_layers(const pkv_layer *layers, int num_layers,
                                        pkv_dtype q_dtype, pkv_dtype new_dtype,
                                        pkv_dtype kv_dtype, float k_scale, float v_scale,
                                        const int32_t *block_tables, const int32_t *seq_lens,
                                        int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int num_blocks,
                                        int max_blocks_per_seq, int max_seq_len, float scale,
                                        pkv_dtype out_dtype, void *workspace,
                                        size_t workspace_bytes, int partition_tokens, int flags,
                                        void *stream);

/*
 * Decode over an fp8 or INT4 cache quantised with one scale per
 * KV head: element (block, h, d, t) stands for code * k_head_scales[h] (K) and
 * code * v_head_scales[h] (V).  k_head_scales, v_head_scales: float32
 * [num_kv_heads] in device memory, non-zero and finite.  Everything else as
 * for pkv_paged_attn_decode (whose scalar k_scale / v_scale are the special
 * case of equal factors).  Other KV dtypes: PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_paged_attn_decode_head_scaled(
    const void *q, pkv_dtype q_dtype, const void *k_cache, const void *v_cache, pkv_dtype kv_dtype,
    const float *k_head_scales, const float *v_head_scales, const int32_t *block_tables,
    const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int block_size, int num_blocks, int max_blocks_per_seq, int max_seq_len, float scale,
    void *out, pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
    int partition_tokens, int flags, void *stream);

/*
 * Paged attention of several query tokens per sequence: chunked prefill
 * ("vLLM e PagedAttention: serving high-throughput", the
 * --enable-chunked-prefill flag) and speculative verification of draft
 * tokens ("Inference optimization" lesson, section on speculative decoding).
 * The queries of sequence s are rows q_start[s] .. q_start[s+1]-1 of q; with
 * n_s of them and L_s = seq_lens[s] cached tokens they are the sequence's last
 * n_s positions (their K/V already written, e.g. by pkv_reshape_and_cache),
 * and query i attends the rows t <= L_s - n_s + i: the causal mask of the
 * lesson's Step 2 scaled_dot_product_attention (triu of offset
 * seq_len_k - seq_len_q + 1).  For every row of q and query head h:
 *   out[row, h, :] = sum_{t <= pos} softmax_t(scale * q[row, h, :] . k_t) v_t
 * with k_t, v_t read through the block table as in pkv_paged_attn_decode and
 * KV head h / (num_q_heads / num_kv_heads).  n_s = 1 for every s is decode.
 *
 *   q            [num_tokens, num_q_heads, head_dim] BF16 (device).
 *   q_start      int32 [num_seqs + 1] (device), non-decreasing, q_start[0] = 0,
 *                q_start[num_seqs] = num_tokens.
 *   k_cache,
 *   v_cache      [num_blocks, num_kv_heads, head_dim, 16] of kv_dtype (device):
 *                BF16, FP8_E5M2, FP8_E4M3 or INT4 (layouts as for
 *                pkv_paged_attn_decode).
 *   k_scale,
 *   v_scale      dequant scales of fp8 / INT4 caches (value = code * scale),
 *                finite and non-zero; ignored for BF16.
 *   block_tables, seq_lens   as for pkv_paged_attn_decode.
 *   max_q_len    host bound on every n_s; max_seq_len bound on every L_s.
 *   out          [num_tokens, num_q_heads, head_dim], F32 or BF16 (device).
 *   workspace    >= pkv_paged_attn_prefill_workspace_size(...) bytes of
 *                device memory, 256-byte aligned; word 0 is the status word
 *                read by pkv_read_status.
 *   partition_tokens   0 automatic, -1 never split a context, > 0 (multiple
 *                of 16) split every context into partitions of that many
 *                tokens merged with log-sum-exp weights.
 *   flags        PKV_FLAG_IMPL_AUTO (bf16 caches: the tcgen05 kernel; fp8 and
 *                INT4 caches: the mma.sync kernel, whose fragments widen the
 *                codes to f16 in registers as decode does), PKV_FLAG_IMPL_TC
 *                (bf16 only; PKV_ERR_UNSUPPORTED otherwise) or
 *                PKV_FLAG_IMPL_MMA, optionally PKV_FLAG_TEST_DROP_FIRST_COPY.
 * head_dim 64 or 128, up to 16 query heads per KV head.  Errors as for
 * pkv_paged_attn_decode; on the device a sequence with n_s > L_s, n_s >
 * max_q_len, or q_start outside [0, num_tokens] is reported as
 * PKV_ERR_OUT_OF_RANGE and its rows are not written.
 */
size_t pkv_paged_attn_prefill_workspace_size(int num_seqs, int num_tokens, int num_q_heads,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int max_q_len, int max_seq_len,
                                             int partition_tokens);
/* The partition the call will use: 0 = none, > 0 tokens per partition,
 * -1 invalid arguments. */
int pkv_paged_attn_prefill_partition_tokens(int num_seqs, int num_tokens, int num_q_heads,
                                            int num_kv_heads, int head_dim, int block_size,
                                            int max_q_len, int max_seq_len,
                                            int partition_tokens);
pkv_status pkv_paged_attn_prefill(const void *q, pkv_dtype q_dtype, const int32_t *q_start,
                                  const void *k_cache, const void *v_cache, pkv_dtype kv_dtype,
                                  float k_scale, float v_scale, const int32_t *block_tables,
                                  const int32_t *seq_lens, int num_seqs, int num_tokens,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int num_blocks, int max_blocks_per_seq,
                                  int max_q_len, int max_seq_len, float scale, void *out,
                                  pkv_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                  int partition_tokens, int flags, void *stream);

/*
 * Decode without a caller workspace (the pages have no counterpart; this is
 * an interface for callers that cannot allocate device memory, e.g. a plugin
 * inside a runtime that owns all device memory, or a loop where cudaMalloc's
 * implicit synchronisation is not allowed).
 *
 * Same arguments and result as pkv_paged_attn_decode, minus the workspace.
 * The scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES inside this
 * library; every GPU that loads the library keeps it allocated until the
 * process exits.  The call allocates nothing and never calls cudaMalloc or
 * cudaFree.
 *  - Sizes whose pkv_paged_attn_workspace_size(...) exceeds
 *    PKV_NOALLOC_SCRATCH_BYTES are rejected with PKV_ERR_WORKSPACE before
 *    anything is enqueued (pass a larger partition_tokens, or -1, to need less).
 *  - The first call in each CUDA context (the device's primary context, or
 *    a context the caller made current) looks up the array's device address
 *    with cudaGetSymbolAddress and remembers it for that context only, since
 *    each context holds its own copy of the array; make that first call
 *    before any stream capture.
 *  - All calls share the one array and it keeps the previous call's contents
 *    (each call clears the parts that must start at zero).  Calls that can
 *    overlap on the GPU (different streams, no ordering between them) race on
 *    it: serialise them.
 *  - The device status word sits in that shared array and is not readable by
 *    the caller; use pkv_paged_attn_decode with a workspace to see it.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
pkv_status pkv_paged_attn_decode_noalloc(const void *q, pkv_dtype q_dtype,
                                         const void *k_cache, const void *v_cache,
                                         pkv_dtype kv_dtype, float k_scale, float v_scale,
                                         const int32_t *block_tables, const int32_t *seq_lens,
                                         int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int block_size, int num_blocks,
                                         int max_blocks_per_seq, int max_seq_len, float scale,
                                         void *out, pkv_dtype out_dtype, int partition_tokens,
                                         int flags, void *stream);

/*
 * Paged cache write: for every token i < num_tokens with
 * slot = slot_mapping[i] >= 0, writes
 *   k_cache[slot / block_size, h, d, slot % block_size] = cvt(k[i, h, d])
 * (and the same for v) for all h < num_kv_heads, d < head_dim.
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim], in_dtype in {F32, BF16}
 *   slot_mapping  int64 [num_tokens]; negative = padding token, skipped.
 *                 Non-negative slots must be distinct (duplicates race).
 *   k_cache,
 *   v_cache       [num_blocks, num_kv_heads, head_dim, block_size] of kv_dtype.
 *   cvt           F32 -> F32 and BF16 -> BF16 copy the bits; F32 -> BF16 rounds
 *                 to nearest even; BF16 -> F32 widens exactly; -> FP8_E5M2 / FP8_E4M3
 *                 stores round-to-nearest-even(x / scale) computed in float32
 *                 and saturated to +-57344 (e5m2) / +-448 (e4m3); -> INT4 the same
 *                 rounding clamped to -8..7.  NaN inputs give a NaN code of
 *                 unspecified payload (INT4: 0).
 *   status        optional device int32 (NULL = none): set to
 *                 PKV_ERR_OUT_OF_RANGE if a slot lies past the pool (that
 *                 token is skipped).  It is never cleared by this call.
 */
pkv_status pkv_reshape_and_cache(const void *k, const void *v, pkv_dtype in_dtype,
                                 const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks,
                                 void *k_cache, void *v_cache, pkv_dtype kv_dtype,
                                 float k_scale, float v_scale, int32_t *status, void *stream);

/*
 * The cache write of pkv_reshape_and_cache for an fp8 or INT4 cache quantised with one
 * scale per KV head: head h's codes are RNE_satfinite(x / k_head_scales[h])
 * (V likewise), the division done in float32.  k_head_scales, v_head_scales:
 * float32 [num_kv_heads] in device memory.  Other KV dtypes:
 * PKV_ERR_UNSUPPORTED.
 */
pkv_status pkv_reshape_and_cache_head_scaled(const void *k, const void *v, pkv_dtype in_dtype,
                                             const int64_t *slot_mapping, int num_tokens,
                                             int num_kv_heads, int head_dim, int block_size,
                                             int num_blocks, void *k_cache, void *v_cache,
                                             pkv_dtype kv_dtype, const float *k_head_scales,
                                             const float *v_head_scales, int32_t *status,
                                             void *stream);

/*
 * Copy-on-write page copies ("Inference optimization" lesson, section
 * "PagedAttention": pages of a shared prompt are stored once; a request that
 * diverges gets its own copy).  For every i < num_pairs, with
 * (src, dst) = (pairs[2i], pairs[2i+1]) (int32, device memory), block dst of
 * k_cache and of v_cache becomes a copy of block src: all num_kv_heads x
 * head_dim x block_size elements, copied bit for bit.  Pairs whose src or dst
 * lies outside [0, num_blocks) are skipped and reported in *status
 * (optional device int32, as for pkv_reshape_and_cache).  A dst must not be
 * the src or dst of another pair of the same call (no chains).  The pairs
 * come from pkv_bm_append.
 */
pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, pkv_dtype kv_dtype, int num_kv_heads,
                           int head_dim, int block_size, int num_blocks, const int32_t *pairs,
                           int num_pairs, int32_t *status, void *stream);

/*
 * Host-side block manager (no GPU calls; thread-safe).  It keeps the page
 * pool of one cache: a free list, a reference count per page and one page
 * table per sequence ("Inference optimization" lesson, section
 * "PagedAttention"; "Continuous Batching e PagedAttention no vLLM", section 3:
 * logical blocks of a sequence map to physical pages anywhere in the pool,
 * the last page may be partly filled, shared pages are stored once).
 * Token t of a sequence lives at slot table[t / block_size] * block_size +
 * t % block_size.  The lowest free page id is always taken first.  Every call
 * either succeeds completely or leaves the manager unchanged.
 *
 *   pkv_bm_create    a pool of num_blocks pages; *out receives the handle
 *                    (release with pkv_bm_destroy).
 *   pkv_bm_add       a new sequence seq_id holding num_tokens tokens (a
 *                    prompt): ceil(num_tokens / block_size) fresh pages;
 *                    slots (optional, [num_tokens]) receives each token's slot.
 *   pkv_bm_fork      child_id starts as parent_id, sharing every page (the
 *                    reference counts go up; nothing is copied).
 *   pkv_bm_append    reserves the next token of each of the n listed
 *                    sequences (distinct ids), in list order: a fresh page
 *                    when the last page is full; when the last page is
 *                    shared, a fresh page plus a (src, dst) copy appended to
 *                    copy_pairs ([n][2], *num_copies of them filled).
 *                    slots[i] receives the new token's slot.  Copy the pairs
 *                    (pkv_copy_blocks) before writing the tokens
 *                    (pkv_reshape_and_cache).
 *   pkv_bm_free      releases a sequence; pages no longer referenced return
 *                    to the pool.
 *   pkv_bm_tables    dense block tables [n][max_blocks_per_seq] (-1 padded)
 *                    and lengths of the listed sequences, for attention.
 *   pkv_bm_num_free, pkv_bm_ref_count   inspection (-1 on bad arguments).
 * Errors: PKV_ERR_INVALID_ARG (unknown or duplicate id, a sequence longer
 * than max_blocks_per_seq pages, null pointers), PKV_ERR_NO_BLOCKS (not
 * enough free pages for the whole call).
 */
typedef struct pkv_block_manager pkv_block_manager;
pkv_status pkv_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                         pkv_block_manager **out);
void pkv_bm_destroy(pkv_block_manager *bm);
pkv_status pkv_bm_add(pkv_block_manager *bm, int seq_id, int num_tokens, int64_t *slots);
pkv_status pkv_bm_fork(pkv_block_manager *bm, int parent_id, int child_id);
pkv_status pkv_bm_append(pkv_block_manager *bm, const int32_t *seq_ids, int n, int64_t *slots,
                         int32_t *copy_pairs, int *num_copies);
pkv_status pkv_bm_free(pkv_block_manager *bm, int seq_id);
pkv_status pkv_bm_tables(pkv_block_manager *bm, const int32_t *seq_ids, int n,
                         int max_blocks_per_seq, int32_t *tables, int32_t *seq_lens);
int pkv_bm_num_free(pkv_block_manager *bm);
int pkv_bm_ref_count(pkv_block_manager *bm, int block);

/*
 * Waits for `stream`, then copies the status word of a decode workspace to
 * *host_status (a pkv_status value); clear != 0 also resets it to PKV_OK.
 */
pkv_status pkv_read_status(void *workspace, int clear, int32_t *host_status, void *stream);

/* A static string naming a status code. */
const char *pkv_status_string(pkv_status status);

/* Library version as 10000*major + 100*minor + patch. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
