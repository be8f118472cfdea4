// Device helpers shared by the decode kernel and the stand-alone merge kernel:
// sequence-length clamping, partition counts, output stores, and the
// log-sum-exp merge of split-sequence partials.
#pragma once

#include <cmath>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

// A length outside [0, max_len] is reported and clamped, so no item reads
// past the table or writes past the workspace's partial rows.
__device__ __forceinline__ int clamp_len(const DecodeParams &p, int L)
{
    const int maxL = p.max_len;
    if (L < 0 || L > maxL) {
        set_status(p.status, PKV_ERR_OUT_OF_RANGE);
        L = L < 0 ? 0 : maxL;
    }
    return L;
}

// Row of q and out that holds sequence s's query: s in plain decode; for a
// several-queries call's one-query sequences, q_rows[s] (-1: sequence s does
// not have exactly one query, or its rows are out of range -- it is skipped).
__device__ __forceinline__ int unit_row(const DecodeParams &p, int s)
{
    if (p.q_rows == nullptr)
        return s;
    const int a = __ldg(p.q_rows + s), b = __ldg(p.q_rows + s + 1);
    return (b - a == 1 && a >= 0 && b <= p.num_rows) ? a : -1;
}

// The attended length of sequence s: its clamped seq_len, or 0 for a
// sequence the call skips (it then writes no output row).
__device__ __forceinline__ int seq_len_of(const DecodeParams &p, int s)
{
    if (p.q_rows != nullptr && unit_row(p, s) < 0)
        return 0;
    return clamp_len(p, __ldg(p.seq_lens + s));
}

// Score scale (log2 domain) and output scale of the units of KV head hkv:
// the per-head factors of an fp8 cache multiply the per-tensor ones.
__device__ __forceinline__ float unit_score_scale(const DecodeParams &p, int hkv)
{
    return p.k_head_scale ? p.score_scale * __ldg(p.k_head_scale + hkv) : p.score_scale;
}
__device__ __forceinline__ float unit_out_scale(const DecodeParams &p, int hkv)
{
    return p.v_head_scale ? p.out_scale * __ldg(p.v_head_scale + hkv) : p.out_scale;
}
// The divisors the fused cache write quantises head hkv's new rows with.
__device__ __forceinline__ float unit_k_quant(const DecodeParams &p, int hkv)
{
    return p.k_head_scale ? p.k_scale * __ldg(p.k_head_scale + hkv) : p.k_scale;
}
__device__ __forceinline__ float unit_v_quant(const DecodeParams &p, int hkv)
{
    return p.v_head_scale ? p.v_scale * __ldg(p.v_head_scale + hkv) : p.v_scale;
}

// The tensors of layer `layer`, by value: a single-layer call's own (kernel
// parameters, read from the constant bank), else the caller's device table
// entry (read-only loads).  kMulti = false: the kernel form compiled for
// single-layer calls only.
template <bool kMulti = true>
__device__ __forceinline__ LayerPtrs layer_ptrs(const DecodeParams &p, int layer)
{
    if (!kMulti || p.layers == nullptr)
        return p.one;
    const unsigned long long *e = reinterpret_cast<const unsigned long long *>(p.layers + layer);
    LayerPtrs lt;
    lt.q = reinterpret_cast<const void *>(__ldg(e + 0));
    lt.new_k = reinterpret_cast<const void *>(__ldg(e + 1));
    lt.new_v = reinterpret_cast<const void *>(__ldg(e + 2));
    lt.k_cache = reinterpret_cast<void *>(__ldg(e + 3));
    lt.v_cache = reinterpret_cast<void *>(__ldg(e + 4));
    lt.out = reinterpret_cast<void *>(__ldg(e + 5));
    return lt;
}

// Whether a layer's tensors can be used: a single-layer call's were checked
// on the host; a table entry needs q, the caches and out non-null and
// 16-byte aligned, and the new rows either absent or both present and
// aligned.  A bad entry is reported (PKV_ERR_INVALID_ARG) and its layer is
// skipped: nothing is read through it or written to it.
template <bool kMulti = true>
__device__ __forceinline__ bool layer_usable(const DecodeParams &p, const LayerPtrs &lt)
{
    if (!kMulti || p.layers == nullptr)
        return true;
    const auto a16 = [](const void *x) {
        return x != nullptr && (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    };
    const bool rows = (lt.new_k == nullptr && lt.new_v == nullptr) ||
                      (a16(lt.new_k) && a16(lt.new_v));
    return a16(lt.q) && a16(lt.k_cache) && a16(lt.v_cache) && a16(lt.out) && rows;
}

// Partitions of a sequence of L tokens (an empty sequence still has one item,
// which writes its zero row).
__device__ __forceinline__ int parts_of(int L, int P) { return L > P ? (L + P - 1) / P : 1; }

// out[row of s, h, 4*q4 .. 4*q4+3] = v (f32 or bf16 output) for a layer's
// `out`; nothing for a sequence the call skips.
__device__ __forceinline__ void store_out4(const DecodeParams &p, void *out, int D, int s, int h,
                                           int q4, float4 v)
{
    const int row = unit_row(p, s);
    if (row < 0)
        return;
    const size_t off = (static_cast<size_t>(row) * p.num_q_heads + h) * D + 4 * q4;
    if (p.out_dtype == PKV_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(out) + off) = v;
    } else {
        uint2 w;
        w.x = pack_bf16(v.x, v.y);
        w.y = pack_bf16(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<unsigned short *>(out) + off) = w;
    }
}

// Merges the nparts partials of (sequence s, KV head hkv) for its G query
// heads and writes the output rows of `out`; gs is the sequence's global
// index l * S + s (its partial rows).  Partition i carries its normalised
// output o_i, the max m_i of its log2-scaled scores and l_i = sum 2^(z - m_i);
// by the associativity of the online-softmax recurrence the full result is
//     M = max_i m_i,  w_i = l_i 2^(m_i - M),  out = sum_i w_i o_i / sum_i w_i.
// Partitions are summed in index order, so the result does not depend on
// which CTA wrote which partial.  Called by all threads of a CTA.
template <int D>
__device__ void merge_partials(const DecodeParams &p, void *out, int s, int gs, int hkv,
                               int nparts)
{
    constexpr int Q4 = D / 4;
    const int G = p.group;
    for (int idx = threadIdx.x; idx < G * Q4; idx += blockDim.x) {
        const int g = idx / Q4, q4 = idx - g * Q4;
        const int h = hkv * G + g;
        const size_t row0 = (static_cast<size_t>(gs) * p.num_q_heads + h) * p.max_parts;
        const float *ml = p.part_ml + 2 * row0;
        float mx = -INFINITY;
        for (int i = 0; i < nparts; ++i)
            mx = fmaxf(mx, __ldcg(ml + 2 * i));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        for (int i = 0; i < nparts; ++i) {
            const float m = __ldcg(ml + 2 * i), l = __ldcg(ml + 2 * i + 1);
            const float w = (m == -INFINITY) ? 0.f : l * exp2f(m - mx);
            wsum += w;
            const float4 o = __ldcg(reinterpret_cast<const float4 *>(p.part_o + (row0 + i) * D) + q4);
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
        }
        const float sc = (wsum > 0.f ? 1.f / wsum : 0.f) * unit_out_scale(p, hkv);
        store_out4(p, out, D, s, h, q4,
                   make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc));
    }
}

}  // namespace pkv
