// Log-sum-exp merge of split-sequence partials.
//
// Each partition p of a sequence carries its normalised output o_p, the max
// m_p of its (log2-scaled) scores and its sum l_p = sum exp2(z - m_p).  The
// online-softmax recurrence of the PagedAttention pseudocode is associative,
// so the exact full-sequence result is
//     M = max_p m_p,  w_p = l_p * 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// One warp per (sequence, query head); sequences with one partition were
// written directly by the decode kernel and are skipped.
#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p)
{
    constexpr int V = D / 32;  // floats per lane
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw >= p.num_seqs * p.num_q_heads)
        return;
    const int s = gw / p.num_q_heads;
    int L = __ldg(p.seq_lens + s);
    const int maxL = p.max_len;
    L = L < 0 ? 0 : (L > maxL ? maxL : L);
    const int n = L > p.partition ? (L + p.partition - 1) / p.partition : 1;
    if (n <= 1)
        return;
    const size_t row0 = static_cast<size_t>(gw) * p.max_parts;
    const float *ml = p.part_ml + 2 * row0;

    float mx = -INFINITY;
    for (int i = lane; i < n; i += 32)
        mx = fmaxf(mx, ml[2 * i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));

    float acc[V];
#pragma unroll
    for (int k = 0; k < V; ++k)
        acc[k] = 0.f;
    float wsum = 0.f;
    for (int i = 0; i < n; ++i) {
        const float m = ml[2 * i], l = ml[2 * i + 1];
        const float w = (m == -INFINITY) ? 0.f : l * exp2f(m - mx);
        wsum += w;
        const float *o = p.part_o + (row0 + i) * D + lane * V;
        if constexpr (V == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(o);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(o);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        }
    }
    const float sc = (wsum > 0.f ? 1.f / wsum : 0.f) * p.out_scale;
    const size_t off = static_cast<size_t>(gw) * D + lane * V;
    if (p.out_dtype == PKV_F32) {
        float *out = static_cast<float *>(p.out) + off;
#pragma unroll
        for (int k = 0; k < V; ++k)
            out[k] = acc[k] * sc;
    } else {
        uint32_t *out = reinterpret_cast<uint32_t *>(static_cast<unsigned short *>(p.out) + off);
#pragma unroll
        for (int k = 0; k < V; k += 2)
            out[k / 2] = pack_bf16(acc[k] * sc, acc[k + 1] * sc);
    }
}

pkv_status launch_merge(const DecodeParams &p, cudaStream_t stream)
{
    const long warps = static_cast<long>(p.num_seqs) * p.num_q_heads;
    const unsigned grid = static_cast<unsigned>((warps * 32 + 127) / 128);
    if (grid == 0)
        return PKV_OK;
    if (p.head_dim == 128)
        merge_kernel<128><<<grid, 128, 0, stream>>>(p);
    else if (p.head_dim == 64)
        merge_kernel<64><<<grid, 128, 0, stream>>>(p);
    else
        return PKV_ERR_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
