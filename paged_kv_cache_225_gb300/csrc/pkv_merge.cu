// Stand-alone log-sum-exp merge of split-sequence partials (the decode
// kernel merges in place by default; PKV_FLAG_SEPARATE_MERGE selects this
// second kernel instead).  One CTA per (layer, sequence, KV head); those with
// more than one partition merge; see merge_partials for the algebra.
#include "pkv_merge.cuh"

namespace pkv {

template <int D>
__global__ void __launch_bounds__(kThreads) merge_kernel(const __grid_constant__ DecodeParams p)
{
    const int gs = blockIdx.x / p.num_kv_heads;  // layer * S + sequence
    const int hkv = blockIdx.x - gs * p.num_kv_heads;
    const int layer = gs / p.num_seqs, s = gs - layer * p.num_seqs;
    const LayerPtrs lt = layer_ptrs(p, layer);
    if (!layer_usable(p, lt))
        return;  // reported by the decode kernel
    const int L = seq_len_of(p, s);
    const int n = parts_of(L, p.partition);
    if (n <= 1)
        return;  // the decode kernel wrote this row directly
    merge_partials<D>(p, lt.out, s, gs, hkv, n);
}

pkv_status launch_merge(const DecodeParams &p, cudaStream_t stream)
{
    const long ctas = static_cast<long>(p.num_layers) * p.num_seqs * p.num_kv_heads;
    if (ctas <= 0)
        return PKV_OK;
    const unsigned grid = static_cast<unsigned>(ctas);
    if (p.head_dim == 128)
        merge_kernel<128><<<grid, kThreads, 0, stream>>>(p);
    else if (p.head_dim == 64)
        merge_kernel<64><<<grid, kThreads, 0, stream>>>(p);
    else
        return PKV_ERR_UNSUPPORTED;
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
