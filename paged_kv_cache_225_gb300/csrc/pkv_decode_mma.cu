// Tensor-core (mma.sync) decode kernels: bf16, fp8 (e5m2, e4m3) and INT4 KV with a bf16
// query, head_dim 64/128, up to 16 query heads per KV head (one or two
// 8-wide N tiles).
#include "pkv_streamk.cuh"

namespace pkv {

bool mma_supports(int kv_dtype, int q_dtype, int head_dim, int group)
{
    return (kv_dtype == PKV_BF16 || is_scaled(kv_dtype)) && q_dtype == PKV_BF16 &&
           (head_dim == 64 || head_dim == 128) && group >= 1 && group <= 16;
}

template <int D>
static pkv_status dispatch(const DecodeParams &p, int kv_dtype, cudaStream_t stream)
{
    const bool two = p.group > 8;
    if (kv_dtype == PKV_BF16)
        return two ? launch_any<MmaBf16Policy<D, 2>>(p, stream)
                   : launch_any<MmaBf16Policy<D, 1>>(p, stream);
    if (kv_dtype == PKV_INT4)
        return two ? launch_any<MmaInt4Policy<D, 2>>(p, stream)
                   : launch_any<MmaInt4Policy<D, 1>>(p, stream);
    if (kv_dtype == PKV_FP8_E4M3)
        return two ? launch_any<MmaFp8Policy<D, 2, compact_ring_budget(2), false, PKV_FP8_E4M3>>(
                         p, stream)
                   : launch_any<MmaFp8Policy<D, 1, compact_ring_budget(1), false, PKV_FP8_E4M3>>(
                         p, stream);
    return two ? launch_any<MmaFp8Policy<D, 2>>(p, stream)
               : launch_any<MmaFp8Policy<D, 1>>(p, stream);
}

pkv_status launch_decode_mma(const DecodeParams &p, int kv_dtype, cudaStream_t stream)
{
    if (!mma_supports(kv_dtype, p.q_dtype, p.head_dim, p.group))
        return PKV_ERR_UNSUPPORTED;
    return p.head_dim == 64 ? dispatch<64>(p, kv_dtype, stream)
                            : dispatch<128>(p, kv_dtype, stream);
}

}  // namespace pkv
