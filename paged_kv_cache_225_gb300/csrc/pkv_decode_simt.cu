// CUDA-core (FFMA) decode kernels: every KV dtype, head_dim 64/128, up to 16
// query heads per KV head (padded to a power of two).  The fp8 dtypes are
// instantiated in pkv_decode_simt_fp8.cu.
#include "pkv_streamk.cuh"

namespace pkv {

template <int KV, int D>
static pkv_status dispatch_group(const DecodeParams &p, cudaStream_t stream)
{
    const int G = p.group;
    if (G <= 1)
        return launch_any<SimtPolicy<KV, D, 1>>(p, stream);
    if (G <= 2)
        return launch_any<SimtPolicy<KV, D, 2>>(p, stream);
    if (G <= 4)
        return launch_any<SimtPolicy<KV, D, 4>>(p, stream);
    if (G <= 8)
        return launch_any<SimtPolicy<KV, D, 8>>(p, stream);
    if (G <= 16)
        return launch_any<SimtPolicy<KV, D, 16>>(p, stream);
    return PKV_ERR_UNSUPPORTED;
}

template <int KV>
static pkv_status dispatch_dim(const DecodeParams &p, cudaStream_t stream)
{
    if (p.head_dim == 64)
        return dispatch_group<KV, 64>(p, stream);
    if (p.head_dim == 128)
        return dispatch_group<KV, 128>(p, stream);
    return PKV_ERR_UNSUPPORTED;
}

pkv_status launch_decode_simt(const DecodeParams &p, int kv_dtype, cudaStream_t stream)
{
    switch (kv_dtype) {
    case PKV_F32:
        return dispatch_dim<PKV_F32>(p, stream);
    case PKV_BF16:
        return dispatch_dim<PKV_BF16>(p, stream);
    case PKV_FP8_E5M2:
    case PKV_FP8_E4M3:
    case PKV_INT4:
        return launch_decode_simt_fp8(p, kv_dtype, stream);
    default:
        return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace pkv
