// CUDA-core (FFMA) decode kernels for the 8- and 4-bit KV dtypes (fp8 e5m2,
// fp8 e4m3, INT4), in a translation unit of their own so the build compiles
// them in parallel.
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

pkv_status launch_decode_simt_fp8(const DecodeParams &p, int kv_dtype, cudaStream_t stream)
{
    switch (kv_dtype) {
    case PKV_FP8_E5M2:
        return dispatch_dim<PKV_FP8_E5M2>(p, stream);
    case PKV_FP8_E4M3:
        return dispatch_dim<PKV_FP8_E4M3>(p, stream);
    case PKV_INT4:
        return dispatch_dim<PKV_INT4>(p, stream);
    default:
        return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace pkv
