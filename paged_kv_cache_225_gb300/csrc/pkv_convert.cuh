// Element conversions of the paged cache write, shared by the cache-write
// kernel and the fused write-and-decode path of the decode kernels.
// F32 -> F32 and BF16 -> BF16 copy the bits; F32 -> BF16 rounds to nearest
// even; BF16 -> F32 widens exactly; -> FP8_E5M2 / FP8_E4M3 store
// round-to-nearest-even(x / scale) in float32, saturated to +-57344 / +-448.
#pragma once

#include <cuda_fp8.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

__device__ __forceinline__ float load_in(const void *src, int dtype, size_t i)
{
    if (dtype == PKV_F32)
        return static_cast<const float *>(src)[i];
    return __uint_as_float(static_cast<uint32_t>(static_cast<const unsigned short *>(src)[i])
                           << 16);
}

// cache[i] = cvt(src[j]) for a cache of `dtype` (generic pointer: global or
// shared memory).
__device__ __forceinline__ void store_kv(void *cache, int dtype, size_t i, const void *src,
                                         int in_dtype, size_t j, float scale)
{
    if (dtype == PKV_F32) {
        static_cast<float *>(cache)[i] = load_in(src, in_dtype, j);
    } else if (dtype == PKV_BF16) {
        unsigned short b;
        if (in_dtype == PKV_BF16)
            b = static_cast<const unsigned short *>(src)[j];
        else
            b = __bfloat16_as_ushort(__float2bfloat16_rn(static_cast<const float *>(src)[j]));
        static_cast<unsigned short *>(cache)[i] = b;
    } else {
        const float x = load_in(src, in_dtype, j) / scale;
        static_cast<unsigned char *>(cache)[i] = static_cast<unsigned char>(__nv_cvt_float_to_fp8(
            x, __NV_SATFINITE, dtype == PKV_FP8_E4M3 ? __NV_E4M3 : __NV_E5M2));
    }
}

// cache[i] = cvt(x) for a value already widened to float (exact for F32 and
// BF16 inputs, so the stored bits equal store_kv's for non-NaN inputs).
__device__ __forceinline__ void store_kv_value(void *cache, int dtype, size_t i, float x,
                                               float scale)
{
    if (dtype == PKV_F32)
        static_cast<float *>(cache)[i] = x;
    else if (dtype == PKV_BF16)
        static_cast<unsigned short *>(cache)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
    else
        static_cast<unsigned char *>(cache)[i] = static_cast<unsigned char>(__nv_cvt_float_to_fp8(
            x / scale, __NV_SATFINITE, dtype == PKV_FP8_E4M3 ? __NV_E4M3 : __NV_E5M2));
}

}  // namespace pkv
