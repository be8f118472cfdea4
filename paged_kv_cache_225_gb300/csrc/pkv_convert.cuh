// Element conversions of the paged cache write, shared by the cache-write
// kernel and the fused write-and-decode path of the decode kernels.
// F32 -> F32 and BF16 -> BF16 copy the bits; F32 -> BF16 rounds to nearest
// even; BF16 -> F32 widens exactly; -> FP8_E5M2 / FP8_E4M3 store
// round-to-nearest-even(x / scale) in float32, saturated to +-57344 / +-448;
// -> INT4 the same rounding clamped to -8..7.
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

// Element i of an INT4 cache (nibble i & 1 of byte i / 2) set to the code of
// round-half-even(x / scale) clamped to -8..7 (NaN -> 0).  Two tokens share
// a byte and may be written at once, so the nibble is replaced with two
// atomics on the aligned 32-bit word (global memory).
__device__ __forceinline__ void store_int4(void *cache, size_t i, float x, float scale)
{
    float qf = rintf(x / scale);
    qf = (qf != qf) ? 0.f : fminf(fmaxf(qf, -8.f), 7.f);
    const uint32_t code = static_cast<uint32_t>(static_cast<int>(qf)) & 0xfu;
    const size_t byte = i >> 1;
    unsigned int *word = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(cache) +
                                                          (byte & ~static_cast<size_t>(3)));
    const int shift = static_cast<int>((byte & 3) * 8 + (i & 1) * 4);
    atomicAnd(word, ~(0xfu << shift));
    atomicOr(word, code << shift);
}

// cache[i] = cvt(src[j]) for a cache of `dtype` (generic pointer: global or
// shared memory; INT4 caches only in global memory).
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
    } else if (dtype == PKV_INT4) {
        store_int4(cache, i, load_in(src, in_dtype, j), scale);
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
    else if (dtype == PKV_INT4)
        store_int4(cache, i, x, scale);
    else
        static_cast<unsigned char *>(cache)[i] = static_cast<unsigned char>(__nv_cvt_float_to_fp8(
            x / scale, __NV_SATFINITE, dtype == PKV_FP8_E4M3 ? __NV_E4M3 : __NV_E5M2));
}

}  // namespace pkv
