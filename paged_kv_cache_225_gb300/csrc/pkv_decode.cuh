// Paged decode attention kernels for sm_103a.
//
// What is computed follows the PagedAttention kernel pseudocode of
// "vLLM e PagedAttention: serving high-throughput": for each sequence and
// query head, walk the logical blocks, look up the physical block in the
// block table, score the block's keys, fold them into a running max / running
// sum softmax, accumulate the value rows, and divide by the sum at the end.
//
// How it is laid out on the GPU (not taken from the pages):
//  * A work item is (sequence, KV head, partition of `partition` tokens).  One
//    CTA of four warps owns an item; the G = Hq/Hkv query heads of the KV head
//    share every K/V page it reads, so each page crosses HBM once per KV head.
//  * The warps split the item's pages round-robin.  Each warp streams its
//    pages through a private ring of R shared-memory stages, filled by 1-D
//    bulk (TMA) copies of the contiguous [head_dim x 16] K and V tiles and
//    completed on an mbarrier; waits are bounded and report a timeout
//    instead of hanging.
//  * Each warp keeps its own softmax state; at the end of an item the four
//    states are merged through shared memory with log-sum-exp weights.  A
//    sequence that fits one partition is written straight to `out`;
//    otherwise the item writes a normalised partial to the workspace and the
//    CTA whose partial completes the sequence (an arrival counter per
//    sequence and KV head) merges them all in partition order.  With
//    PKV_FLAG_SEPARATE_MERGE the merge runs as a second kernel instead
//    (pkv_merge.cu); both give the same bits.
//  * In split mode the grid is persistent: CTAs pull items from an atomic
//    counter and map the item index to (sequence, partition) with a warp
//    prefix scan over the per-sequence partition counts.
//  * With few (sequence, KV head) units the automatic schedule is stream-K
//    instead (pkv_streamk.cuh): equal page ranges per CTA, same policies.
//  * Per page, scores and the value accumulation run either on CUDA cores
//    (SimtPolicy) or on tensor cores with mma.sync (MmaBf16Policy,
//    MmaFp8Policy): S^T = K^T Q^T puts the page's 16 tokens on the MMA's M
//    dimension and the (up to 8) grouped heads on N; P^T is transposed in
//    registers with movmatrix and O^T = V P^T puts head_dim on M.
#pragma once

#include <climits>
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_convert.cuh"
#include "pkv_internal.h"
#include "pkv_merge.cuh"

// Shared-memory budget of one warp's page ring (bytes); the stage count
// follows from it (2..8 stages).  16 KB (two 8 KB bf16 stages) leaves room
// for three CTAs per SM, which hides each CTA's item-boundary bubbles better
// than deeper rings with fewer CTAs (measured on GB300).
#ifndef PKV_RING_BYTES_PER_WARP
#define PKV_RING_BYTES_PER_WARP (16 * 1024)
#endif


namespace pkv {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per bounded wait

template <int KV> struct KvBytes;
template <> struct KvBytes<PKV_F32> { static constexpr int v = 4; };
template <> struct KvBytes<PKV_BF16> { static constexpr int v = 2; };
template <> struct KvBytes<PKV_FP8_E5M2> { static constexpr int v = 1; };
template <> struct KvBytes<PKV_FP8_E4M3> { static constexpr int v = 1; };

// Per-CTA shared memory the stream-K kernel plans for (two CTAs per SM) and
// the ring budget per warp it may use at most.
#ifndef PKV_CTA_SMEM_TARGET
#define PKV_CTA_SMEM_TARGET (113 * 1024)
#endif
#ifndef PKV_STREAMK_RING_BYTES_PER_WARP
#define PKV_STREAMK_RING_BYTES_PER_WARP (24 * 1024)
#endif

// Merge scratch of one warp: O[GP][D], m[GP], l[GP] in fp32, padded to a
// multiple of 4 floats so every warp's O rows stay 16-byte aligned for float4
// reads.
__host__ __device__ constexpr int scratch_floats(int GP, int D)
{
    return (GP * D + 2 * GP + 3) / 4 * 4;
}
__host__ __device__ constexpr int scratch_bytes(int GP, int D)
{
    return kWarps * scratch_floats(GP, D) * 4;
}

// Ring bytes per warp for a kernel whose other shared memory (policy data and
// a separate merge scratch) takes `other` bytes of the per-CTA target.
__host__ __device__ constexpr int ring_budget(int other)
{
    return (PKV_CTA_SMEM_TARGET - other - 256) / kWarps < PKV_STREAMK_RING_BYTES_PER_WARP
               ? (PKV_CTA_SMEM_TARGET - other - 256) / kWarps
               : PKV_STREAMK_RING_BYTES_PER_WARP;
}

// Per-warp ring geometry: `Budget` bytes of page stages per warp.
template <int KV, int D, int Budget> struct Ring {
    static constexpr int kTileBytes = tile_bytes(KV, D);  // one K or V page tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kRaw = Budget / kStageBytes;
    static constexpr int R = kRaw < 2 ? 2 : (kRaw > 8 ? 8 : kRaw);
    static constexpr int kRingBytes = R * kStageBytes;
};

__device__ __forceinline__ float load_q(const DecodeParams &p, const void *q, size_t idx)
{
    if (p.q_dtype == PKV_F32)
        return static_cast<const float *>(q)[idx];
    const unsigned short b = static_cast<const unsigned short *>(q)[idx];
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// ============================================================== CUDA cores

// Scores: lane (t, half) owns token t of the page and half of head_dim; the
// two halves are summed with one shuffle.  Values: lane owns head_dim rows
// lane + 32j and walks the page's valid tokens.  GT = heads padded to 2^k.
template <int KV, int D, int GT, int Budget = PKV_RING_BYTES_PER_WARP>
struct SimtPolicy {
    using RingT = Ring<KV, D, Budget>;
    static constexpr int R = RingT::R;
    static constexpr int kTileBytes = RingT::kTileBytes;
    static constexpr int kStageBytes = RingT::kStageBytes;
    static constexpr int kRingBytes = RingT::kRingBytes;
    static constexpr int kDim = D;
    static constexpr int GP = GT;
    static constexpr int kHalf = D / 2;
    static constexpr int kQHalfStride = kHalf * GT + 4;  // pad: the halves hit other banks
    static constexpr int kExtraBytes = (2 * kQHalfStride + kWarps * kBlockSize * GT) * 4;
    static constexpr int DJ = D / 32;
    // The same policy with a separate merge scratch and the ring that fits.
    using StreamK = SimtPolicy<KV, D, GT, ring_budget(kExtraBytes + scratch_bytes(GT, D))>;

    struct State {
        float m[GT];
        float l[GT];
        float o[DJ][GT];
    };
    static constexpr bool kStaged = false;  // reads K/V straight from the stage
    static constexpr bool kSharedBegin = true;  // begin() writes the query to shared memory
    // No separate single-layer kernel form (its many instantiations are built
    // once, in the layered form that serves both).
    static constexpr bool kSingleForm = false;
    static constexpr int kMinBlocks = 2;        // CTAs per SM the registers are bounded for
    struct Frags {};
    __device__ static void load(Frags &, const unsigned char *, const unsigned char *, int) {}
    __device__ static void compute(State &, Frags &, int, int, float) {}

    __device__ static float kv_at(const unsigned char *tile, int idx)
    {
        if constexpr (KV == PKV_F32)
            return reinterpret_cast<const float *>(tile)[idx];
        else if constexpr (KV == PKV_BF16)
            return __uint_as_float(
                static_cast<uint32_t>(reinterpret_cast<const unsigned short *>(tile)[idx]) << 16);
        else if constexpr (KV == PKV_FP8_E5M2)
            return e5m2_to_float(tile[idx]);
        else if constexpr (KV == PKV_FP8_E4M3)
            return e4m3_to_float(tile[idx]);
        else
            return int4_to_float(tile[idx >> 1], idx & 1);
    }

    // One page row V[d][0..15] widened to floats.
    __device__ static void kv_row(const unsigned char *tile, int d, float (&v)[kBlockSize])
    {
        if constexpr (KV == PKV_F32) {
            const float4 *r = reinterpret_cast<const float4 *>(tile + d * kBlockSize * 4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4 x = r[i];
                v[4 * i] = x.x;
                v[4 * i + 1] = x.y;
                v[4 * i + 2] = x.z;
                v[4 * i + 3] = x.w;
            }
        } else if constexpr (KV == PKV_BF16) {
            const uint4 *r = reinterpret_cast<const uint4 *>(tile + d * kBlockSize * 2);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint4 x = r[i];
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * i + 2 * k] = bf16_lo(w[k]);
                    v[8 * i + 2 * k + 1] = bf16_hi(w[k]);
                }
            }
        } else if constexpr (KV == PKV_INT4) {
            const uint2 x = *reinterpret_cast<const uint2 *>(tile + d * (kBlockSize / 2));
            const uint32_t w[2] = {x.x, x.y};
#pragma unroll
            for (int k = 0; k < 2; ++k)
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    v[8 * k + b] = static_cast<float>(
                        static_cast<int>(((w[k] >> (4 * b)) & 0xfu) ^ 0x8u) - 8);
        } else {
            const uint4 x = *reinterpret_cast<const uint4 *>(tile + d * kBlockSize);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    v[4 * k + b] = KV == PKV_FP8_E5M2 ? e5m2_to_float(w[k] >> (8 * b))
                                                      : e4m3_to_float(w[k] >> (8 * b));
        }
    }

    __device__ static void begin(State &st, const DecodeParams &p, const void *q, int s, int hkv,
                                 int lane, unsigned char *extra)
    {
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            st.m[g] = -INFINITY;
            st.l[g] = 0.f;
#pragma unroll
            for (int j = 0; j < DJ; ++j)
                st.o[j][g] = 0.f;
        }
        float *sq = reinterpret_cast<float *>(extra);
        const int G = p.group;
        for (int idx = threadIdx.x; idx < D * GT; idx += kThreads) {
            const int d = idx / GT, g = idx - d * GT;
            float v = 0.f;
            if (g < G && q != nullptr)  // null: a skipped layer's unit, zero query
                v = load_q(p, q, (static_cast<size_t>(s) * p.num_q_heads + hkv * G + g) * D + d);
            const int half = d / kHalf;
            sq[half * kQHalfStride + (d - half * kHalf) * GT + g] = v;
        }
        (void)lane;
    }

    __device__ static void page(State &st, const unsigned char *sK, const unsigned char *sV,
                                int valid, int lane, int warp, unsigned char *extra, float c)
    {
        const float *sq = reinterpret_cast<const float *>(extra);
        float *sp = reinterpret_cast<float *>(extra) + 2 * kQHalfStride + warp * kBlockSize * GT;
        const int t = lane & 15, half = lane >> 4;
        const float *qh = sq + half * kQHalfStride;
        float acc[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g)
            acc[g] = 0.f;
#pragma unroll 8
        for (int i = 0; i < kHalf; ++i) {
            const float k = kv_at(sK, (half * kHalf + i) * kBlockSize + t);
#pragma unroll
            for (int g = 0; g < GT; ++g)
                acc[g] = fmaf(qh[i * GT + g], k, acc[g]);
        }
        float alpha[GT];
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            acc[g] += __shfl_xor_sync(kFullMask, acc[g], 16);
            const float sc = (t < valid) ? acc[g] * c : -INFINITY;
            float mx = sc;
#pragma unroll
            for (int off = 1; off < 16; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(kFullMask, mx, off));
            const float mnew = fmaxf(st.m[g], mx);
            alpha[g] = (st.m[g] == -INFINITY) ? 0.f : exp2f(st.m[g] - mnew);
            const float pr = (t < valid) ? exp2f(sc - mnew) : 0.f;
            st.l[g] = st.l[g] * alpha[g] + (half == 0 ? pr : 0.f);
            st.m[g] = mnew;
            if (half == 0)
                sp[t * GT + g] = pr;
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < DJ; ++j) {
            float v[kBlockSize];
            kv_row(sV, lane + 32 * j, v);
#pragma unroll
            for (int g = 0; g < GT; ++g)
                st.o[j][g] *= alpha[g];
#pragma unroll
            for (int tt = 0; tt < kBlockSize; ++tt) {
                if (tt < valid) {
#pragma unroll
                    for (int g = 0; g < GT; ++g)
                        st.o[j][g] = fmaf(sp[tt * GT + g], v[tt], st.o[j][g]);
                }
            }
        }
        __syncwarp();
    }

    __device__ static void finish(State &st, float *so, float *sm, float *sl, int lane)
    {
#pragma unroll
        for (int g = 0; g < GT; ++g) {
            float l = st.l[g];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1)
                l += __shfl_xor_sync(kFullMask, l, off);
            if (lane == 0) {
                sm[g] = st.m[g];
                sl[g] = l;
            }
#pragma unroll
            for (int j = 0; j < DJ; ++j)
                so[g * D + lane + 32 * j] = st.o[j][g];
        }
    }
};

// ============================================================ tensor cores

// Shared by the bf16 and fp8 tensor-core policies: online-softmax update of
// one N tile from S^T accumulators.  tokA/tokB are the page tokens of the
// accumulator rows r and r+8 this lane holds; heads 8n+2c, 8n+2c+1.
struct MmaSoftmax {
    // Scores may run up to 2^kLazy above the running max before the max is
    // raised: p = 2^(s - m) then stays <= 2^8, harmless in fp32, and the
    // cross-lane max reduction and the O rescale are skipped on most pages.
    // (m, l, O) stay mutually consistent, so the result is the same softmax.
    static constexpr float kLazy = 8.f;

    __device__ static float ex2(float x)
    {
        float y;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
        return y;
    }

    // Returns true when the running max moved (the caller rescales O by alpha).
    __device__ static bool update(const float (&sacc)[4], int tokA, int tokB, int valid, float c,
                                  float (&m)[2], float (&l)[2], float (&p)[4], float (&alpha)[2])
    {
        const float s0 = tokA < valid ? sacc[0] * c : -INFINITY;
        const float s1 = tokA < valid ? sacc[1] * c : -INFINITY;
        const float s2 = tokB < valid ? sacc[2] * c : -INFINITY;
        const float s3 = tokB < valid ? sacc[3] * c : -INFINITY;
        const bool fast = s0 <= m[0] + kLazy && s2 <= m[0] + kLazy && s1 <= m[1] + kLazy &&
                          s3 <= m[1] + kLazy;
        if (__all_sync(kFullMask, fast)) {
            // m finite here: masked positions (s = -inf) give p = 0.
            p[0] = ex2(s0 - m[0]);
            p[1] = ex2(s1 - m[1]);
            p[2] = ex2(s2 - m[0]);
            p[3] = ex2(s3 - m[1]);
            l[0] += p[0] + p[2];
            l[1] += p[1] + p[3];
            return false;
        }
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        alpha[0] = (m[0] == -INFINITY) ? 0.f : ex2(m[0] - mn0);
        alpha[1] = (m[1] == -INFINITY) ? 0.f : ex2(m[1] - mn1);
        p[0] = tokA < valid ? ex2(s0 - mn0) : 0.f;
        p[1] = tokA < valid ? ex2(s1 - mn1) : 0.f;
        p[2] = tokB < valid ? ex2(s2 - mn0) : 0.f;
        p[3] = tokB < valid ? ex2(s3 - mn1) : 0.f;
        l[0] = l[0] * alpha[0] + p[0] + p[2];
        l[1] = l[1] * alpha[1] + p[1] + p[3];
        m[0] = mn0;
        m[1] = mn1;
        return true;
    }
};

template <int D, int NT>
struct MmaStateBase {
    static constexpr int KS = D / 16;  // 16-wide k steps of q.K
    static constexpr int MT = D / 16;  // 16-row tiles of head_dim in O^T
    struct State {
        float o[MT][NT][4];
        float m[NT][2];
        float l[NT][2];
        uint32_t qf[KS][NT][2];
    };

    __device__ static void reset(State &st)
    {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    st.o[mt][n][e] = 0.f;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            st.m[n][0] = st.m[n][1] = -INFINITY;
            st.l[n][0] = st.l[n][1] = 0.f;
        }
    }

    // Query fragments (B operand of S^T = K^T Q^T): lane (r, c) holds
    // q[head 8n+r][16ks + 2c, +1] and [16ks + 8 + 2c, +1]; heads >= G are 0,
    // and so is every head when q is null (a skipped layer's unit).
    template <bool F16>
    __device__ static void load_q_frags(State &st, const DecodeParams &p, const void *q, int s,
                                        int hkv, int lane)
    {
        const int r = lane >> 2, c = lane & 3;
        const int G = p.group;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int g = 8 * n + r;
            const bool ok = g < G && q != nullptr;
            const size_t row = (static_cast<size_t>(s) * p.num_q_heads + hkv * G + (ok ? g : 0)) * D;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int d = 16 * ks + 8 * hh + 2 * c;
                    uint32_t w = 0;
                    if (ok) {
                        if (!F16) {
                            w = *reinterpret_cast<const uint32_t *>(
                                static_cast<const unsigned short *>(q) + row + d);
                        } else {
                            const float a = load_q(p, q, row + d), b = load_q(p, q, row + d + 1);
                            w = pack_f16(a, b);
                        }
                    }
                    st.qf[ks][n][hh] = w;
                }
            }
        }
    }

    // O^T accumulator element (mt, n, e) is O[head 8n + 2c + (e&1)][16mt + r + 8(e>>1)].
    __device__ static void finish(State &st, float *so, float *sm, float *sl, int lane)
    {
        const int r = lane >> 2, c = lane & 3;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = st.l[n][e];
                l += __shfl_xor_sync(kFullMask, l, 4);
                l += __shfl_xor_sync(kFullMask, l, 8);
                l += __shfl_xor_sync(kFullMask, l, 16);
                if (r == 0) {
                    sm[8 * n + 2 * c + e] = st.m[n][e];
                    sl[8 * n + 2 * c + e] = l;
                }
            }
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    so[(8 * n + 2 * c + (e & 1)) * D + 16 * mt + r + 8 * (e >> 1)] = st.o[mt][n][e];
        }
    }

    __device__ static void rescale(State &st, int n, const float (&alpha)[2])
    {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            st.o[mt][n][0] *= alpha[0];
            st.o[mt][n][1] *= alpha[1];
            st.o[mt][n][2] *= alpha[0];
            st.o[mt][n][3] *= alpha[1];
        }
    }
};

// bf16 KV: the page tile is [D][16] bf16 (32-byte rows).  K^T fragments come
// from ldmatrix.trans, V fragments from ldmatrix.  P is split into a bf16 high
// part and a bf16 residual so that P V keeps ~16 mantissa bits.
//
// Staged: the whole page is first copied into registers (64 per lane), so
// the ring stage can be refilled before the math runs; the math then no
// longer holds a stage, which keeps more copies in flight.
template <int D, int NT, int Budget = PKV_RING_BYTES_PER_WARP, bool Staged = false>
struct MmaBf16Policy : MmaStateBase<D, NT> {
    using Base = MmaStateBase<D, NT>;
    using State = typename Base::State;
    using RingT = Ring<PKV_BF16, D, Budget>;
    // The same policy with a separate merge scratch and the ring that fits.
    // Stream-K stages pages in registers when G <= 8 (no spills there).
    using StreamK = MmaBf16Policy<D, NT, ring_budget(scratch_bytes(8 * NT, D)), NT == 1>;
    static constexpr int R = RingT::R;
    static constexpr int kTileBytes = RingT::kTileBytes;
    static constexpr int kStageBytes = RingT::kStageBytes;
    static constexpr int kRingBytes = RingT::kRingBytes;
    static constexpr int kDim = D;
    static constexpr int GP = 8 * NT;
    static constexpr int kExtraBytes = 0;
    static constexpr int KS = Base::KS, MT = Base::MT;
    static constexpr bool kStaged = Staged;
    static constexpr bool kSharedBegin = false;  // begin() only fills registers
    static constexpr bool kSingleForm = true;    // single-layer calls get their own form
    static constexpr int kMinBlocks = 2;

    struct Frags {
        uint32_t k[KS][4];  // K^T A fragments, one per 16-wide k step
        uint32_t v[MT][4];  // V A fragments, one per 16-row head_dim tile
    };

    __device__ static void begin(State &st, const DecodeParams &p, const void *q, int s, int hkv,
                                 int lane, unsigned char *)
    {
        Base::reset(st);
        Base::template load_q_frags<false>(st, p, q, s, hkv, lane);
    }

    __device__ static void load(Frags &f, const unsigned char *sK, const unsigned char *sV,
                                int lane)
    {
        const int mi = lane >> 3, ri = lane & 7;
        // ldmatrix row addresses.  K (.trans): matrix mi covers head_dim rows
        // 8(mi>>1).. and token half mi&1.  V: rows 8(mi&1).., token half mi>>1.
        const uint32_t ka = smem_u32(sK) + (ri + 8 * (mi >> 1)) * 32 + (mi & 1) * 16;
        const uint32_t va = smem_u32(sV) + (ri + 8 * (mi & 1)) * 32 + (mi >> 1) * 16;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            ldsm_x4_t(f.k[ks], ka + ks * 16 * 32);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
            ldsm_x4(f.v[mt], va + mt * 16 * 32);
    }

    __device__ static void compute(State &st, Frags &f, int valid, int lane, float c)
    {
        const int r = lane >> 2, cc = lane & 3;
        // S^T = K^T Q^T in two independent accumulation chains (even / odd k).
        float sacc[NT][4], sodd[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] = sodd[n][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_bf16((ks & 1) ? sodd[n] : sacc[n], f.k[ks], st.qf[ks][n][0], st.qf[ks][n][1]);
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] += sodd[n][e];

        uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float pr[4], alpha[2];
            if (MmaSoftmax::update(sacc[n], r, r + 8, valid, c, st.m[n], st.l[n], pr, alpha))
                Base::rescale(st, n, alpha);
            const uint32_t hx = pack_bf16(pr[0], pr[1]);
            const uint32_t hy = pack_bf16(pr[2], pr[3]);
            const uint32_t lx = pack_bf16(pr[0] - bf16_lo(hx), pr[1] - bf16_hi(hx));
            const uint32_t ly = pack_bf16(pr[2] - bf16_lo(hy), pr[3] - bf16_hi(hy));
            bh0[n] = movmatrix_t(hx);
            bh1[n] = movmatrix_t(hy);
            bl0[n] = movmatrix_t(lx);
            bl1[n] = movmatrix_t(ly);
        }

        if (valid < kBlockSize) {  // last page of a sequence: zero the unused tokens
            const uint32_t mlo = (2 * cc < valid ? 0x0000ffffu : 0u) |
                                 (2 * cc + 1 < valid ? 0xffff0000u : 0u);
            const uint32_t mhi = (8 + 2 * cc < valid ? 0x0000ffffu : 0u) |
                                 (9 + 2 * cc < valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                f.v[mt][0] &= mlo;
                f.v[mt][1] &= mlo;
                f.v[mt][2] &= mhi;
                f.v[mt][3] &= mhi;
            }
        }
        // High parts of P first, residuals second: products into the same
        // accumulator sit MT instructions apart.
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_bf16(st.o[mt][n], f.v[mt], bh0[n], bh1[n]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_bf16(st.o[mt][n], f.v[mt], bl0[n], bl1[n]);
    }

    __device__ static void page(State &st, const unsigned char *sK, const unsigned char *sV,
                                int valid, int lane, int, unsigned char *, float c)
    {
        Frags f;
        load(f, sK, sV, lane);
        compute(st, f, valid, lane, c);
    }

    __device__ static void finish(State &st, float *so, float *sm, float *sl, int lane)
    {
        Base::finish(st, so, sm, sl, lane);
    }
};

// fp8 KV (e5m2 or e4m3): the page tile is [D][16] bytes (16-byte rows), read
// by ldmatrix as 16-bit pairs; each code is widened to an f16, exactly (e5m2:
// byte_perm places it as the f16's high byte; e4m3: cvt.f16x2.e4m3x2).  Token order inside a fragment is
// permuted consistently on both operands (see the byte selectors).  Staged
// like the bf16 policy: 32 registers hold a page's raw codes.
// Ring bytes per warp and CTAs per SM of the fp8 item kernel.  Its pages are
// half the bytes of bf16 pages and it is bound by pages per second rather
// than bytes, so four CTAs with three 4 KB stages per warp (registers capped
// at 128, no spills) beat three CTAs with four stages: measured on GB300,
// fp8 chat layer 34.7 -> 29.8 us, 70B e4m3 layer 171 -> 160 us.
#ifndef PKV_FP8_RING_BYTES_PER_WARP
#define PKV_FP8_RING_BYTES_PER_WARP (12 * 1024)
#endif
#ifndef PKV_FP8_MIN_BLOCKS
#define PKV_FP8_MIN_BLOCKS 4
#endif

// Two-tile head groups keep three CTAs per SM and a 12 KB ring (their merge
// scratch needs more than 8 KB per warp).
__host__ __device__ constexpr int compact_ring_budget(int nt)
{
    return nt == 1 ? PKV_FP8_RING_BYTES_PER_WARP : 12 * 1024;
}

template <int D, int NT, int Budget = compact_ring_budget(NT), bool Staged = false,
          int KV = PKV_FP8_E5M2>
struct MmaFp8Policy : MmaStateBase<D, NT> {
    using Base = MmaStateBase<D, NT>;
    using State = typename Base::State;
    using RingT = Ring<KV, D, Budget>;
    // The same policy with a separate merge scratch and the ring that fits.
    // Stream-K stages pages in registers when G <= 8 (no spills there).
    using StreamK = MmaFp8Policy<D, NT, ring_budget(scratch_bytes(8 * NT, D)), NT == 1, KV>;
    static constexpr int R = RingT::R;
    static constexpr int kTileBytes = RingT::kTileBytes;
    static constexpr int kStageBytes = RingT::kStageBytes;
    static constexpr int kRingBytes = RingT::kRingBytes;
    static constexpr int kDim = D;
    static constexpr int GP = 8 * NT;
    static constexpr int kExtraBytes = 0;
    static constexpr int KS = Base::KS, MT = Base::MT;
    static constexpr bool kStaged = Staged;
    static constexpr bool kSharedBegin = false;  // begin() only fills registers
    static constexpr bool kSingleForm = true;    // single-layer calls get their own form
    // Two N tiles (more than 8 heads per KV head) need more registers than
    // four CTAs per SM leave: three there.
    static constexpr int kMinBlocks = Staged ? 2 : (NT == 1 ? PKV_FP8_MIN_BLOCKS : 3);
    static constexpr uint32_t kSelEven = 0x2404u;  // bytes 0, 2 -> high bytes of two f16
    static constexpr uint32_t kSelOdd = 0x3414u;   // bytes 1, 3 -> high bytes of two f16
    // e4m3: byte 0 / 2 (or 1 / 3) into the low byte of each half, the sign of
    // that byte replicated over the half's high byte.
    static constexpr uint32_t kSignSelEven = 0xA280u;
    static constexpr uint32_t kSignSelOdd = 0xB391u;

    // Codes (bytes 0, 2) or (bytes 1, 3) of w as an f16x2 word.  e5m2 is the
    // high byte of the binary16 with the same value.  e4m3: the code's sign
    // to bit 15 and its 7 exponent/mantissa bits to bits 13..7 make a binary16
    // of exactly 2^-8 times the code's value, normal and subnormal codes alike
    // (both formats have 3 ... 10 mantissa bits and biases 7 / 15); the host
    // folds the 2^8 into the score and output scales (kE4m3Shift).  With the
    // sign replicated over the high byte, one shift by 7 puts the sign's
    // lowest copy at bit 15 and the 7 bits at 13..7; the mask drops the rest
    // (the code's own sign at bit 14, the other copies): three ALU operations
    // per pair of codes.
    __device__ static uint32_t widen(uint32_t w, bool odd)
    {
        if constexpr (KV == PKV_FP8_E5M2)
            return e5m2x2_to_f16x2(w, odd ? kSelOdd : kSelEven);  // codes in high bytes
        else
            return (prmt(w, 0u, odd ? kSignSelOdd : kSignSelEven) << 7) & 0xbf80bf80u;
    }

    struct Frags {
        uint32_t k[KS / 2][4];  // raw codes of 32 head_dim rows of K per entry
        uint32_t v[MT / 2][4];  // raw codes of 32 head_dim rows of V per entry
    };

    __device__ static void begin(State &st, const DecodeParams &p, const void *q, int s, int hkv,
                                 int lane, unsigned char *)
    {
        Base::reset(st);
        Base::template load_q_frags<true>(st, p, q, s, hkv, lane);
    }

    __device__ static void load(Frags &f, const unsigned char *sK, const unsigned char *sV,
                                int lane)
    {
        const int mi = lane >> 3, ri = lane & 7;
        // Both tiles: matrix mi of one ldmatrix.x4 is head_dim rows 8mi..8mi+7.
        const uint32_t ka = smem_u32(sK) + (8 * mi + ri) * 16;
        const uint32_t va = smem_u32(sV) + (8 * mi + ri) * 16;
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp)
            ldsm_x4_t(f.k[kp], ka + kp * 32 * 16);
#pragma unroll
        for (int mp = 0; mp < MT / 2; ++mp)
            ldsm_x4(f.v[mp], va + mp * 32 * 16);
    }

    __device__ static void compute(State &st, Frags &f, int valid, int lane, float c)
    {
        const int r = lane >> 2, cc = lane & 3;
        // S^T: A row r <-> token 2r, row r+8 <-> token 2r+1; two accumulation
        // chains (the two k steps of each ldmatrix.x4).
        float sacc[NT][4], sodd[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] = sodd[n][e] = 0.f;
#pragma unroll
        for (int kp = 0; kp < KS / 2; ++kp) {
            const uint32_t *w = f.k[kp];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t a[4] = {widen(w[2 * h], false), widen(w[2 * h], true),
                                       widen(w[2 * h + 1], false), widen(w[2 * h + 1], true)};
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    mma_f16(h ? sodd[n] : sacc[n], a, st.qf[2 * kp + h][n][0],
                            st.qf[2 * kp + h][n][1]);
            }
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] += sodd[n][e];

        // P^T: k slots (2c, 2c+1) <-> tokens (4c, 4c+2), (2c+8, 2c+9) <-> (4c+1, 4c+3).
        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float pr[4], alpha[2];
            if (MmaSoftmax::update(sacc[n], 2 * r, 2 * r + 1, valid, c, st.m[n], st.l[n], pr,
                                   alpha))
                Base::rescale(st, n, alpha);
            b0[n] = movmatrix_t(pack_f16(pr[0], pr[1]));
            b1[n] = movmatrix_t(pack_f16(pr[2], pr[3]));
        }

        uint32_t me = 0xffffffffu, mo = 0xffffffffu;
        if (valid < kBlockSize) {
            me = (4 * cc < valid ? 0x0000ffffu : 0u) | (4 * cc + 2 < valid ? 0xffff0000u : 0u);
            mo = (4 * cc + 1 < valid ? 0x0000ffffu : 0u) |
                 (4 * cc + 3 < valid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mp = 0; mp < MT / 2; ++mp) {
            const uint32_t *w = f.v[mp];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t a[4] = {widen(w[2 * h], false) & me, widen(w[2 * h + 1], false) & me,
                                       widen(w[2 * h], true) & mo, widen(w[2 * h + 1], true) & mo};
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    mma_f16(st.o[2 * mp + h][n], a, b0[n], b1[n]);
            }
        }
    }

    __device__ static void page(State &st, const unsigned char *sK, const unsigned char *sV,
                                int valid, int lane, int, unsigned char *, float c)
    {
        Frags f;
        load(f, sK, sV, lane);
        compute(st, f, valid, lane, c);
    }

    __device__ static void finish(State &st, float *so, float *sm, float *sl, int lane)
    {
        Base::finish(st, so, sm, sl, lane);
    }
};

// INT4 KV: the page tile is [D][8] bytes (token 2j of a head_dim row in the
// low nibble of byte j).  Fragments are gathered with byte / halfword loads
// in the fp8 policy's token order (fragment row r <-> token 2r, row r+8 <->
// token 2r+1), so one byte holds the two tokens a lane needs for a head_dim
// row; nibbles become exact binary16 integers with the 0x6400 exponent trick
// (1024 + (n ^ 8) - 1032 = the signed nibble).  Scales multiply outside.
template <int D, int NT, int Budget = compact_ring_budget(NT), bool Staged = false>
struct MmaInt4Policy : MmaStateBase<D, NT> {
    using Base = MmaStateBase<D, NT>;
    using State = typename Base::State;
    using RingT = Ring<PKV_INT4, D, Budget>;
    using StreamK = MmaInt4Policy<D, NT, ring_budget(scratch_bytes(8 * NT, D)), NT == 1>;
    static constexpr int R = RingT::R;
    static constexpr int kTileBytes = RingT::kTileBytes;
    static constexpr int kStageBytes = RingT::kStageBytes;
    static constexpr int kRingBytes = RingT::kRingBytes;
    static constexpr int kDim = D;
    static constexpr int GP = 8 * NT;
    static constexpr int kExtraBytes = 0;
    static constexpr int KS = Base::KS, MT = Base::MT;
    static constexpr bool kStaged = Staged;
    static constexpr bool kSharedBegin = false;
    static constexpr bool kSingleForm = true;
    static constexpr int kMinBlocks = Staged ? 2 : (NT == 1 ? PKV_FP8_MIN_BLOCKS : 3);
    static constexpr int kRow = kBlockSize / 2;  // bytes of one head_dim row

    // Low (odd = false) or high nibbles of the two bytes of y (bits 0-7 and
    // 16-23) as an f16x2 word of signed integers.  A low nibble n under the
    // 0x6400 exponent reads 1024 + (n ^ 8); a high nibble is masked in place,
    // reads 1024 + 16 (n ^ 8), and is scaled by 1/16 in the same (exact) FMA:
    // one ALU operation per pair either way, no shift.
    __device__ static uint32_t widen(uint32_t y, bool odd)
    {
        if (!odd) {
            const uint32_t h = (y & 0x000f000fu) ^ 0x64086408u;
            const __half2 v =
                __hsub2(*reinterpret_cast<const __half2 *>(&h),
                        __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));
            return *reinterpret_cast<const uint32_t *>(&v);
        }
        const uint32_t h = (y & 0x00f000f0u) ^ 0x64806480u;
        const __half2 sixteenth = __halves2half2(__ushort_as_half(0x2c00), __ushort_as_half(0x2c00));
        const __half2 minus72 = __halves2half2(__ushort_as_half(0xd480), __ushort_as_half(0xd480));
        const __half2 v = __hfma2(*reinterpret_cast<const __half2 *>(&h), sixteenth, minus72);
        return *reinterpret_cast<const uint32_t *>(&v);
    }

    // Each entry holds two bytes, at bits 0-7 and 16-23.
    struct Frags {
        uint32_t k[KS][2];  // per k step: bytes g of rows (d0, d0+1) and (d0+8, d0+9)
        uint32_t v[MT][2];  // per head_dim tile: bytes 2c, 2c+1 of rows g and g + 8
    };

    __device__ static void begin(State &st, const DecodeParams &p, const void *q, int s, int hkv,
                                 int lane, unsigned char *)
    {
        Base::reset(st);
        Base::template load_q_frags<true>(st, p, q, s, hkv, lane);
    }

    __device__ static void load(Frags &f, const unsigned char *sK, const unsigned char *sV,
                                int lane)
    {
        const int g = lane >> 2, c = lane & 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            // Bytes of two rows side by side: a multiply-add (FMA pipe), not a
            // byte permute (ALU pipe).
            const unsigned char *r = sK + (16 * ks + 2 * c) * kRow + g;
            f.k[ks][0] = static_cast<uint32_t>(r[kRow]) * 65536u + static_cast<uint32_t>(r[0]);
            f.k[ks][1] =
                static_cast<uint32_t>(r[9 * kRow]) * 65536u + static_cast<uint32_t>(r[8 * kRow]);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const unsigned char *r = sV + (16 * mt + g) * kRow + 2 * c;
            f.v[mt][0] = __byte_perm(*reinterpret_cast<const unsigned short *>(r), 0u, 0x4140u);
            f.v[mt][1] =
                __byte_perm(*reinterpret_cast<const unsigned short *>(r + 8 * kRow), 0u, 0x4140u);
        }
    }

    __device__ static void compute(State &st, Frags &f, int valid, int lane, float c)
    {
        const int r = lane >> 2, cc = lane & 3;
        float sacc[NT][4], sodd[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] = sodd[n][e] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint32_t a[4] = {widen(f.k[ks][0], false), widen(f.k[ks][0], true),
                                   widen(f.k[ks][1], false), widen(f.k[ks][1], true)};
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_f16((ks & 1) ? sodd[n] : sacc[n], a, st.qf[ks][n][0], st.qf[ks][n][1]);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sacc[n][e] += sodd[n][e];

        uint32_t b0[NT], b1[NT];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            float pr[4], alpha[2];
            if (MmaSoftmax::update(sacc[n], 2 * r, 2 * r + 1, valid, c, st.m[n], st.l[n], pr,
                                   alpha))
                Base::rescale(st, n, alpha);
            b0[n] = movmatrix_t(pack_f16(pr[0], pr[1]));
            b1[n] = movmatrix_t(pack_f16(pr[2], pr[3]));
        }
        // Past the sequence end the codes are finite and P is 0: no V mask.
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const uint32_t a[4] = {widen(f.v[mt][0], false), widen(f.v[mt][1], false),
                                   widen(f.v[mt][0], true), widen(f.v[mt][1], true)};
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_f16(st.o[mt][n], a, b0[n], b1[n]);
        }
        (void)cc;
    }

    __device__ static void page(State &st, const unsigned char *sK, const unsigned char *sV,
                                int valid, int lane, int, unsigned char *, float c)
    {
        Frags f;
        load(f, sK, sV, lane);
        compute(st, f, valid, lane, c);
    }

    __device__ static void finish(State &st, float *so, float *sm, float *sl, int lane)
    {
        Base::finish(st, so, sm, sl, lane);
    }
};

// ==================================================================== kernel

// Fused cache write.  The new token of a sequence is its position L - 1; its
// converted K/V rows are written into the cache slot and fenced against the
// copy engine's reads before the bulk copy of that page is issued, so the
// ordinary page copy brings the new token in with the rest.  The item
// kernel stages the rows at item start and writes them on the issue path of
// the page; the stream-K kernel writes all tokens of its range at start.
// Bytes of one warp's staging buffer for the new K and V rows (head_dim up
// to 128 elements of up to 4 bytes each, K then V).
constexpr int kNewRowBytes = 2 * 128 * 4;

// Starts copying the new K and V rows of (s, hkv) into `buf` (shared memory)
// without waiting; write_new_token_from(buf) consumes them.
__device__ __forceinline__ void prefetch_new_rows(const DecodeParams &p, const LayerPtrs &lt,
                                                  int s, int hkv, int D, unsigned char *buf,
                                                  int lane)
{
    const int eb = p.new_dtype == PKV_F32 ? 4 : 2;
    const int row_bytes = D * eb;  // multiple of 16
    const size_t src0 = (static_cast<size_t>(s) * p.num_kv_heads + hkv) * row_bytes;
    for (int c = lane; c < 2 * row_bytes / 16; c += 32) {
        const bool is_v = c * 16 >= row_bytes;
        const int off = c * 16 - (is_v ? row_bytes : 0);
        const unsigned char *src =
            static_cast<const unsigned char *>(is_v ? lt.new_v : lt.new_k) + src0 + off;
        cp_async_16(buf + (is_v ? row_bytes : 0) + off, src);
    }
    cp_async_commit();
}

// Writes the new token of (s, hkv) from the rows prefetch_new_rows staged in
// shared memory into slot (L - 1) % 16 of block phys, then fences the writes
// against the bulk copy of that page that follows.  kc_head / vc_head point
// at KV head hkv's tile of block 0 of the layer's caches.
__device__ __forceinline__ void write_new_token_from(const DecodeParams &p, const void *kc_head,
                                                     const void *vc_head, int hkv, int L,
                                                     int phys, int D, const unsigned char *buf,
                                                     int lane)
{
    cp_async_wait_all();
    __syncwarp();
    const int t = (L - 1) % kBlockSize;
    const int row_bytes = D * (p.new_dtype == PKV_F32 ? 4 : 2);
    const size_t dst0 = static_cast<size_t>(phys) * p.num_kv_heads * D;
    void *kc = const_cast<void *>(kc_head);
    void *vc = const_cast<void *>(vc_head);
    const float kq = unit_k_quant(p, hkv), vq = unit_v_quant(p, hkv);
    for (int d = lane; d < D; d += 32) {
        const size_t g = (dst0 + d) * kBlockSize + t;
        store_kv(kc, p.kv_dtype, g, buf, p.new_dtype, d, kq);
        store_kv(vc, p.kv_dtype, g, buf + row_bytes, p.new_dtype, d, vq);
    }
    fence_proxy_async_all();
    __syncwarp();
}

// The converted K/V rows of the listed new tokens stored into their slots,
// without a fence (the caller fences before the copies it orders).  Entry e
// of `w` is (s, hkv, L, phys, layer): that layer's rows new_k/new_v[s, hkv]
// go to slot (L - 1) % 16 of block phys of its caches.  Each lane handles
// head_dim elements lane + 32j; all loads of a pair of entries are issued
// before their stores.
template <bool kMulti>
__device__ __forceinline__ void write_token_rows(const DecodeParams &p, const int (*w)[5], int e0,
                                                 int n, int step, int D, int lane)
{
    constexpr int kJ = 4;  // head_dim <= 128
    for (int e = e0; e < n; e += 2 * step) {
        float kv[2][kJ], vv[2][kJ];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int ee = e + x * step;
            if (ee >= n)
                break;
            const LayerPtrs lt = layer_ptrs<kMulti>(p, w[ee][4]);
            const size_t src0 = (static_cast<size_t>(w[ee][0]) * p.num_kv_heads + w[ee][1]) * D;
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int d = lane + 32 * j;
                if (d < D) {
                    kv[x][j] = load_in(lt.new_k, p.new_dtype, src0 + d);
                    vv[x][j] = load_in(lt.new_v, p.new_dtype, src0 + d);
                }
            }
        }
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int ee = e + x * step;
            if (ee >= n)
                break;
            const int t = (w[ee][2] - 1) % kBlockSize;
            const size_t dst0 = (static_cast<size_t>(w[ee][3]) * p.num_kv_heads + w[ee][1]) * D;
            const float kq = unit_k_quant(p, w[ee][1]), vq = unit_v_quant(p, w[ee][1]);
            const LayerPtrs lt = layer_ptrs<kMulti>(p, w[ee][4]);
            void *kc = lt.k_cache;
            void *vc = lt.v_cache;
#pragma unroll
            for (int j = 0; j < kJ; ++j) {
                const int d = lane + 32 * j;
                if (d < D) {
                    const size_t g = (dst0 + d) * kBlockSize + t;
                    store_kv_value(kc, p.kv_dtype, g, kv[x][j], kq);
                    store_kv_value(vc, p.kv_dtype, g, vv[x][j], vq);
                }
            }
        }
    }
}


// Item phases of the partitioned schedule: every full partition first, then
// the remainders -- at most one per sequence, shorter than a partition --
// in size classes, largest first (three: remainder >= 2P/3, >= P/3, the
// rest, which includes the single item of an empty sequence).  Handing out the
// largest items first and the shortest last leaves the grid's final wave
// with short items.
// Remainder size classes (same box, 70B bf16 / e4m3 / INT4 layers at
// 4096-token partitions, us): three 230.2 / 124.6 / 143.2, five 229.8 /
// 125.8 / 142.5, eight 236.4 / 129.3 / 144.1.
#ifndef PKV_REMAINDER_CLASSES
#define PKV_REMAINDER_CLASSES 3
#endif
constexpr int kPhases = 1 + PKV_REMAINDER_CLASSES;
__device__ __forceinline__ int full_parts(int L, int P) { return L / P; }
__device__ __forceinline__ int phase_parts(int L, int P, int ph)
{
    if (ph == 0)
        return L / P;
    const int r = L % P;
    if (r == 0 && L != 0)
        return 0;  // no remainder
    constexpr int nc = kPhases - 1;
    const int cls = 1 + (nc - 1) - static_cast<int>((static_cast<long long>(r) * nc) / P);
    return cls == ph ? 1 : 0;
}

// Warp-collective scan over sequences: finds the sequence holding unit u of
// phase ph, in which sequence s contributes phase_parts(L_s) units.
// `cur_s` / `cur_base` remember where the previous search of that phase
// ended (u only grows).  Returns false when u lies past the last sequence.
__device__ inline bool find_unit(const DecodeParams &p, int u, int ph, int &cur_s,
                                 int &cur_base, int lane, int &s_out, int &k_out, int &L_out)
{
    const int S = p.num_seqs, P = p.partition;
    for (;;) {
        const int sl = cur_s + lane;
        int n = 0, Ls = 0;
        if (sl < S) {
            Ls = seq_len_of(p, sl);
            n = phase_parts(Ls, P, ph);
        }
        int incl = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off)
                incl += t;
        }
        const int tot = __shfl_sync(kFullMask, incl, 31);
        if (u < cur_base + tot) {
            const unsigned bal = __ballot_sync(kFullMask, cur_base + incl > u);
            const int ln = __ffs(bal) - 1;
            const int excl = __shfl_sync(kFullMask, incl - n, ln);
            s_out = cur_s + ln;
            k_out = u - cur_base - excl;
            L_out = __shfl_sync(kFullMask, Ls, ln);
            return true;
        }
        if (cur_s + 32 >= S)
            return false;
        cur_base += tot;
        cur_s += 32;
    }
}

// Items of each phase over all sequences of one layer (warp-collective).
__device__ __forceinline__ void count_phases(const DecodeParams &p, int lane, int (&n)[kPhases])
{
#pragma unroll
    for (int ph = 0; ph < kPhases; ++ph)
        n[ph] = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
        int L = 0;
        const bool in = s0 + lane < p.num_seqs;
        if (in)
            L = seq_len_of(p, s0 + lane);
#pragma unroll
        for (int ph = 0; ph < kPhases; ++ph) {
            int c = in ? phase_parts(L, p.partition, ph) : 0;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                c += __shfl_xor_sync(kFullMask, c, off);
            n[ph] += c;
        }
    }
}

// Combines the four warps' (m, l, O) states of one item (at the start of each
// warp's ring) and writes the output rows of `out` (one partition) or the
// item's normalised partial (split sequences; gs = layer * S + s).
template <int D, int GP>
__device__ void merge_item(const DecodeParams &p, void *out, const unsigned char *smem,
                           int ring_bytes, int s, int gs, int hkv, int part, int nparts)
{
    constexpr int Q4 = D / 4;
    const int G = p.group;
    for (int idx = threadIdx.x; idx < G * Q4; idx += kThreads) {
        const int g = idx / Q4, q4 = idx - g * Q4;
        float mw[kWarps], mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *sm = reinterpret_cast<const float *>(smem + w * ring_bytes) + GP * D;
            mw[w] = sm[g];
            mx = fmaxf(mx, mw[w]);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *so = reinterpret_cast<const float *>(smem + w * ring_bytes);
            const float f = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - mx);
            const float4 o = reinterpret_cast<const float4 *>(so + g * D)[q4];
            acc.x += f * o.x;
            acc.y += f * o.y;
            acc.z += f * o.z;
            acc.w += f * o.w;
            lsum += f * so[GP * D + GP + g];
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int h = hkv * G + g;
        if (nparts == 1) {
            const float sc = inv * unit_out_scale(p, hkv);
            store_out4(p, out, D, s, h, q4,
                       make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc));
        } else {
            const size_t row = (static_cast<size_t>(gs) * p.num_q_heads + h) * p.max_parts + part;
            reinterpret_cast<float4 *>(p.part_o + row * D)[q4] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (q4 == 0) {
                p.part_ml[2 * row] = mx;
                p.part_ml[2 * row + 1] = lsum;
            }
        }
    }
}

// kMulti = false: the form for single-layer calls, with the layer logic
// compiled out (tensor-core policies); true: any number of layers.
template <class Pol, bool kMulti>
__global__ void __launch_bounds__(kThreads, Pol::kMinBlocks)
    decode_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int D = Pol::kDim;
    static_assert((Pol::GP * D + 2 * Pol::GP) * 4 <= Pol::kRingBytes,
                  "merge scratch must fit in one warp's ring");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_item[8];
    // Warp 0's item scheduler (kept in shared memory, not registers, across
    // the page loop): scan cursors of the item phases (reset when the layer
    // changes) and the per-layer item counts of the phases.
    __shared__ int s_sched[4 * kPhases];
    __shared__ int s_abort;
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned char *ring = smem + warp * Pol::kRingBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kWarps * Pol::kRingBytes) + warp * Pol::R;
    unsigned char *extra = smem + kWarps * Pol::kRingBytes + kWarps * Pol::R * sizeof(uint64_t);
    unsigned char *newrow = extra + Pol::kExtraBytes + warp * kNewRowBytes;

    if (lane == 0)
        for (int st = 0; st < Pol::R; ++st)
            mbar_init(&bars[st], 1);
    if (threadIdx.x == 0)
        s_abort = 0;
    fence_mbar_init();
    __syncthreads();

    const int Hkv = p.num_kv_heads;
    const int S = p.num_seqs;
    const int P = p.partition;
    const size_t tile_stride = static_cast<size_t>(Pol::kTileBytes);
    const size_t block_stride = static_cast<size_t>(Hkv) * tile_stride;

    uint32_t pages_done = 0;  // pages this warp has consumed (ring position / phase)
    // s_sched: per phase ph, scan cursor (sequence, base) at 2 ph and
    // 2 ph + 1, the layer the cursor belongs to at kLayer + ph, and the
    // phase's item count per layer at kCount + ph.
    enum { kLayer = 2 * kPhases, kCount = 3 * kPhases };
    if (p.split && warp == 0) {
        int n[kPhases];
        count_phases(p, lane, n);
        if (lane == 0)
            for (int ph = 0; ph < kPhases; ++ph) {
                s_sched[2 * ph] = s_sched[2 * ph + 1] = 0;
                s_sched[kLayer + ph] = 0;
                s_sched[kCount + ph] = n[ph];
            }
        __syncwarp();
    }
    bool first = true;

    for (;;) {
        // ---------------------------------------------- next work item
        if (warp == 0) {
            int s = 0, part = 0, hkv = 0, L = 0, nparts = 1, item = 0, done = 0, layer = 0;
            if (p.split && !kMulti) {
                unsigned v = 0;
                if (lane == 0)
                    v = atomicAdd(p.counter, 1u);
                item = static_cast<int>(__shfl_sync(kFullMask, v, 0));
                // The phases in order: full partitions, then the remainders
                // by size class.
                int u = item / Hkv;
                hkv = item - u * Hkv;
                int ph = 0;
                while (ph < kPhases - 1 && u >= s_sched[kCount + ph]) {
                    u -= s_sched[kCount + ph];
                    ++ph;
                }
                int cs = s_sched[2 * ph], cb = s_sched[2 * ph + 1], k = 0;
                const bool found = find_unit(p, u, ph, cs, cb, lane, s, k, L);
                part = ph ? full_parts(L, P) : k;
                __syncwarp();
                if (lane == 0) {
                    s_sched[2 * ph] = cs;
                    s_sched[2 * ph + 1] = cb;
                }
                done = found ? 0 : 1;
                nparts = parts_of(L, P);
            } else if (p.split) {
                unsigned v = 0;
                if (lane == 0)
                    v = atomicAdd(p.counter, 1u);
                item = static_cast<int>(__shfl_sync(kFullMask, v, 0));
                // The phases in order, every layer's items of a phase before
                // the next phase; layer-major inside each phase.
                long r = item;
                int ph = 0;
                while (ph < kPhases - 1 &&
                       r >= static_cast<long>(s_sched[kCount + ph]) * Hkv * p.num_layers) {
                    r -= static_cast<long>(s_sched[kCount + ph]) * Hkv * p.num_layers;
                    ++ph;
                }
                const long per = static_cast<long>(s_sched[kCount + ph]) * Hkv;
                layer = per > 0 ? static_cast<int>(r / per) : p.num_layers;
                bool found = false;
                if (layer < p.num_layers) {
                    r -= static_cast<long>(layer) * per;
                    const int u = static_cast<int>(r / Hkv);
                    hkv = static_cast<int>(r - static_cast<long>(u) * Hkv);
                    int k = 0;
                    int cs = s_sched[2 * ph], cb = s_sched[2 * ph + 1];
                    if (layer != s_sched[kLayer + ph])
                        cs = cb = 0;
                    found = find_unit(p, u, ph, cs, cb, lane, s, k, L);
                    part = ph ? full_parts(L, P) : k;
                    __syncwarp();
                    if (lane == 0) {
                        s_sched[2 * ph] = cs;
                        s_sched[2 * ph + 1] = cb;
                        s_sched[kLayer + ph] = layer;
                    }
                }
                done = found ? 0 : 1;
                nparts = parts_of(L, P);
            } else {
                item = first ? static_cast<int>(blockIdx.x) : INT_MAX;
                if (item >= S * Hkv * (kMulti ? p.num_layers : 1)) {
                    done = 1;
                } else {
                    layer = kMulti ? item / (S * Hkv) : 0;
                    const int r = item - layer * (S * Hkv);
                    s = r / Hkv;
                    hkv = r - s * Hkv;
                    L = seq_len_of(p, s);
                }
            }
            if (lane == 0) {
                s_item[0] = s;
                s_item[1] = part;
                s_item[2] = hkv;
                s_item[3] = L;
                s_item[4] = nparts;
                s_item[5] = item;
                s_item[6] = done;
                s_item[7] = layer;
            }
        }
        first = false;
        __syncthreads();
        if (s_item[6])
            break;
        const int s = s_item[0], part = s_item[1], hkv = s_item[2], L = s_item[3];
        const int nparts = s_item[4], item = s_item[5], layer = s_item[7];
        const LayerPtrs lt = layer_ptrs<kMulti>(p, layer);
        if (!layer_usable<kMulti>(p, lt)) {  // uniform: every thread reads the same entry
            if (threadIdx.x == 0)
                set_status(p.status, PKV_ERR_INVALID_ARG);
            __syncthreads();  // s_item is rewritten for the next item
            continue;
        }
        const float c = unit_score_scale(p, hkv);

        // ---------------------------------------------- this warp's pages
        const int t0 = part * P;
        const int t1 = min(L, t0 + P);
        const int pg0 = t0 / kBlockSize;
        const int npages = t1 > t0 ? (t1 - t0 + kBlockSize - 1) / kBlockSize : 0;
        const int nw = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;
        const int32_t *bt = p.block_tables + static_cast<size_t>(s) * p.max_blocks + pg0 + warp;
        const size_t head_off = static_cast<size_t>(hkv) * tile_stride;
        const unsigned char *kbase = static_cast<const unsigned char *>(lt.k_cache) + head_off;
        const unsigned char *vbase = static_cast<const unsigned char *>(lt.v_cache) + head_off;

        int id_reg = -1, id_chunk = -1;
        uint32_t okmask = 0;
        // Warp-collective: physical id of this warp's page i (32 ids per load).
        auto page_id = [&](int i) -> int {
            const int ch = i >> 5;
            if (ch != id_chunk) {
                const int j = (ch << 5) + lane;
                id_reg = j < nw ? __ldg(bt + kWarps * j) : -1;
                id_chunk = ch;
            }
            return __shfl_sync(kFullMask, id_reg, i & 31);
        };
        // Fused cache write: the warp that owns the sequence's last page
        // stages the new rows now and writes them just before that page's
        // copy is issued.
        const int i_new = (p.append && lt.new_k != nullptr && t1 == L && L > 0 && npages > 0 &&
                           (npages - 1) % kWarps == warp)
                              ? (npages - 1) / kWarps
                              : -1;
        if (i_new >= 0)
            prefetch_new_rows(p, lt, s, hkv, D, newrow, lane);
        auto issue = [&](int i) {
            const int phys = page_id(i);
            const int stg = (pages_done + i) % Pol::R;
            const bool ok = phys >= 0 && phys < p.num_blocks;
            if (i == i_new && ok)
                write_new_token_from(p, kbase, vbase, hkv, L, phys, D, newrow, lane);
            okmask = ok ? (okmask | (1u << stg)) : (okmask & ~(1u << stg));
            if (lane == 0) {
                uint64_t *bar = &bars[stg];
                if (!ok) {
                    set_status(p.status, PKV_ERR_OUT_OF_RANGE);
                    mbar_arrive(bar);
                } else {
                    mbar_arrive_expect_tx(bar, 2 * Pol::kTileBytes);
                    const bool drop = p.drop_first_copy && item == 0 && warp == 0 && i == 0;
                    if (!drop) {
                        const size_t off = static_cast<size_t>(phys) * block_stride;
                        unsigned char *dst = ring + stg * Pol::kStageBytes;
                        bulk_g2s(dst, kbase + off, Pol::kTileBytes, bar);
                        bulk_g2s(dst + Pol::kTileBytes, vbase + off, Pol::kTileBytes, bar);
                    }
                }
            }
        };

        int issued = 0;
        const int pre = nw < Pol::R ? nw : Pol::R;
        for (; issued < pre; ++issued)
            issue(issued);

        typename Pol::State st;
        {
            const int qrow = unit_row(p, s);  // s, or the routed query's row
            Pol::begin(st, p, qrow >= 0 ? lt.q : nullptr, qrow >= 0 ? qrow : 0, hkv, lane,
                       extra);
        }
        __syncthreads();  // policy shared data (SIMT query) is ready

        for (int i = 0; i < nw; ++i) {
            const uint32_t n = pages_done + i;
            const int stg = n % Pol::R;
            const uint32_t parity = (n / Pol::R) & 1u;
            const bool ok = mbar_wait_bounded(&bars[stg], parity, kWaitLimitNs);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) {
                    set_status(p.status, PKV_ERR_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                // Let every other copy already in flight land before leaving.
                for (int j = i + 1; j < issued; ++j) {
                    const uint32_t n2 = pages_done + j;
                    mbar_wait_bounded(&bars[n2 % Pol::R], (n2 / Pol::R) & 1u, kWaitLimitNs);
                }
                break;
            }
            const bool have = (okmask >> stg) & 1u;
            const int tok0 = (pg0 + warp + kWarps * i) * kBlockSize;
            const int valid = min(kBlockSize, t1 - tok0);
            const unsigned char *sk = ring + stg * Pol::kStageBytes;
            typename Pol::Frags fr;
            if (have) {
                if constexpr (Pol::kStaged)
                    Pol::load(fr, sk, sk + Pol::kTileBytes, lane);
                else
                    Pol::page(st, sk, sk + Pol::kTileBytes, valid, lane, warp, extra, c);
            }
            // The stage is free: reads are ordered before the next bulk copy.
            fence_proxy_async();
            __syncwarp();
            if (issued < nw) {
                issue(issued);
                ++issued;
            }
            if constexpr (Pol::kStaged)
                if (have)
                    Pol::compute(st, fr, valid, lane, c);
        }
        pages_done += nw;
        if (i_new >= 0)
            cp_async_wait_all();  // staged rows landed even if their page was skipped

        // ---------------------------------------------- merge the warps
        {
            float *so = reinterpret_cast<float *>(ring);
            float *sm = so + Pol::GP * D;
            float *sl = sm + Pol::GP;
            Pol::finish(st, so, sm, sl, lane);
        }
        __syncthreads();
        // The item's coordinates again from shared memory (unchanged until
        // the next item), rather than registers held across the page loop.
        const int ms = s_item[0], mpart = s_item[1], mhkv = s_item[2], mnparts = s_item[4];
        const int mlayer = kMulti ? s_item[7] : 0;
        const int gs = mlayer * S + ms;  // workspace index of (layer, sequence)
        void *out = layer_ptrs<kMulti>(p, mlayer).out;
        merge_item<D, Pol::GP>(p, out, smem, Pol::kRingBytes, ms, gs, mhkv, mpart, mnparts);
        if (mnparts > 1 && p.fused_merge) {
            // Publish this partial; the CTA that completes the sequence's last
            // partial merges all of them.  The barrier orders every thread's
            // partial writes before thread 0's gpu-scope fence and arrival.
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                const unsigned old =
                    atomicAdd(p.arrive + static_cast<size_t>(gs) * Hkv + mhkv, 1u);
                s_last = (old == static_cast<unsigned>(mnparts - 1)) ? 1 : 0;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                merge_partials<D>(p, out, ms, gs, mhkv, mnparts);
            }
        }
        // The rings were used as generic scratch: order that before the next
        // item's bulk copies into them.
        fence_proxy_async();
        __syncthreads();
        if (*static_cast<volatile int *>(&s_abort))
            break;
    }
}

template <class Pol>
constexpr int decode_smem_bytes()
{
    return kWarps * Pol::kRingBytes + kWarps * Pol::R * 8 + Pol::kExtraBytes +
           kWarps * kNewRowBytes;
}

// Launches decode_kernel<Pol, kMulti>: one CTA per item without split, else a
// persistent grid sized from the occupancy of this instantiation.
template <class Pol, bool kMulti>
pkv_status launch_policy(const DecodeParams &p, cudaStream_t stream)
{
    constexpr int smem = decode_smem_bytes<Pol>();
    // Resident CTAs per SM, once the shared-memory attribute is set (per context).
    static ContextCache cache;
    int occ = 1;
    const pkv_status rc = cache.get(&occ, [](int *v) -> pkv_status {
        if (cudaFuncSetAttribute(decode_kernel<Pol, kMulti>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, decode_kernel<Pol, kMulti>, kThreads,
                                                          smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        *v = o > 0 ? o : 1;
        return PKV_OK;
    });
    if (rc != PKV_OK)
        return rc;
    long grid;
    if (p.split) {
        const long items =
            static_cast<long>(p.num_layers) * p.num_seqs * p.num_kv_heads * p.max_parts;
        const long slots = static_cast<long>(occ) * device_sm_count();
        grid = items < slots ? items : slots;
    } else {
        grid = static_cast<long>(p.num_layers) * p.num_seqs * p.num_kv_heads;
    }
    if (grid <= 0)
        return PKV_OK;
    decode_kernel<Pol, kMulti><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
