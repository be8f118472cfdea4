// Paged attention of several query tokens per sequence for sm_103a: chunked
// prefill and speculative verification, on mma.sync tensor-core fragments.
// The automatic kernel is the tcgen05 form in pkv_prefill_tc.cu; this one
// runs with PKV_FLAG_IMPL_MMA.  launch_prefill (end of file) picks between
// them; the log-sum-exp merge of split rows serves both.
//
// What is computed: the block-table walk of the PagedAttention kernel
// pseudocode ("vLLM e PagedAttention: serving high-throughput") with the
// causal mask of the "Inference optimization" lesson (Step 2,
// scaled_dot_product_attention, triu mask of offset
// seq_len_k - seq_len_q + 1).  The n queries of a sequence of L cached tokens
// are its last n positions; query i attends the rows t <= L - n + i.
//
// How it is laid out on the GPU (not taken from the pages):
//  * A row is one (query token, grouped query head) pair; the n * G rows of
//    (sequence, KV head) are cut into blocks of up to 64.  A work item is
//    (sequence, KV head, partition of the context, row block); every K/V
//    page the item needs crosses HBM once for all of its rows.
//  * A persistent grid pulls items from an atomic counter.  The CTA's four
//    warps stream the item's pages through one shared ring of bulk (TMA)
//    copies: lane 0 of warp 0 issues them in page order; a full barrier per
//    stage carries the copied bytes, an empty barrier per stage counts the
//    warps that have read it.  Every wait is bounded.
//  * Each warp owns a 16-row tile (two 8-wide MMA N tiles).  With fewer than
//    64 rows the spare warps split the pages instead: warp w takes row tile
//    w % RT and every PG-th page, RT * PG = 4.
//  * Per page and warp, S^T = K^T Q^T and O^T = V P^T run on mma.sync as in
//    the decode kernel; the causal limit of each row masks its scores.
//  * The warps' softmax states are merged through shared memory at the end
//    of the item.  A row whose visible context fits one partition is written
//    to `out`; the others leave normalised partials (o, m, l) that
//    prefill_merge_kernel combines with log-sum-exp weights.
#include "pkv_prefill.cuh"

namespace pkv {

namespace {

constexpr int kRowTile = 16;                  // rows per warp tile
// Rows per work item (a multiple of 16, at most four warp tiles).
#ifndef PKV_PREFILL_ROW_BLOCK
#define PKV_PREFILL_ROW_BLOCK (kWarps * kRowTile)
#endif
constexpr int kRowBlock = PKV_PREFILL_ROW_BLOCK;
static_assert(kRowBlock % kRowTile == 0 && kRowBlock <= kWarps * kRowTile, "row block");
// Page ring per CTA and the CTAs per SM the registers are bounded for.
// Three CTAs with 64 KB rings (168 registers, fragments read from the stage)
// beat two with 96 KB rings by 20-25% (measured on GB300: 70B layer with five
// queries per sequence 894 -> 695 us); four would spill.
#ifndef PKV_PREFILL_RING_BYTES
#define PKV_PREFILL_RING_BYTES (64 * 1024)
#endif
#ifndef PKV_PREFILL_MIN_CTAS
#define PKV_PREFILL_MIN_CTAS 3
#endif
constexpr int kPrefillRingBytes = PKV_PREFILL_RING_BYTES;

template <int KV, int D> struct PrefillGeom {
    static constexpr int kTileBytes = tile_bytes(KV, D);   // one K or V page tile
    static constexpr int kStageBytes = 2 * kTileBytes;     // K then V
    static constexpr int NS = kPrefillRingBytes / kStageBytes;
    static constexpr int kRingBytes = NS * kStageBytes;
    static constexpr int kScratchFloats = kRowTile * D + 2 * kRowTile;  // O, m, l of a warp
    static constexpr int kSmem = kRingBytes + 2 * NS * 8;
    static_assert(kWarps * kScratchFloats * 4 <= kRingBytes, "merge scratch fits in the ring");
    static_assert((kScratchFloats * 4) % 16 == 0, "warp scratch keeps float4 alignment");
};

__device__ __forceinline__ void mbar_inval(uint64_t *bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Online-softmax update of one N tile with a per-row visibility limit: token
// tok of the page is seen by row column e when tok < lim[e].
__device__ __forceinline__ bool causal_update(const float (&sacc)[4], int tokA, int tokB,
                                              const int (&lim)[2], float c, float (&m)[2],
                                              float (&l)[2], float (&pr)[4], float (&alpha)[2])
{
    const bool a0 = tokA < lim[0], a1 = tokA < lim[1];
    const bool b0 = tokB < lim[0], b1 = tokB < lim[1];
    const float s0 = a0 ? sacc[0] * c : -INFINITY;
    const float s1 = a1 ? sacc[1] * c : -INFINITY;
    const float s2 = b0 ? sacc[2] * c : -INFINITY;
    const float s3 = b1 ? sacc[3] * c : -INFINITY;
    constexpr float kLazy = MmaSoftmax::kLazy;
    const bool fast = s0 <= m[0] + kLazy && s2 <= m[0] + kLazy && s1 <= m[1] + kLazy &&
                      s3 <= m[1] + kLazy;
    if (__all_sync(kFullMask, fast)) {
        // A row that has seen nothing yet keeps m = -inf: its masked scores
        // give p = 0 explicitly (never 2^(-inf - -inf)).
        pr[0] = a0 ? MmaSoftmax::ex2(s0 - m[0]) : 0.f;
        pr[1] = a1 ? MmaSoftmax::ex2(s1 - m[1]) : 0.f;
        pr[2] = b0 ? MmaSoftmax::ex2(s2 - m[0]) : 0.f;
        pr[3] = b1 ? MmaSoftmax::ex2(s3 - m[1]) : 0.f;
        l[0] += pr[0] + pr[2];
        l[1] += pr[1] + pr[3];
        return false;
    }
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFullMask, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFullMask, mx1, off));
    }
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    alpha[0] = (m[0] == -INFINITY) ? 0.f : MmaSoftmax::ex2(m[0] - mn0);
    alpha[1] = (m[1] == -INFINITY) ? 0.f : MmaSoftmax::ex2(m[1] - mn1);
    pr[0] = a0 ? MmaSoftmax::ex2(s0 - mn0) : 0.f;
    pr[1] = a1 ? MmaSoftmax::ex2(s1 - mn1) : 0.f;
    pr[2] = b0 ? MmaSoftmax::ex2(s2 - mn0) : 0.f;
    pr[3] = b1 ? MmaSoftmax::ex2(s3 - mn1) : 0.f;
    l[0] = l[0] * alpha[0] + pr[0] + pr[2];
    l[1] = l[1] * alpha[1] + pr[1] + pr[3];
    m[0] = mn0;
    m[1] = mn1;
    return true;
}

// One page for one warp's 16 rows: scores, causal softmax, P V, with the
// fragments read straight from the stage: K per k step while S^T
// accumulates, V after the softmax, so the two sets are never live together
// (the caller holds the stage until this returns).  `lim` holds the
// visible-token count of the page for each of the lane's four row columns;
// NT = 1 when the tile's rows all sit in its first 8-row N tile (the second
// tile's state then stays empty).
template <int D, int NT>
__device__ __forceinline__ void prefill_page_smem(typename MmaStateBase<D, 2>::State &st,
                                                  const unsigned char *sK,
                                                  const unsigned char *sV, int valid,
                                                  const int (&lim)[2][2], int lane, float c)
{
    using Base = MmaStateBase<D, 2>;
    constexpr int KS = Base::KS, MT = Base::MT;
    const int r = lane >> 2, cc = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const uint32_t ka = smem_u32(sK) + (ri + 8 * (mi >> 1)) * 32 + (mi & 1) * 16;
    const uint32_t va = smem_u32(sV) + (ri + 8 * (mi & 1)) * 32 + (mi >> 1) * 16;
    float sacc[NT][4], sodd[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sacc[n][e] = sodd[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        uint32_t kf[4];
        ldsm_x4_t(kf, ka + ks * 16 * 32);
#pragma unroll
        for (int n = 0; n < NT; ++n)
            mma_bf16((ks & 1) ? sodd[n] : sacc[n], kf, st.qf[ks][n][0], st.qf[ks][n][1]);
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sacc[n][e] += sodd[n][e];

    uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        float pr[4], alpha[2];
        if (causal_update(sacc[n], r, r + 8, lim[n], c, st.m[n], st.l[n], pr, alpha))
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
    uint32_t vf[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
        ldsm_x4(vf[mt], va + mt * 16 * 32);
    if (valid < kBlockSize) {  // past the sequence end: zero V (may hold NaN)
        const uint32_t mlo = (2 * cc < valid ? 0x0000ffffu : 0u) |
                             (2 * cc + 1 < valid ? 0xffff0000u : 0u);
        const uint32_t mhi = (8 + 2 * cc < valid ? 0x0000ffffu : 0u) |
                             (9 + 2 * cc < valid ? 0xffff0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            vf[mt][0] &= mlo;
            vf[mt][1] &= mlo;
            vf[mt][2] &= mhi;
            vf[mt][3] &= mhi;
        }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n)
            mma_bf16(st.o[mt][n], vf[mt], bh0[n], bh1[n]);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int n = 0; n < NT; ++n)
            mma_bf16(st.o[mt][n], vf[mt], bl0[n], bl1[n]);
}

// fp8 (e5m2 / e4m3) page for one warp's 16 rows: the decode fp8 policy's
// fragments (codes widened to f16 in registers; S^T row r <-> page token 2r,
// row r + 8 <-> token 2r + 1, and the matching P^T slots), the per-row causal
// limit of causal_update, and V zeroed past the sequence end.  K fragments
// are read before the softmax and V fragments after it.
template <int KV, int D, int NT>
__device__ __forceinline__ void prefill_page_fp8(typename MmaStateBase<D, 2>::State &st,
                                                 const unsigned char *sK,
                                                 const unsigned char *sV, int valid,
                                                 const int (&lim)[2][2], int lane, float c)
{
    using Base = MmaStateBase<D, 2>;
    using Pol = MmaFp8Policy<D, 1, compact_ring_budget(1), false, KV>;  // widening only
    constexpr int KS = Base::KS, MT = Base::MT;
    const int r = lane >> 2, cc = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    float sacc[NT][4], sodd[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sacc[n][e] = sodd[n][e] = 0.f;
    const uint32_t ka = smem_u32(sK) + (8 * mi + ri) * 16;
#pragma unroll
    for (int kp = 0; kp < KS / 2; ++kp) {
        uint32_t w[4];
        ldsm_x4_t(w, ka + kp * 32 * 16);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t a[4] = {Pol::widen(w[2 * h], false), Pol::widen(w[2 * h], true),
                                   Pol::widen(w[2 * h + 1], false), Pol::widen(w[2 * h + 1], true)};
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
    uint32_t b0[NT], b1[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        float pr[4], alpha[2];
        if (causal_update(sacc[n], 2 * r, 2 * r + 1, lim[n], c, st.m[n], st.l[n], pr, alpha))
            Base::rescale(st, n, alpha);
        b0[n] = movmatrix_t(pack_f16(pr[0], pr[1]));
        b1[n] = movmatrix_t(pack_f16(pr[2], pr[3]));
    }
    // P^T slots (2c, 2c+1) <-> tokens (4c, 4c+2), (2c+8, 2c+9) <-> (4c+1, 4c+3).
    uint32_t me = 0xffffffffu, mo = 0xffffffffu;
    if (valid < kBlockSize) {  // past the sequence end: zero V (may hold NaN)
        me = (4 * cc < valid ? 0x0000ffffu : 0u) | (4 * cc + 2 < valid ? 0xffff0000u : 0u);
        mo = (4 * cc + 1 < valid ? 0x0000ffffu : 0u) | (4 * cc + 3 < valid ? 0xffff0000u : 0u);
    }
    const uint32_t va = smem_u32(sV) + (8 * mi + ri) * 16;
#pragma unroll
    for (int mp = 0; mp < MT / 2; ++mp) {
        uint32_t w[4];
        ldsm_x4(w, va + mp * 32 * 16);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t a[4] = {Pol::widen(w[2 * h], false) & me,
                                   Pol::widen(w[2 * h + 1], false) & me,
                                   Pol::widen(w[2 * h], true) & mo,
                                   Pol::widen(w[2 * h + 1], true) & mo};
#pragma unroll
            for (int n = 0; n < NT; ++n)
                mma_f16(st.o[2 * mp + h][n], a, b0[n], b1[n]);
        }
    }
}

// INT4 page for one warp's 16 rows: the decode INT4 policy's fragments
// (nibble pairs gathered with byte / halfword loads and widened to exact f16
// integers; same token order as fp8) with the per-row causal limit.  Codes
// past the sequence end are finite and P is 0 there: no V mask.
template <int D, int NT>
__device__ __forceinline__ void prefill_page_int4(typename MmaStateBase<D, 2>::State &st,
                                                  const unsigned char *sK,
                                                  const unsigned char *sV,
                                                  const int (&lim)[2][2], int lane, float c)
{
    using Base = MmaStateBase<D, 2>;
    using Pol = MmaInt4Policy<D, 1>;  // widening only
    constexpr int KS = Base::KS, MT = Base::MT;
    constexpr int kRow = Pol::kRow;
    const int r = lane >> 2, cc = lane & 3;
    float sacc[NT][4], sodd[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e)
            sacc[n][e] = sodd[n][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const unsigned char *row = sK + (16 * ks + 2 * cc) * kRow + r;
        const uint32_t k0 = static_cast<uint32_t>(row[kRow]) * 65536u +
                            static_cast<uint32_t>(row[0]);
        const uint32_t k1 = static_cast<uint32_t>(row[9 * kRow]) * 65536u +
                            static_cast<uint32_t>(row[8 * kRow]);
        const uint32_t a[4] = {Pol::widen(k0, false), Pol::widen(k0, true), Pol::widen(k1, false),
                               Pol::widen(k1, true)};
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
        if (causal_update(sacc[n], 2 * r, 2 * r + 1, lim[n], c, st.m[n], st.l[n], pr, alpha))
            Base::rescale(st, n, alpha);
        b0[n] = movmatrix_t(pack_f16(pr[0], pr[1]));
        b1[n] = movmatrix_t(pack_f16(pr[2], pr[3]));
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        const unsigned char *row = sV + (16 * mt + r) * kRow + 2 * cc;
        const uint32_t v0 = __byte_perm(*reinterpret_cast<const unsigned short *>(row), 0u, 0x4140u);
        const uint32_t v1 =
            __byte_perm(*reinterpret_cast<const unsigned short *>(row + 8 * kRow), 0u, 0x4140u);
        const uint32_t a[4] = {Pol::widen(v0, false), Pol::widen(v1, false), Pol::widen(v0, true),
                               Pol::widen(v1, true)};
#pragma unroll
        for (int n = 0; n < NT; ++n)
            mma_f16(st.o[mt][n], a, b0[n], b1[n]);
    }
}

// One page of one warp's row tile in the cache's dtype.
template <int KV, int D, int NT>
__device__ __forceinline__ void prefill_page(typename MmaStateBase<D, 2>::State &st,
                                             const unsigned char *sK, const unsigned char *sV,
                                             int valid, const int (&lim)[2][2], int lane, float c)
{
    if constexpr (KV == PKV_BF16)
        prefill_page_smem<D, NT>(st, sK, sV, valid, lim, lane, c);
    else if constexpr (KV == PKV_INT4)
        prefill_page_int4<D, NT>(st, sK, sV, lim, lane, c);
    else
        prefill_page_fp8<KV, D, NT>(st, sK, sV, valid, lim, lane, c);
}

__device__ __forceinline__ void store_row4(const PrefillParams &p, int D, int token, int h,
                                           int q4, float4 v)
{
    const size_t off = (static_cast<size_t>(token) * p.num_q_heads + h) * D + 4 * q4;
    if (p.out_dtype == PKV_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off) = v;
    } else {
        uint2 w;
        w.x = pack_bf16(v.x, v.y);
        w.y = pack_bf16(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<unsigned short *>(p.out) + off) = w;
    }
}

template <int KV, int D>
__global__ void __launch_bounds__(kThreads, PKV_PREFILL_MIN_CTAS)
    prefill_kernel(const PrefillParams p)
{
    using Geo = PrefillGeom<KV, D>;
    using Base = MmaStateBase<D, 2>;
    constexpr int NS = Geo::NS;
    constexpr int KS = Base::KS;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Geo::kRingBytes);
    uint64_t *empty = full + NS;
    __shared__ int s_item[8];
    __shared__ int s_ok[NS];
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const float c = p.score_scale;
    int cur_s = 0, cur_base = 0;  // warp 0's scan position
    bool initialised = false;
    bool first = true;

    for (;;) {
        if (threadIdx.x == 0) {
            s_item[0] = static_cast<int>(atomicAdd(p.counter, 1u));
            s_abort = 0;
        }
        __syncthreads();
        if (warp == 0) {
            PrefillItem it;
            const bool ok = find_prefill_item<kRowBlock>(p, s_item[0], cur_s, cur_base, lane, it);
            if (lane == 0) {
                s_item[1] = ok ? 1 : 0;
                if (ok) {
                    s_item[2] = it.s;
                    s_item[3] = it.hkv;
                    s_item[4] = it.part;
                    s_item[5] = it.rb;
                    s_item[6] = it.L;
                    s_item[7] = it.nq;
                    // Barriers restart for each item; the empty count is the
                    // number of warps that read each page.
                    const int rows = it.nq * G - it.rb * kRowBlock;
                    const int nrows = rows < kRowBlock ? rows : kRowBlock;
                    const int rt = (nrows + kRowTile - 1) / kRowTile;
                    const int rtp = rt == 3 ? 4 : rt;
                    for (int i = 0; i < NS; ++i) {
                        if (initialised) {
                            mbar_inval(&full[i]);
                            mbar_inval(&empty[i]);
                        }
                        mbar_init(&full[i], 1);
                        mbar_init(&empty[i], rtp);
                    }
                    fence_mbar_init();
                }
            }
            if (__shfl_sync(kFullMask, ok ? 1 : 0, 0))
                initialised = true;
        }
        __syncthreads();
        if (!s_item[1])
            break;
        const int s = s_item[2], hkv = s_item[3], part = s_item[4], rb = s_item[5];
        const int L = s_item[6], nq = s_item[7];
        const int q0 = __ldg(p.q_start + s);  // validated by the scan

        // ------------------------------------------------ item geometry
        const int rows = nq * G;
        const int row0 = rb * kRowBlock;
        const int nrows = min(kRowBlock, rows - row0);
        const int RT = (nrows + kRowTile - 1) / kRowTile;
        const int RTp = RT == 3 ? 4 : RT;
        const int PG = kWarps / RTp;
        const int rt = warp % RTp, pg = warp / RTp;
        const int q_first = L - nq;  // position of query 0
        const int pos_max = q_first + (row0 + nrows - 1) / G;
        const int P = p.partition;
        const int t0 = part * P;
        int t1 = t0 + P < L ? t0 + P : L;
        t1 = t1 < pos_max + 1 ? t1 : pos_max + 1;
        const int pg0 = t0 / kBlockSize;
        const int npages = t1 > t0 ? (t1 - t0 + kBlockSize - 1) / kBlockSize : 0;

        // ------------------------------------------- this warp's rows
        typename Base::State st;
        Base::reset(st);
        const int tile0 = row0 + rt * kRowTile;  // first row of the warp's tile
        const bool two_tiles = nrows - rt * kRowTile > 8;  // rows in the second N tile
        int pos[2][2];
        {
            const int r = lane >> 2, cc = lane & 3;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int R = tile0 + 8 * n + r;
                const bool ok = R - row0 < nrows;
                const int tok = q0 + (ok ? R / G : 0);
                const int h = hkv * G + (ok ? R % G : 0);
                const size_t qrow = (static_cast<size_t>(tok) * p.num_q_heads + h) * D;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int d = 16 * ks + 8 * hh + 2 * cc;
                        uint32_t w = ok ? *reinterpret_cast<const uint32_t *>(
                                              static_cast<const unsigned short *>(p.q) + qrow + d)
                                        : 0u;
                        // fp8 / INT4 pages are widened to f16: the query too.
                        if constexpr (KV != PKV_BF16)
                            w = pack_f16(bf16_lo(w), bf16_hi(w));
                        st.qf[ks][n][hh] = w;
                    }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int Rc = tile0 + 8 * n + 2 * cc + e;
                    pos[n][e] = (Rc - row0 < nrows) ? q_first + Rc / G : -1;
                }
            }
        }

        // ------------------------------------------------ page stream
        const int32_t *table = p.block_tables + static_cast<size_t>(s) * p.max_blocks + pg0;
        const size_t tile_stride = static_cast<size_t>(Geo::kTileBytes);
        const size_t block_stride = tile_stride * p.num_kv_heads;
        int issued = 0;  // pages issued (warp 0)
        bool aborted = false;
        auto issue_one = [&](int k) {
            const int stg = k % NS;
            const int phys = __ldg(table + k);
            const bool ok = phys >= 0 && phys < p.num_blocks;
            s_ok[stg] = ok ? 1 : 0;
            if (!ok) {
                set_status(p.status, PKV_ERR_OUT_OF_RANGE);
                mbar_arrive(&full[stg]);
                return;
            }
            mbar_arrive_expect_tx(&full[stg], 2 * Geo::kTileBytes);
            if (p.drop_first_copy && first && blockIdx.x == 0 && k == 0)
                return;
            const size_t off = static_cast<size_t>(phys) * block_stride + hkv * tile_stride;
            unsigned char *dst = smem + stg * Geo::kStageBytes;
            bulk_g2s(dst, static_cast<const unsigned char *>(p.k_cache) + off, Geo::kTileBytes,
                     &full[stg]);
            bulk_g2s(dst + Geo::kTileBytes, static_cast<const unsigned char *>(p.v_cache) + off,
                     Geo::kTileBytes, &full[stg]);
        };
        // Warp 0 only: issue pages < limit; blocking waits for free stages
        // when `block`, else stops at the first stage still in use.
        auto issue_upto = [&](int limit, bool block) {
            while (issued < npages && issued < limit) {
                if (issued >= NS) {
                    const int stg = issued % NS;
                    const uint32_t par = static_cast<uint32_t>((issued / NS) - 1) & 1u;
                    int ready = 0;
                    if (lane == 0)
                        ready = block ? mbar_wait_bounded(&empty[stg], par, kWaitLimitNs)
                                      : mbar_try_wait(&empty[stg], par);
                    ready = __shfl_sync(kFullMask, ready, 0);
                    if (!ready) {
                        if (block) {
                            if (lane == 0) {
                                set_status(p.status, PKV_ERR_TIMEOUT);
                                atomicExch(&s_abort, 1);
                            }
                            aborted = true;
                        }
                        return;
                    }
                }
                if (lane == 0)
                    issue_one(issued);
                ++issued;
            }
        };
        if (warp == 0)
            issue_upto(NS, false);

        for (int j = pg; j < npages && !aborted; j += PG) {
            if (warp == 0) {
                issue_upto(j + 1, true);
                if (aborted)
                    break;
            }
            const int stg = j % NS;
            const uint32_t par = static_cast<uint32_t>(j / NS) & 1u;
            const bool ok = mbar_wait_bounded(&full[stg], par, kWaitLimitNs);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) {
                    set_status(p.status, PKV_ERR_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                aborted = true;
                break;
            }
            const bool have = s_ok[stg] != 0;
            const unsigned char *sk = smem + stg * Geo::kStageBytes;
            // A warp whose row tile is empty (three tiles of rows on four
            // warps) only releases the stage.
            const bool work = have && rt < RT;
            if (work) {
                const int tb = (pg0 + j) * kBlockSize;  // position of the page's token 0
                const int valid = min(kBlockSize, L - tb);
                int lim[2][2];
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int v = pos[n][e] - tb + 1;
                        lim[n][e] = v < valid ? v : valid;
                    }
                if (two_tiles)
                    prefill_page<KV, D, 2>(st, sk, sk + Geo::kTileBytes, valid, lim, lane, c);
                else
                    prefill_page<KV, D, 1>(st, sk, sk + Geo::kTileBytes, valid, lim, lane, c);
            }
            // The stage is free once every lane's reads are done.
            fence_proxy_async();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[stg]);
            if (warp == 0)
                issue_upto(j + NS, false);
        }
        // Warp 0 issues whatever the other warps still wait for.
        if (warp == 0 && !aborted)
            issue_upto(npages, true);
        __syncthreads();
        if (s_abort) {
            // Let every copy still in flight land before the ring is reused.
            if (warp == 0 && lane == 0)
                for (int k = issued > NS ? issued - NS : 0; k < issued; ++k)
                    mbar_wait_bounded(&full[k % NS], static_cast<uint32_t>(k / NS) & 1u,
                                      kWaitLimitNs);
            __syncthreads();
        }

        // ---------------------------------------------- merge the warps
        float *scratch = reinterpret_cast<float *>(smem);
        {
            float *mine = scratch + warp * Geo::kScratchFloats;
            Base::finish(st, mine, mine + kRowTile * D, mine + kRowTile * D + kRowTile, lane);
        }
        __syncthreads();
        constexpr int Q4 = D / 4;
        for (int idx = threadIdx.x; idx < nrows * Q4; idx += kThreads) {
            const int r = idx / Q4, q4 = idx - r * Q4;
            const int rtr = r / kRowTile, rr = r % kRowTile;
            const int R = row0 + r;
            const int i = R / G;
            const int h = hkv * G + R % G;
            const int pos_r = q_first + i;
            const int nparts_r = p.max_parts > 1 ? parts_of(pos_r + 1, P) : 1;
            if (part >= nparts_r)
                continue;  // this partition is past the row's last visible token
            float mw[kWarps], mx = -INFINITY;
            for (int g = 0; g < PG; ++g) {
                const float *sw = scratch + (rtr + RTp * g) * Geo::kScratchFloats;
                mw[g] = sw[kRowTile * D + rr];
                mx = fmaxf(mx, mw[g]);
            }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            float lsum = 0.f;
            for (int g = 0; g < PG; ++g) {
                const float *sw = scratch + (rtr + RTp * g) * Geo::kScratchFloats;
                const float fw = (mw[g] == -INFINITY) ? 0.f : exp2f(mw[g] - mx);
                const float4 o = reinterpret_cast<const float4 *>(sw + rr * D)[q4];
                acc.x += fw * o.x;
                acc.y += fw * o.y;
                acc.z += fw * o.z;
                acc.w += fw * o.w;
                lsum += fw * sw[kRowTile * D + kRowTile + rr];
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            const float4 o4 = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (nparts_r == 1) {
                const float sc = p.out_scale;
                store_row4(p, D, q0 + i, h, q4,
                           make_float4(o4.x * sc, o4.y * sc, o4.z * sc, o4.w * sc));
            } else {
                const size_t prow =
                    (static_cast<size_t>(q0 + i) * p.num_q_heads + h) * p.max_parts + part;
                reinterpret_cast<float4 *>(p.part_o + prow * D)[q4] = o4;
                if (q4 == 0) {
                    p.part_ml[2 * prow] = mx;
                    p.part_ml[2 * prow + 1] = lsum;
                }
            }
        }
        __syncthreads();  // scratch (the ring) is read before the next item refills it
        first = false;
    }
}

// Log-sum-exp merge of the partials of one (query token, KV head): the rows
// whose visible context spans more than one partition.
template <int D>
__global__ void __launch_bounds__(kThreads) prefill_merge_kernel(const PrefillParams p)
{
    const int t = blockIdx.x / p.num_kv_heads;
    const int hkv = blockIdx.x - t * p.num_kv_heads;
    // The sequence of token t: q_start[lo] <= t < q_start[hi].  Each warp
    // probes 32 points per round, narrowing the range 32-fold (two rounds of
    // independent loads up to 1024 sequences, where halving takes ten
    // dependent ones).  A non-monotone q_start gives some s that the checks
    // below reject.
    const int lane = threadIdx.x & 31;
    int lo = 0, hi = p.num_seqs;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int at = lo + lane * step;
        const bool le = lane == 0 || (at < hi && __ldg(p.q_start + at) <= t);
        const unsigned bal = __ballot_sync(kFullMask, le);
        const int last = 31 - __clz(bal);
        lo += last * step;
        hi = min(hi, lo + step);
    }
    const int s = lo;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > p.max_len ? p.max_len : L);
    const int a = __ldg(p.q_start + s), b = __ldg(p.q_start + s + 1);
    if (a < 0 || b > p.num_tokens || b < a || b - a > L || b - a > p.max_q_len || t < a || t >= b)
        return;  // reported by the attention kernel
    if (p.skip_single && b - a == 1)
        return;  // a one-query sequence: served by the decode kernels
    const int pos = L - (b - a) + (t - a);
    const int nparts = parts_of(pos + 1, p.partition);
    if (nparts <= 1)
        return;  // written directly
    constexpr int Q4 = D / 4;
    const int G = p.group;
    for (int idx = threadIdx.x; idx < G * Q4; idx += blockDim.x) {
        const int g = idx / Q4, q4 = idx - g * Q4;
        const int h = hkv * G + g;
        const size_t row0 = (static_cast<size_t>(t) * p.num_q_heads + h) * p.max_parts;
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
            const float4 o =
                __ldcg(reinterpret_cast<const float4 *>(p.part_o + (row0 + i) * D) + q4);
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
        }
        const float sc = (wsum > 0.f ? 1.f / wsum : 0.f) * p.out_scale;
        store_row4(p, D, t, h, q4, make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc));
    }
}

template <int KV, int D>
pkv_status launch_prefill_d(const PrefillParams &p, cudaStream_t stream)
{
    using Geo = PrefillGeom<KV, D>;
    // Resident CTAs per SM, once the shared-memory attribute is set (per context).
    static ContextCache cache;
    int occ = 1;
    const pkv_status rc = cache.get(&occ, [](int *v) -> pkv_status {
        if (cudaFuncSetAttribute(prefill_kernel<KV, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, prefill_kernel<KV, D>, kThreads,
                                                          Geo::kSmem) != cudaSuccess)
            return PKV_ERR_CUDA;
        *v = o > 0 ? o : 1;
        return PKV_OK;
    });
    if (rc != PKV_OK)
        return rc;
    const long blocks = (static_cast<long>(p.max_q_len) * p.group + kRowBlock - 1) / kRowBlock;
    const long items = static_cast<long>(p.num_seqs) * p.num_kv_heads * p.max_parts * blocks;
    const long slots = static_cast<long>(occ) * device_sm_count();
    const long grid = items < slots ? items : slots;
    if (grid <= 0)
        return PKV_OK;
    prefill_kernel<KV, D><<<static_cast<unsigned>(grid), kThreads, Geo::kSmem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess)
        return PKV_ERR_CUDA;
    return launch_prefill_merge(p, stream);
}

}  // namespace

pkv_status launch_prefill_merge(const PrefillParams &p, cudaStream_t stream)
{
    if (p.max_parts <= 1 || p.num_tokens <= 0)
        return PKV_OK;
    const long mgrid = static_cast<long>(p.num_tokens) * p.num_kv_heads;
    if (p.head_dim == 128)
        prefill_merge_kernel<128><<<static_cast<unsigned>(mgrid), kThreads, 0, stream>>>(p);
    else
        prefill_merge_kernel<64><<<static_cast<unsigned>(mgrid), kThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <int KV>
static pkv_status launch_prefill_kv(const PrefillParams &p, cudaStream_t stream)
{
    return p.head_dim == 128 ? launch_prefill_d<KV, 128>(p, stream)
                             : launch_prefill_d<KV, 64>(p, stream);
}

pkv_status launch_prefill(const PrefillParams &p, int kv_dtype, cudaStream_t stream)
{
    if (p.group < 1 || p.group > 16)
        return PKV_ERR_UNSUPPORTED;
    if (p.head_dim != 128 && p.head_dim != 64)
        return PKV_ERR_UNSUPPORTED;
    switch (kv_dtype) {
    case PKV_BF16:
        if (p.impl == PKV_FLAG_IMPL_TC)
            return launch_prefill_tc(p, stream);
        return launch_prefill_kv<PKV_BF16>(p, stream);
    // fp8 and INT4 caches: the mma.sync kernel (its fragments widen the codes
    // in registers, as the decode kernels do).
    case PKV_FP8_E5M2:
        return p.impl == PKV_FLAG_IMPL_TC ? PKV_ERR_UNSUPPORTED
                                          : launch_prefill_kv<PKV_FP8_E5M2>(p, stream);
    case PKV_FP8_E4M3:
        return p.impl == PKV_FLAG_IMPL_TC ? PKV_ERR_UNSUPPORTED
                                          : launch_prefill_kv<PKV_FP8_E4M3>(p, stream);
    case PKV_INT4:
        return p.impl == PKV_FLAG_IMPL_TC ? PKV_ERR_UNSUPPORTED
                                          : launch_prefill_kv<PKV_INT4>(p, stream);
    default:
        return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace pkv
