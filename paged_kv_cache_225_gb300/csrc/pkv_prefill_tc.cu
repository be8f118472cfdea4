// Paged attention of several query tokens per sequence on the tcgen05 tensor
// cores of sm_103a (chunked prefill, speculative verification).
//
// What is computed is the same as the mma.sync form in pkv_prefill.cu: the
// block-table walk of the PagedAttention kernel pseudocode ("vLLM e
// PagedAttention: serving high-throughput") with the causal mask of the
// "Inference optimization" lesson (Step 2, scaled_dot_product_attention,
// triu mask of offset seq_len_k - seq_len_q + 1); query i of the n queries of
// a sequence of L cached tokens attends the rows t <= L - n + i.
//
// How it is laid out on the GPU (not taken from the pages):
//  * An item is (sequence, KV head, context partition, block of up to M
//    rows), a row being one (query token, grouped query head) pair; M = 128,
//    or 64 when no sequence has more rows.  Every K/V page crosses HBM once
//    per item.
//  * Six warps with fixed roles.  Warp 4 (producer) pulls items from an
//    atomic counter, hands them to the others through a two-slot queue, and
//    copies K and V with tensor-map (TMA) loads into a ring of stages of two
//    pages each.  Warp 5 (one thread) issues the MMAs.  Warps 0-3 own one row
//    per thread (the row's TMEM lane): Q, softmax, P, rescaling, output.
//  * Tensor memory holds O (M x head_dim f32), two score buffers of 32
//    columns and the item's Q (bf16 pairs, the A operand of S).
//    Per chunk of two pages: S = Q K^T (M rows, N = 32 tokens, head_dim / 16
//    MMAs of K = 16); each row's thread reads its 32 scores, applies the
//    causal limit and the online softmax, and writes P back over its
//    consumed scores as a bf16 high part and a bf16 residual; then
//    O += P_hi V + P_lo V (M rows, N = head_dim, K = 16 per page) with P
//    read from tensor memory.  The scores of chunk i + 1 are issued before
//    P V of chunk i.
//  * The running max is updated lazily (only when a score exceeds it by
//    2^8); O is then rescaled in TMEM by the rows' threads once the previous
//    P V has completed.
//  * Each page tile [head_dim][16 tokens] (32-byte rows) is copied whole by
//    one tensor-map load in the 32-byte swizzle mode: row d lands at 32 d
//    with its two 16-byte halves exchanged when bit 7 of the address is set,
//    which is the 32-byte-swizzled operand layout of the MMA (atoms of 8
//    rows x 32 bytes).  Every 32-byte sector of the cache is requested once
//    and whole.  The two K tiles of a stage are adjacent, so one MMA with
//    N = 32 reads both (MN-major); V tiles are read K-major.
//  * Every wait is bounded; a timeout records PKV_ERR_TIMEOUT, stops every
//    role, lets copies and MMAs in flight finish and frees TMEM.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is looked up at run time

#include "pkv_prefill.cuh"

namespace pkv {

namespace {

// Rows per item = the MMA's M: 128, or 64 when no sequence has more than 64
// rows (speculative verification: 5 queries x 8 grouped heads = 40).  An
// M = 64 accumulator holds row 16 w + i in lane 32 w + i (i < 16) of TMEM
// lane quarter w; the A operand read from TMEM (Q, P) uses the same lanes.
template <int M> __host__ __device__ constexpr int tc_rows_ok()
{
    return M == 64 || M == 128;
}
constexpr int kTcThreads = 192;
constexpr int kQueue = 4;  // item queue slots (the producer publishes up to three items ahead)
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;

// Pages per softmax step.  Two keeps O, two score buffers and Q inside 256
// TMEM columns (two CTAs per SM); four needs 320 (one CTA per SM, a 192 KB
// ring): measured slower on GB300 (70B verification 420 -> 455 us).
#ifndef PKV_TC_CHUNK
#define PKV_TC_CHUNK 2
#endif
constexpr int kChunk = PKV_TC_CHUNK;
static_assert(kChunk == 2 || kChunk == 4, "two or four pages per step");

template <int D> struct TcGeom {
    static constexpr int kTile = D * kBlockSize * 2;  // one K or V page tile (bf16)
    static constexpr int kRow = kBlockSize * 2;       // one head_dim row: 32 bytes
    static constexpr int kVOff = kChunk * kTile;      // V tiles follow the K tiles
    static constexpr int kStage = 2 * kChunk * kTile;
    static constexpr int kSCols = kChunk * kBlockSize;  // score columns per buffer
    static constexpr int kTmemUsed = D + 2 * kSCols + D / 2;  // O, two score buffers, Q
    static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
    static constexpr int NS = (kTmemCols == 256 ? 96 * 1024 : 192 * 1024) / kStage;
    static constexpr int kSmem = NS * kStage;
    // Two score / P buffers; a third (scores two chunks ahead) would push Q
    // out of tensor memory and cut the ring to four stages: measured slower
    // (70B verification 419 -> 496 us).
    static constexpr int kSBufs = 2;
    static constexpr int kSCol = D;                     // score buffers after O
    static constexpr int kQCol = D + kSBufs * kSCols;   // Q as bf16 pairs: D / 2 columns
    static_assert(kQCol + D / 2 <= kTmemCols, "O, scores and Q fit the allocation");
    static_assert(NS >= 4, "ring holds the chunks in use and copies ahead");
};

// ------------------------------------------------------------ tcgen05 / TMA

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a 32-byte-swizzled operand (atoms of
// 8 rows x 32 bytes, the 16-byte halves of a row exchanged where address bit
// 7 is set): start address, the leading byte offset (MN-major: distance
// between atoms along M / N; unused K-major), the stride byte offset
// (distance between 8-row groups), descriptor version 1, layout code 6
// (32-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw32(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3fffu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(6) << 61;
    return d;
}

// Instruction descriptor of kind::f16: f32 accumulator, bf16 A and B, A
// K-major, B K-major or MN-major, N and M.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A B with A read from tensor memory (row m in lane m, elements 2c
// and 2c + 1 of a row in the low and high halves of column c) and B from a
// shared-memory descriptor; D is overwritten when accumulate is false.
__device__ __forceinline__ void tc_mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                          uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1u : 0u));
}

// Arrives on bar once every MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Sixteen-lane accesses of an M = 64 accumulator (a warp's 16 rows in lanes
// 0-15 of its quarter).  Thread i of the warp holds rows i / 4 and i / 4 + 8.
// 16x256b, four repetitions of 8 columns: registers 4 j .. 4 j + 3 are
// columns 8 j + 2 (i % 4) and 8 j + 2 (i % 4) + 1 of the first row, then the
// same columns of the second.  16x128b, four repetitions of 4 columns:
// registers 2 j and 2 j + 1 are column 4 j + i % 4 of the two rows.
__device__ __forceinline__ void tmem_ld_r16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st_r16(uint32_t taddr, const float (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_c8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile(
        "tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// 3-D tensor-map load of one box into shared memory, completing on bar.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, const volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

// Every lane waits (each needs the barrier's ordering); the warp agrees on
// the outcome so that it stays converged for the .sync.aligned TMEM accesses.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, const volatile int *abort)
{
    const bool ok = tc_wait(bar, parity, abort);
    return __all_sync(kFullMask, ok);
}

__device__ __forceinline__ void tc_fail(const PrefillParams &p, volatile int *abort)
{
    set_status(p.status, PKV_ERR_TIMEOUT);
    *abort = 1;
}

__device__ __forceinline__ void store_out2(const PrefillParams &p, int D, size_t orow, int col,
                                           float2 v)
{
    const size_t off = orow * D + col;
    if (p.out_dtype == PKV_F32)
        *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + off) = v;
    else
        *reinterpret_cast<uint32_t *>(static_cast<unsigned short *>(p.out) + off) =
            pack_bf16(v.x, v.y);
}

__device__ __forceinline__ void store_out4(const PrefillParams &p, int D, size_t orow, int q4,
                                           float4 v)
{
    const size_t off = orow * D + 4 * q4;
    if (p.out_dtype == PKV_F32) {
        *reinterpret_cast<float4 *>(static_cast<float *>(p.out) + off) = v;
    } else {
        uint2 w;
        w.x = pack_bf16(v.x, v.y);
        w.y = pack_bf16(v.z, v.w);
        *reinterpret_cast<uint2 *>(static_cast<unsigned short *>(p.out) + off) = w;
    }
}

struct TcMaps {
    CUtensorMap k, v;  // K / V caches, one box = one page tile
};

struct TcItem {
    int valid, s, hkv, part, rb, L, nq;
};

__device__ __forceinline__ TcItem read_item(const int *slot)
{
    TcItem it;
    it.valid = slot[0];
    it.s = slot[1];
    it.hkv = slot[2];
    it.part = slot[3];
    it.rb = slot[4];
    it.L = slot[5];
    it.nq = slot[6];
    return it;
}

template <int D, int kTcRows, bool kPhased>
__global__ void __launch_bounds__(kTcThreads, kChunk == 2 ? 2 : 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ TcMaps maps)
{
    using Geo = TcGeom<D>;
    static_assert(tc_rows_ok<kTcRows>(), "M is 64 or 128");
    constexpr int NS = Geo::NS;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[NS], empty[NS];
    constexpr int SB = Geo::kSBufs;
    __shared__ __align__(8) uint64_t s_full[SB], p_full[SB], pv_done[SB];
    __shared__ __align__(8) uint64_t item_full[kQueue], item_empty[kQueue];
    __shared__ __align__(8) uint64_t q_full, o_free, drain;
    __shared__ int s_item[kQueue][8];
    __shared__ int s_ok[NS][kChunk];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    volatile int *abort = &s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&pv_done[i], 1);
        }
        for (int i = 0; i < kQueue; ++i) {
            mbar_init(&item_full[i], 1);
            mbar_init(&item_empty[i], 5);  // the MMA thread and the four softmax warps
        }
        mbar_init(&q_full, 4);
        mbar_init(&o_free, 4);
        mbar_init(&drain, 1);
        s_abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_u32(&s_tmem)),
            "r"(Geo::kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int G = p.group;
    const uint32_t smem0 = smem_u32(smem);

    if (smem0 & 255u) {
        // The swizzled tiles need 256-byte aligned stages: report, run nothing.
        if (threadIdx.x == 0)
            set_status(p.status, PKV_ERR_UNSUPPORTED);
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------- producer
        // Items are claimed from the counter one at a time, when the
        // previous item's copies are all issued (claiming earlier unbalances
        // the CTAs' last items).  The query rows of a claimed item are
        // prefetched into L2 for the softmax warps, which load them a ring's
        // worth of chunks later.
        // Split contexts (kPhased): item phases (largest items first) and
        // each phase's scan position.  Unsplit calls keep sequence order
        // (measured on the unsplit chunked prefill: 267 -> 283 us with the
        // phases).
        int nph[kPrefillPhases];
        if constexpr (kPhased) {
            count_prefill_phases<kTcRows>(p, lane, nph);
        } else {
#pragma unroll
            for (int ph = 0; ph < kPrefillPhases; ++ph)
                nph[ph] = 0;
        }
        int cur[2 * kPrefillPhases];
#pragma unroll
        for (int i = 0; i < 2 * kPrefillPhases; ++i)
            cur[i] = 0;
        uint32_t gc = 0;  // chunks issued by this CTA
        bool stop = false;
        for (int k = 0; !stop; ++k) {
            unsigned u = 0;
            if (lane == 0)
                u = atomicAdd(p.counter, 1u);
            u = __shfl_sync(kFullMask, u, 0);
            PrefillItem it;
            bool ok = false;
            int r = static_cast<int>(u);
            if constexpr (!kPhased) {
                ok = find_prefill_item<kTcRows>(p, r, cur[0], cur[1], lane, it);
            } else {
#pragma unroll
                for (int ph = 0; ph < kPrefillPhases; ++ph) {
                    if (!ok && (r < nph[ph] || ph == kPrefillPhases - 1)) {
                        ok = find_prefill_item_phase<kTcRows>(p, r, ph, cur[2 * ph],
                                                              cur[2 * ph + 1], lane, it);
                        r = INT_MAX;  // found or past the end: no later phase
                    } else if (!ok) {
                        r -= nph[ph];
                    }
                }
            }
            const int slot = k % kQueue;
            int free_ok = 1;
            if (k >= kQueue && lane == 0)
                free_ok = tc_wait(&item_empty[slot], ((k - kQueue) / kQueue) & 1, abort);
            free_ok = __shfl_sync(kFullMask, free_ok, 0);
            if (!free_ok) {
                if (lane == 0)
                    tc_fail(p, abort);
                break;
            }
            if (lane == 0) {
                int *w = s_item[slot];
                w[0] = ok ? 1 : 0;
                w[1] = it.s;
                w[2] = it.hkv;
                w[3] = it.part;
                w[4] = it.rb;
                w[5] = it.L;
                w[6] = it.nq;
                mbar_arrive(&item_full[slot]);
            }
            if (!ok)
                break;
            const int row0 = it.rb * kTcRows;
            const int nrows = min(kTcRows, it.nq * G - row0);
            for (int r = lane; r < nrows; r += 32) {
                const int R = row0 + r;
                const unsigned char *qrow =
                    static_cast<const unsigned char *>(p.q) +
                    (static_cast<size_t>(it.q0 + R / G) * p.num_q_heads + it.hkv * G + R % G) * D * 2;
#pragma unroll
                for (int b = 0; b < D * 2; b += 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow + b));
            }
            int pg0, npages;
            item_pages(p, it.L, it.nq, row0, nrows, it.part, pg0, npages);
            const int32_t *table = p.block_tables + static_cast<size_t>(it.s) * p.max_blocks + pg0;
            for (int j0 = 0; j0 < npages && !stop; j0 += 32) {
                const int ent = j0 + lane < npages ? __ldg(table + j0 + lane) : -1;
                const int n = min(32, npages - j0);  // even unless it ends the item
                for (int jj = 0; jj < n; jj += kChunk, ++gc) {
                    const int stg = static_cast<int>(gc % NS);
                    int ready = 1;
                    if (gc >= NS && lane == 0)
                        ready = tc_wait(&empty[stg], ((gc / NS) - 1) & 1, abort);
                    ready = __shfl_sync(kFullMask, ready, 0);
                    if (!ready) {
                        if (lane == 0)
                            tc_fail(p, abort);
                        stop = true;
                        break;
                    }
                    int phys[kChunk];
#pragma unroll
                    for (int x = 0; x < kChunk; ++x)
                        phys[x] = __shfl_sync(kFullMask, ent, (jj + x) & 31);
                    if (lane == 0) {
                        int good[kChunk], ngood = 0;
#pragma unroll
                        for (int x = 0; x < kChunk; ++x) {
                            const bool present = jj + x < n;
                            good[x] = present && phys[x] >= 0 && phys[x] < p.num_blocks;
                            if (present && !good[x])
                                set_status(p.status, PKV_ERR_OUT_OF_RANGE);
                            s_ok[stg][x] = good[x];
                            ngood += good[x];
                        }
                        if (ngood == 0) {
                            mbar_arrive(&full[stg]);
                        } else {
                            mbar_arrive_expect_tx(&full[stg], ngood * 2 * Geo::kTile);
                            unsigned char *st = smem + stg * Geo::kStage;
#pragma unroll
                            for (int x = 0; x < kChunk; ++x) {
                                if (!good[x] ||
                                    (p.drop_first_copy && blockIdx.x == 0 && gc == 0 && x == 0))
                                    continue;
                                unsigned char *dk = st + x * Geo::kTile;
                                unsigned char *dv = st + Geo::kVOff + x * Geo::kTile;
                                const int c2 = phys[x] * p.num_kv_heads + it.hkv;
                                tma_load_3d(dk, &maps.k, 0, 0, c2, &full[stg]);
                                tma_load_3d(dv, &maps.v, 0, 0, c2, &full[stg]);
                            }
                        }
                    }
                }
            }
        }
        if (*abort && lane == 0) {
            // Let every copy still in flight land before the CTA exits.
            const uint32_t lo = gc > NS ? gc - NS : 0;
            for (uint32_t q = lo; q < gc; ++q)
                mbar_wait_bounded(&full[q % NS], (q / NS) & 1, kWaitLimitNs);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t kIdS = tc_idesc(kTcRows, Geo::kSCols, true);
            constexpr uint32_t kIdPV = tc_idesc(kTcRows, D, false);
            uint32_t gc = 0;       // chunks
            uint32_t counted = 0;  // items with pages
            bool failed = false;
            bool o_started = false, o_wait = false;
            // P V of chunk c: waits for its P, and before the first P V of an
            // item for the previous item's output to have been read.
            auto issue_pv = [&](uint32_t c) -> bool {
                if (!tc_wait(&p_full[c % SB], (c / SB) & 1, abort))
                    return false;
                if (o_wait) {
                    if (!tc_wait(&o_free, (counted - 2) & 1, abort))
                        return false;
                    o_wait = false;
                }
                tc_fence_after();
                const int stg = static_cast<int>(c % NS);
                const uint32_t pcol = tmem + Geo::kSCol + Geo::kSCols * (c % SB);
#pragma unroll
                for (int x = 0; x < kChunk; ++x) {
                    if (!s_ok[stg][x])
                        continue;
                    // K-major: one 32-byte row (16 tokens) per dim, 8-dim groups 256 B apart.
                    const uint64_t vdesc = smem_desc_sw32(
                        smem0 + stg * Geo::kStage + Geo::kVOff + x * Geo::kTile, 16,
                        8 * Geo::kRow);
                    tc_mma_ta(tmem, pcol + 8 * x, vdesc, kIdPV, o_started);
                    tc_mma_ta(tmem, pcol + Geo::kSCols / 2 + 8 * x, vdesc, kIdPV, true);
                    o_started = true;
                }
                tc_commit(&pv_done[c % SB]);
                tc_commit(&empty[stg]);
                return true;
            };
            for (int k = 0; !failed; ++k) {
                const int slot = k % kQueue;
                if (!tc_wait(&item_full[slot], (k / kQueue) & 1, abort)) {
                    failed = true;
                    break;
                }
                const TcItem it = read_item(s_item[slot]);
                mbar_arrive(&item_empty[slot]);
                if (!it.valid)
                    break;
                const int row0 = it.rb * kTcRows;
                const int nrows = min(kTcRows, it.nq * G - row0);
                int pg0, npages;
                item_pages(p, it.L, it.nq, row0, nrows, it.part, pg0, npages);
                if (npages == 0)
                    continue;
                if (!tc_wait(&q_full, counted & 1, abort)) {
                    failed = true;
                    break;
                }
                ++counted;
                o_started = false;
                o_wait = counted >= 2;
                const int nchunks = (npages + kChunk - 1) / kChunk;
                // Scores run SB - 1 chunks ahead of P V.
                for (int j = 0; j < nchunks; ++j, ++gc) {
                    const int stg = static_cast<int>(gc % NS);
                    if (!tc_wait(&full[stg], (gc / NS) & 1, abort)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    // Scores of both pages in one MMA per k step (absent or
                    // bad pages leave stale columns that the softmax masks).
                    // MN-major: 16 tokens per row, the second page's tile
                    // one tile further (the leading offset), 8-dim groups
                    // 256 B apart; k step ks starts at dim 16 ks.
                    const uint32_t scol = tmem + Geo::kSCol + Geo::kSCols * (gc % SB);
                    const uint32_t kaddr = smem0 + stg * Geo::kStage;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        tc_mma_ta(scol, tmem + Geo::kQCol + 8 * ks,
                                  smem_desc_sw32(kaddr + ks * 16 * Geo::kRow, Geo::kTile,
                                                 8 * Geo::kRow),
                                  kIdS, ks > 0);
                    tc_commit(&s_full[gc % SB]);
                    if (j >= SB - 1 && !issue_pv(gc - (SB - 1))) {
                        failed = true;
                        break;
                    }
                }
                if (failed)
                    break;
                for (int r = nchunks < SB - 1 ? nchunks : SB - 1; r >= 1 && !failed; --r)
                    failed = !issue_pv(gc - r);
                if (failed)
                    break;
            }
            if (failed)
                tc_fail(p, abort);
            // Every MMA issued has completed before TMEM is freed.
            tc_commit(&drain);
            mbar_wait_bounded(&drain, 0, kWaitLimitNs);
        }
    } else if constexpr (kTcRows == 128) {
        // ---------------------------------------- Q, softmax and output
        const int t = threadIdx.x;  // row of the item = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const float c = p.score_scale;
        constexpr float kLazy = MmaSoftmax::kLazy;
        constexpr int kTok = Geo::kSCols;  // tokens per chunk
        uint32_t gc = 0;
        int k = 0;  // queue entries read

        struct RowItem {
            TcItem it;
            int pg0, npages, q0, qi, h, pos;
            bool row_ok;
        };
        // Next queue item with pages (true), or the end of the work (false,
        // ended) or an abort (false, !ended).
        auto next_item = [&](RowItem &ri, bool &ended) -> bool {
            for (;;) {
                const int slot = k % kQueue;
                if (!warp_wait(&item_full[slot], (k / kQueue) & 1, abort)) {
                    ended = false;
                    return false;
                }
                const TcItem it = read_item(s_item[slot]);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&item_empty[slot]);
                ++k;
                if (!it.valid) {
                    ended = true;
                    return false;
                }
                const int row0 = it.rb * kTcRows;
                const int nrows = min(kTcRows, it.nq * G - row0);
                int pg0, npages;
                item_pages(p, it.L, it.nq, row0, nrows, it.part, pg0, npages);
                if (npages == 0)
                    continue;
                ri.it = it;
                ri.pg0 = pg0;
                ri.npages = npages;
                ri.q0 = __ldg(p.q_start + it.s);  // validated by the item scan
                ri.row_ok = t < nrows;
                const int R = row0 + (ri.row_ok ? t : 0);
                ri.qi = R / G;
                ri.h = it.hkv * G + R % G;
                ri.pos = it.L - it.nq + ri.qi;  // position of this row's query
                return true;
            }
        };
        // Q row (zero past the item) into tensor memory, every load issued
        // before the first store.  Callers have seen the scores of every
        // chunk of the previous item, so no MMA still reads the old Q.
        auto load_q = [&](const RowItem &ri) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const unsigned short *>(p.q) +
                (static_cast<size_t>(ri.q0 + ri.qi) * p.num_q_heads + ri.h) * D);
            uint4 v[D / 8];
#pragma unroll
            for (int e = 0; e < D / 8; ++e)
                v[e] = ri.row_ok ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
            // bf16 pairs, element 2c of the row in the low half of column c.
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    r[4 * e] = v[c0 / 4 + e].x;
                    r[4 * e + 1] = v[c0 / 4 + e].y;
                    r[4 * e + 2] = v[c0 / 4 + e].z;
                    r[4 * e + 3] = v[c0 / 4 + e].w;
                }
                tmem_st16u(tmem + lane_base + Geo::kQCol + c0, r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&q_full);
        };

        RowItem cur;
        bool ended = false;
        bool have = next_item(cur, ended);
        bool failed = !have && !ended;
        if (have)
            load_q(cur);
        while (have) {
            float m = -INFINITY, l = 0.f;
            bool o_valid = false;
            const int npages = cur.npages;
            const int32_t *table =
                p.block_tables + static_cast<size_t>(cur.it.s) * p.max_blocks + cur.pg0;
            // Block-table entries of pages [32w, 32w + 32) in `ent`, the next
            // window already on its way in `ent_next`.
            int ent = lane < npages ? __ldg(table + lane) : -1;
            int ent_next = 32 + lane < npages ? __ldg(table + 32 + lane) : -1;
            const int nchunks = (npages + kChunk - 1) / kChunk;
            // A warp whose 32 rows all lie past the item's rows (items of
            // fewer than 128 rows: 40 in speculative verification) skips the
            // score, softmax and P work and the output; it still waits for
            // each chunk's scores (its threads zero V past the sequence end
            // after the copy landed) and makes every arrival.  Its rows of P
            // and O hold stale values that feed only rows never written.
            const bool live = __any_sync(kFullMask, cur.row_ok);
            for (int j = 0; j < nchunks; ++j, ++gc) {
                const int jp = j * kChunk;  // first page of the chunk
                if (jp > 0 && (jp & 31) == 0) {
                    ent = ent_next;
                    ent_next = jp + 32 + lane < npages ? __ldg(table + jp + 32 + lane) : -1;
                }
                bool good[kChunk];
                bool any_good = false;
#pragma unroll
                for (int x = 0; x < kChunk; ++x) {
                    const int phys = __shfl_sync(kFullMask, ent, (jp + x) & 31);
                    good[x] = jp + x < npages && phys >= 0 && phys < p.num_blocks;
                    any_good = any_good || good[x];
                }
                if (!warp_wait(&s_full[gc % SB], (gc / SB) & 1, abort)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t scol = tmem + lane_base + Geo::kSCol + Geo::kSCols * (gc % SB);
                const int tb = (cur.pg0 + jp) * kBlockSize;  // position of the chunk's token 0
                if (live) {
                    // Scaled scores, -inf where the row does not see the token.
                    float xs[kTok];
#pragma unroll
                    for (int x = 0; x < kChunk; ++x) {
                        float part[16];
                        tmem_ld16(scol + 16 * x, part);
                        int v = cur.pos - (tb + 16 * x) + 1;
                        v = v < 0 ? 0 : (v > kBlockSize ? kBlockSize : v);
                        const int lim = (cur.row_ok && good[x]) ? v : 0;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            xs[16 * x + e] = e < lim ? part[e] * c : -INFINITY;
                    }
                    float mx;
                    {
                        float r[kTok / 2];
#pragma unroll
                        for (int e = 0; e < kTok / 2; ++e)
                            r[e] = fmaxf(xs[e], xs[e + kTok / 2]);
#pragma unroll
                        for (int w = kTok / 4; w >= 1; w >>= 1)
#pragma unroll
                            for (int e = 0; e < w; ++e)
                                r[e] = fmaxf(r[e], r[e + w]);
                        mx = r[0];
                    }
                    const bool need = mx > m + kLazy;  // false when nothing is visible
                    float alpha = 1.f;
                    if (need) {
                        alpha = m == -INFINITY ? 0.f : MmaSoftmax::ex2(m - mx);
                        l *= alpha;
                        m = mx;
                    }
                    if (o_valid && __any_sync(kFullMask, need)) {
                        // O holds earlier chunks: rescale it once their P V is done.
                        if (!warp_wait(&pv_done[(gc - 1) % SB], ((gc - 1) / SB) & 1, abort)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 16) {
                            float ov[16];
                            tmem_ld16(tmem + lane_base + c0, ov);
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                ov[e] *= alpha;
                            tmem_st16(tmem + lane_base + c0, ov);
                        }
                        tmem_wait_st();
                    }
                    // P over the consumed scores: high parts in the first half of
                    // the buffer, residuals in the second (bf16 pairs).  A row
                    // that has seen nothing keeps m = -inf and P = 0.
                    const bool seen = m != -INFINITY;
                    uint32_t hi[kTok / 2], lo[kTok / 2];
                    float psum = 0.f;
#pragma unroll
                    for (int e = 0; e < kTok; e += 2) {
                        const float a = seen ? MmaSoftmax::ex2(xs[e] - m) : 0.f;
                        const float b = seen ? MmaSoftmax::ex2(xs[e + 1] - m) : 0.f;
                        psum += a + b;
                        hi[e / 2] = pack_bf16(a, b);
                        lo[e / 2] = pack_bf16(a - bf16_lo(hi[e / 2]), b - bf16_hi(hi[e / 2]));
                    }
                    l += psum;
#pragma unroll
                    for (int c0 = 0; c0 < kTok / 2; c0 += 16) {
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = hi[c0 + e];
                        tmem_st16u(scol + c0, w);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = lo[c0 + e];
                        tmem_st16u(scol + kTok / 2 + c0, w);
                    }
                    tmem_wait_st();
                }  // live
                if (failed)
                    break;
                // Past the sequence end the V tile may hold anything (NaN):
                // zero those tokens, since P = 0 does not cancel NaN.
                bool zeroed = false;
#pragma unroll
                for (int x = 0; x < kChunk; ++x) {
                    const int valid = cur.it.L - (tb + 16 * x);
                    if (good[x] && valid > 0 && valid < kBlockSize) {
                        if (t < D) {
                            // Row t of the swizzled tile: half h of the row
                            // sits at half h ^ (bit 2 of t).
                            unsigned short *vt = reinterpret_cast<unsigned short *>(
                                smem + (gc % NS) * Geo::kStage + Geo::kVOff + x * Geo::kTile +
                                t * Geo::kRow);
                            const int sw = static_cast<int>(smem_u32(vt) >> 7) & 1;
                            for (int e = valid; e < kBlockSize; ++e)
                                vt[(((e >> 3) ^ sw) << 3) + (e & 7)] = 0;
                        }
                        zeroed = true;
                    }
                }
                if (zeroed)
                    fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[gc % SB]);
                o_valid = o_valid || any_good;
            }
            if (failed)
                break;

            // The next item's Q first, so that its scores and copies run
            // while this item's output rows are written.
            RowItem nxt;
            bool nended = false;
            const bool have_next = next_item(nxt, nended);
            if (!have_next && !nended) {
                failed = true;
                break;
            }
            if (have_next)
                load_q(nxt);

            // ------------------------------------------------ output rows
            if (o_valid && live) {
                if (!warp_wait(&pv_done[(gc - 1) % SB], ((gc - 1) / SB) & 1, abort)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
            }
            const int nparts_r = p.max_parts > 1 ? parts_of(cur.pos + 1, p.partition) : 1;
            const bool write = cur.row_ok && cur.it.part < nparts_r;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t orow = static_cast<size_t>(cur.q0 + cur.qi) * p.num_q_heads + cur.h;
#pragma unroll 1
            for (int c0 = 0; c0 < (live ? D : 0); c0 += 16) {
                float ov[16];
                if (o_valid) {
                    tmem_ld16(tmem + lane_base + c0, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ov[e] = 0.f;
                }
                if (!write)
                    continue;
                if (nparts_r == 1) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        store_out4(p, D, orow, c0 / 4 + q4,
                                   make_float4(ov[4 * q4] * inv, ov[4 * q4 + 1] * inv,
                                               ov[4 * q4 + 2] * inv, ov[4 * q4 + 3] * inv));
                } else {
                    const size_t prow = orow * p.max_parts + cur.it.part;
                    float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * D + c0);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4)
                        dst[q4] = make_float4(ov[4 * q4] * inv, ov[4 * q4 + 1] * inv,
                                              ov[4 * q4 + 2] * inv, ov[4 * q4 + 3] * inv);
                }
            }
            if (write && nparts_r > 1) {
                const size_t prow = orow * p.max_parts + cur.it.part;
                p.part_ml[2 * prow] = m;
                p.part_ml[2 * prow + 1] = l;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&o_free);
            cur = nxt;
            have = have_next;
        }
        if (failed)
            tc_fail(p, abort);
    } else {
        // ------------------------- Q, softmax and output, 64-row items
        // Warp w owns rows 16 w .. 16 w + 15 (TMEM lanes 0-15 of its
        // quarter).  Each thread holds two of them, rows g and g + 8 of the
        // warp's sixteen, and a quarter of each chunk's columns (8 of 32);
        // the four threads of a row combine their maxima by shuffles and
        // their sums at the end.
        const int t = threadIdx.x;  // V rows zeroed by this thread (t < head_dim)
        const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
        const int g = lane >> 2, qd = lane & 3;
        const float c = p.score_scale;
        constexpr float kLazy = MmaSoftmax::kLazy;
        constexpr int kTok = Geo::kSCols;  // tokens per chunk
        static_assert(kTok == 32, "four 16x256b repetitions cover a chunk's scores");
        uint32_t gc = 0;
        int k = 0;  // queue entries read

        struct RowPair {
            TcItem it;
            int pg0, npages, q0;
            bool ok[2];
            int qi[2], h[2], pos[2];  // rows 16 w + g and 16 w + g + 8
            bool q_ok;                // lane < 16: Q row 16 w + lane
            int q_qi, q_h;
        };
        auto next_item = [&](RowPair &ri, bool &ended) -> bool {
            for (;;) {
                const int slot = k % kQueue;
                if (!warp_wait(&item_full[slot], (k / kQueue) & 1, abort)) {
                    ended = false;
                    return false;
                }
                const TcItem it = read_item(s_item[slot]);
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&item_empty[slot]);
                ++k;
                if (!it.valid) {
                    ended = true;
                    return false;
                }
                const int row0 = it.rb * kTcRows;
                const int nrows = min(kTcRows, it.nq * G - row0);
                int pg0, npages;
                item_pages(p, it.L, it.nq, row0, nrows, it.part, pg0, npages);
                if (npages == 0)
                    continue;
                ri.it = it;
                ri.pg0 = pg0;
                ri.npages = npages;
                ri.q0 = __ldg(p.q_start + it.s);  // validated by the item scan
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int r = 16 * warp + g + 8 * x;
                    ri.ok[x] = r < nrows;
                    const int R = row0 + (ri.ok[x] ? r : 0);
                    ri.qi[x] = R / G;
                    ri.h[x] = it.hkv * G + R % G;
                    ri.pos[x] = it.L - it.nq + ri.qi[x];
                }
                const int rq = 16 * warp + lane;
                ri.q_ok = lane < 16 && rq < nrows;
                const int RQ = row0 + (ri.q_ok ? rq : 0);
                ri.q_qi = RQ / G;
                ri.q_h = it.hkv * G + RQ % G;
                return true;
            }
        };
        // Q row (zero past the item) into tensor memory, lanes 0-15 of the
        // quarter; callers have seen every score of the previous item.
        auto load_q = [&](const RowPair &ri) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const unsigned short *>(p.q) +
                (static_cast<size_t>(ri.q0 + ri.q_qi) * p.num_q_heads + ri.q_h) * D);
            uint4 v[D / 8];
#pragma unroll
            for (int e = 0; e < D / 8; ++e)
                v[e] = ri.q_ok ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 16) {
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    r[4 * e] = v[c0 / 4 + e].x;
                    r[4 * e + 1] = v[c0 / 4 + e].y;
                    r[4 * e + 2] = v[c0 / 4 + e].z;
                    r[4 * e + 3] = v[c0 / 4 + e].w;
                }
                tmem_st16u(tmem + lane_base + Geo::kQCol + c0, r);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&q_full);
        };

        RowPair cur;
        bool ended = false;
        bool have = next_item(cur, ended);
        bool failed = !have && !ended;
        if (have)
            load_q(cur);
        while (have) {
            float m[2] = {-INFINITY, -INFINITY};
            float l[2] = {0.f, 0.f};  // this thread's columns only
            bool o_valid = false;
            const int npages = cur.npages;
            const int32_t *table =
                p.block_tables + static_cast<size_t>(cur.it.s) * p.max_blocks + cur.pg0;
            int ent = lane < npages ? __ldg(table + lane) : -1;
            int ent_next = 32 + lane < npages ? __ldg(table + 32 + lane) : -1;
            const int nchunks = (npages + kChunk - 1) / kChunk;
            const bool live = __any_sync(kFullMask, cur.ok[0] || cur.ok[1]);
            for (int j = 0; j < nchunks; ++j, ++gc) {
                const int jp = j * kChunk;
                if (jp > 0 && (jp & 31) == 0) {
                    ent = ent_next;
                    ent_next = jp + 32 + lane < npages ? __ldg(table + jp + 32 + lane) : -1;
                }
                bool good[kChunk];
                bool any_good = false;
#pragma unroll
                for (int x = 0; x < kChunk; ++x) {
                    const int phys = __shfl_sync(kFullMask, ent, (jp + x) & 31);
                    good[x] = jp + x < npages && phys >= 0 && phys < p.num_blocks;
                    any_good = any_good || good[x];
                }
                if (!warp_wait(&s_full[gc % SB], (gc / SB) & 1, abort)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t scol = tmem + lane_base + Geo::kSCol + Geo::kSCols * (gc % SB);
                const int tb = (cur.pg0 + jp) * kBlockSize;
                if (live) {
                    // xs[4 r + 2 x + e]: row x, column 8 r + 2 qd + e; scaled,
                    // -inf where the row does not see the token.
                    float xs[16];
                    tmem_ld_r16(scol, xs);
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int x = 0; x < 2; ++x)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int col = 8 * r + 2 * qd + e;
                                const bool vis = cur.ok[x] && good[r >> 1] && tb + col <= cur.pos[x];
                                xs[4 * r + 2 * x + e] = vis ? xs[4 * r + 2 * x + e] * c : -INFINITY;
                            }
                    float mx[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        float a = fmaxf(fmaxf(xs[2 * x], xs[2 * x + 1]),
                                        fmaxf(xs[4 + 2 * x], xs[5 + 2 * x]));
                        float b = fmaxf(fmaxf(xs[8 + 2 * x], xs[9 + 2 * x]),
                                        fmaxf(xs[12 + 2 * x], xs[13 + 2 * x]));
                        a = fmaxf(a, b);
                        a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 1));
                        mx[x] = fmaxf(a, __shfl_xor_sync(kFullMask, a, 2));
                    }
                    bool need_any = false;
                    float alpha[2] = {1.f, 1.f};
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        if (mx[x] > m[x] + kLazy) {  // false when nothing is visible
                            alpha[x] = m[x] == -INFINITY ? 0.f : MmaSoftmax::ex2(m[x] - mx[x]);
                            l[x] *= alpha[x];
                            m[x] = mx[x];
                            need_any = true;
                        }
                    }
                    if (o_valid && __any_sync(kFullMask, need_any)) {
                        // O holds earlier chunks: rescale it once their P V is done.
                        if (!warp_wait(&pv_done[(gc - 1) % SB], ((gc - 1) / SB) & 1, abort)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after();
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            float ov[16];
                            tmem_ld_r16(tmem + lane_base + c0, ov);
#pragma unroll
                            for (int r = 0; r < 4; ++r)
#pragma unroll
                                for (int x = 0; x < 2; ++x) {
                                    ov[4 * r + 2 * x] *= alpha[x];
                                    ov[4 * r + 2 * x + 1] *= alpha[x];
                                }
                            tmem_st_r16(tmem + lane_base + c0, ov);
                        }
                        tmem_wait_st();
                    }
                    // P over the consumed scores: high parts in the first
                    // half of the buffer, residuals in the second; column
                    // 4 r + qd of a row holds its tokens 8 r + 2 qd, + 1.
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int r = 0; r < 4; ++r)
#pragma unroll
                        for (int x = 0; x < 2; ++x) {
                            const bool seen = m[x] != -INFINITY;
                            const float a = seen ? MmaSoftmax::ex2(xs[4 * r + 2 * x] - m[x]) : 0.f;
                            const float b =
                                seen ? MmaSoftmax::ex2(xs[4 * r + 2 * x + 1] - m[x]) : 0.f;
                            l[x] += a + b;
                            const uint32_t w = pack_bf16(a, b);
                            hi[2 * r + x] = w;
                            lo[2 * r + x] = pack_bf16(a - bf16_lo(w), b - bf16_hi(w));
                        }
                    tmem_st_c8(scol, hi);
                    tmem_st_c8(scol + kTok / 2, lo);
                    tmem_wait_st();
                }  // live
                if (failed)
                    break;
                // Past the sequence end the V tile may hold anything (NaN):
                // zero those tokens, since P = 0 does not cancel NaN.
                bool zeroed = false;
#pragma unroll
                for (int x = 0; x < kChunk; ++x) {
                    const int valid = cur.it.L - (tb + 16 * x);
                    if (good[x] && valid > 0 && valid < kBlockSize) {
                        if (t < D) {
                            unsigned short *vt = reinterpret_cast<unsigned short *>(
                                smem + (gc % NS) * Geo::kStage + Geo::kVOff + x * Geo::kTile +
                                t * Geo::kRow);
                            const int sw = static_cast<int>(smem_u32(vt) >> 7) & 1;
                            for (int e = valid; e < kBlockSize; ++e)
                                vt[(((e >> 3) ^ sw) << 3) + (e & 7)] = 0;
                        }
                        zeroed = true;
                    }
                }
                if (zeroed)
                    fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&p_full[gc % SB]);
                o_valid = o_valid || any_good;
            }
            if (failed)
                break;

            RowPair nxt;
            bool nended = false;
            const bool have_next = next_item(nxt, nended);
            if (!have_next && !nended) {
                failed = true;
                break;
            }
            if (have_next)
                load_q(nxt);

            // ------------------------------------------------ output rows
            if (o_valid && live) {
                if (!warp_wait(&pv_done[(gc - 1) % SB], ((gc - 1) / SB) & 1, abort)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
            }
            float inv[2];
            bool write[2];
            int nparts_r[2];
            size_t orow[2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                l[x] += __shfl_xor_sync(kFullMask, l[x], 1);
                l[x] += __shfl_xor_sync(kFullMask, l[x], 2);
                nparts_r[x] = p.max_parts > 1 ? parts_of(cur.pos[x] + 1, p.partition) : 1;
                write[x] = cur.ok[x] && cur.it.part < nparts_r[x];
                inv[x] = l[x] > 0.f ? 1.f / l[x] : 0.f;
                orow[x] = static_cast<size_t>(cur.q0 + cur.qi[x]) * p.num_q_heads + cur.h[x];
            }
#pragma unroll 1
            for (int c0 = 0; c0 < (live ? D : 0); c0 += 32) {
                float ov[16];
                if (o_valid) {
                    tmem_ld_r16(tmem + lane_base + c0, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ov[e] = 0.f;
                }
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    if (!write[x])
                        continue;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int col = c0 + 8 * r + 2 * qd;
                        const float2 v = make_float2(ov[4 * r + 2 * x] * inv[x],
                                                     ov[4 * r + 2 * x + 1] * inv[x]);
                        if (nparts_r[x] == 1) {
                            store_out2(p, D, orow[x], col, v);
                        } else {
                            const size_t prow = orow[x] * p.max_parts + cur.it.part;
                            *reinterpret_cast<float2 *>(p.part_o + prow * D + col) = v;
                        }
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < 2; ++x)
                if (write[x] && nparts_r[x] > 1 && qd == 0) {
                    const size_t prow = orow[x] * p.max_parts + cur.it.part;
                    p.part_ml[2 * prow] = m[x];
                    p.part_ml[2 * prow + 1] = l[x];
                }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&o_free);
            cur = nxt;
            have = have_next;
        }
        if (failed)
            tc_fail(p, abort);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(Geo::kTmemCols)
                     : "memory");
    }
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Every [head_dim][16] tile of a bf16 cache, viewed as
// [num_blocks * num_kv_heads][head_dim][16]: one box is a page tile, stored
// in the 32-byte swizzle mode (the box's 32-byte rows fill the swizzle span).
bool encode_tile(EncodeTiledFn enc, CUtensorMap *map, const void *cache, int D, long tiles)
{
    const cuuint64_t dims[3] = {kBlockSize, static_cast<cuuint64_t>(D),
                                static_cast<cuuint64_t>(tiles)};
    const cuuint64_t strides[2] = {kBlockSize * 2, static_cast<cuuint64_t>(D) * kBlockSize * 2};
    const cuuint32_t box[3] = {kBlockSize, static_cast<cuuint32_t>(D), 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(cache), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int kTcRows, bool kPhased>
pkv_status launch_tc_d(const PrefillParams &p, cudaStream_t stream)
{
    using Geo = TcGeom<D>;
    // Resident CTAs per SM, once the attributes are set (per context).
    static ContextCache cache;
    int occ = 1;
    const pkv_status crc = cache.get(&occ, [](int *out_occ) -> pkv_status {
        // Two CTAs per SM need the largest shared-memory carveout.
        if (cudaFuncSetAttribute(prefill_tc_kernel<D, kTcRows, kPhased>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Geo::kSmem) != cudaSuccess ||
            cudaFuncSetAttribute(prefill_tc_kernel<D, kTcRows, kPhased>,
                                 cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return PKV_ERR_CUDA;
        // Resident CTAs per SM from the kernel's own resources (the
        // occupancy query reports one for this kernel on GB300, although
        // two fit and run: measured 605 -> 421 us on the 70B verification
        // layer): shared memory, registers and the 512 TMEM columns.
        cudaFuncAttributes fa;
        int dev = 0, smem_sm = 0, reserved = 0;
        if (cudaFuncGetAttributes(&fa, prefill_tc_kernel<D, kTcRows, kPhased>) != cudaSuccess ||
            cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
                cudaSuccess)
            return PKV_ERR_CUDA;
        const long per_cta = static_cast<long>(Geo::kSmem) + static_cast<long>(fa.sharedSizeBytes) +
                             reserved;
        const long by_smem = smem_sm / per_cta;
        const long regs = static_cast<long>((fa.numRegs * 32 + 255) / 256 * 256) * (kTcThreads / 32);
        const long by_regs = regs > 0 ? 65536 / regs : 1;
        long o = 512 / Geo::kTmemCols;
        o = o < by_smem ? o : by_smem;
        o = o < by_regs ? o : by_regs;
        *out_occ = o < 1 ? 1 : static_cast<int>(o);
        return PKV_OK;
    });
    if (crc != PKV_OK)
        return crc;
    EncodeTiledFn enc = encoder();
    if (!enc)
        return PKV_ERR_CUDA;
    const long tiles = static_cast<long>(p.num_blocks) * p.num_kv_heads;
    if (tiles >= (1L << 31))
        return PKV_ERR_UNSUPPORTED;
    TcMaps maps;
    if (!encode_tile(enc, &maps.k, p.k_cache, D, tiles) ||
        !encode_tile(enc, &maps.v, p.v_cache, D, tiles))
        return PKV_ERR_CUDA;
    const long blocks = (static_cast<long>(p.max_q_len) * p.group + kTcRows - 1) / kTcRows;
    const long items = static_cast<long>(p.num_seqs) * p.num_kv_heads * p.max_parts * blocks;
    const long slots = static_cast<long>(occ) * device_sm_count();
    const long grid = items < slots ? items : slots;
    if (grid <= 0)
        return PKV_OK;
    prefill_tc_kernel<D, kTcRows, kPhased><<<static_cast<unsigned>(grid), kTcThreads, Geo::kSmem, stream>>>(p, maps);
    if (cudaGetLastError() != cudaSuccess)
        return PKV_ERR_CUDA;
    return launch_prefill_merge(p, stream);
}

}  // namespace

pkv_status launch_prefill_tc(const PrefillParams &p, cudaStream_t stream)
{
    // 64-row items when every sequence's rows fit one (no padding to 128);
    // the size-ordered item phases when contexts are split.
    const bool m64 = static_cast<long>(p.max_q_len) * p.group <= 64;
    const bool split = p.max_parts > 1;
    if (p.head_dim == 128)
        return m64 ? (split ? launch_tc_d<128, 64, true>(p, stream)
                            : launch_tc_d<128, 64, false>(p, stream))
                   : (split ? launch_tc_d<128, 128, true>(p, stream)
                            : launch_tc_d<128, 128, false>(p, stream));
    return m64 ? (split ? launch_tc_d<64, 64, true>(p, stream)
                        : launch_tc_d<64, 64, false>(p, stream))
               : (split ? launch_tc_d<64, 128, true>(p, stream)
                        : launch_tc_d<64, 128, false>(p, stream));
}

}  // namespace pkv
