// Stream-K paged decode: the automatic schedule of the decode kernels.
//
// The work is the flattened page space: unit u = (layer l, sequence s, KV
// head hkv) in order u = (l*S + s)*Hkv + hkv, each contributing
// np_u = max(1, ceil(L_s/16)) pages (an empty sequence has one virtual page
// that copies nothing and yields a zero row); the layers share the lengths,
// so each layer spans the same number of pages.  With T pages in total and C resident CTAs, CTA c owns
// the contiguous page range [a_c, a_{c+1}), a_c = floor(c*T/C), so every CTA
// streams the same number of pages +-1 and the grid has no tail.
//
// Inside a CTA, warp w takes every fourth page of the range (w, w+4, ...) and
// streams them through its ring of bulk-copy stages continuously, across
// unit boundaries, so the copy engine never waits for bookkeeping.  The range
// cuts each unit it touches into a segment; at every segment end the four
// warps' online-softmax states are merged (shared memory).  A segment that is
// the whole unit writes the output rows; a unit cut by range boundaries
// leaves one partial per CTA that touches it -- only a CTA's first and last
// segments can be partial, so a CTA owns two partial slots -- and the CTA
// that writes the unit's last partial merges them with log-sum-exp weights,
// in CTA order (deterministic).
#pragma once

#include "pkv_decode.cuh"

namespace pkv {

// Pages of one unit (sequence length L after clamping).
__device__ __forceinline__ int unit_pages(int L) { return L > 0 ? (L + kBlockSize - 1) / kBlockSize : 1; }

// Block-wide sum of one int per thread (all threads get the result).
__device__ __forceinline__ long long block_sum(long long v, long long *red)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(kFullMask, v, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        red[threadIdx.x >> 5] = v;
    __syncthreads();
    long long t = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
        t += red[w];
    return t;
}

// New tokens listed per round of the fused cache write.
constexpr int kWriteBatch = 16;

// A unit of the flattened page space and its global page offset.
struct Unit {
    int layer, s, hkv, L, np;
    long long off;
};

// The next unit; past the last sequence of the last layer, s == num_seqs.
template <bool kMulti>
__device__ __forceinline__ void unit_next(const DecodeParams &p, Unit &u)
{
    u.off += u.np;
    if (++u.hkv == p.num_kv_heads) {
        u.hkv = 0;
        if (++u.s == p.num_seqs && kMulti && u.layer + 1 < p.num_layers) {
            u.s = 0;
            ++u.layer;
        }
        u.L = u.s < p.num_seqs ? seq_len_of(p, u.s) : 0;
        u.np = unit_pages(u.L);
    }
}

// CTA owning global page x when T pages are cut into C ranges
// (a_c = floor(c*T/C), requires T >= C): the largest c with a_c <= x.
__device__ __forceinline__ int owner_cta(long long x, long long T, int C)
{
    return static_cast<int>(((x + 1) * C - 1) / T);
}

__device__ __forceinline__ long long range_start(int c, long long T, int C)
{
    return static_cast<long long>(c) * T / C;
}

// Merges the partials of unit u = (s, hkv) of a layer, whose pages
// [off, off+np) were cut among CTAs c0..c1, and writes its output rows of
// that layer's `out`.
template <int D>
__device__ void merge_streamk_partials(const DecodeParams &p, void *out, int s, int hkv,
                                       long long off, int np, long long T, int C)
{
    constexpr int Q4 = D / 4;
    const int G = p.group;
    const int c0 = owner_cta(off, T, C), c1 = owner_cta(off + np - 1, T, C);
    const int slot0 = range_start(c0, T, C) < off ? 1 : 0;  // u is c0's last segment
    for (int idx = threadIdx.x; idx < G * Q4; idx += blockDim.x) {
        const int g = idx / Q4, q4 = idx - g * Q4;
        float mx = -INFINITY;
        for (int c = c0; c <= c1; ++c) {
            const size_t row = (static_cast<size_t>(c) * 2 + (c == c0 ? slot0 : 0)) * G + g;
            mx = fmaxf(mx, __ldcg(p.part_ml + 2 * row));
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float wsum = 0.f;
        for (int c = c0; c <= c1; ++c) {
            const size_t row = (static_cast<size_t>(c) * 2 + (c == c0 ? slot0 : 0)) * G + g;
            const float m = __ldcg(p.part_ml + 2 * row), l = __ldcg(p.part_ml + 2 * row + 1);
            const float w = (m == -INFINITY) ? 0.f : l * exp2f(m - mx);
            wsum += w;
            const float4 o = __ldcg(reinterpret_cast<const float4 *>(p.part_o + row * D) + q4);
            acc.x += w * o.x;
            acc.y += w * o.y;
            acc.z += w * o.z;
            acc.w += w * o.w;
        }
        const float sc = (wsum > 0.f ? 1.f / wsum : 0.f) * unit_out_scale(p, hkv);
        store_out4(p, out, D, s, hkv * G + g, q4,
                   make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc));
    }
}

// Combines the four warps' states of one segment (merge scratch) into the
// output rows of `out` (complete unit; null out: a skipped layer, nothing is
// written) or the CTA's partial slot `slot`.
template <int D, int GP>
__device__ void merge_segment(const DecodeParams &p, void *out, const float *scratch, int s,
                              int hkv, bool complete, int c, int slot)
{
    constexpr int Q4 = D / 4;
    constexpr int W = scratch_floats(GP, D);
    const int G = p.group;
    for (int idx = threadIdx.x; idx < G * Q4; idx += kThreads) {
        const int g = idx / Q4, q4 = idx - g * Q4;
        float mw[kWarps], mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            mw[w] = scratch[w * W + GP * D + g];
            mx = fmaxf(mx, mw[w]);
        }
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float *so = scratch + w * W;
            const float f = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - mx);
            const float4 o = reinterpret_cast<const float4 *>(so + g * D)[q4];
            acc.x += f * o.x;
            acc.y += f * o.y;
            acc.z += f * o.z;
            acc.w += f * o.w;
            lsum += f * so[GP * D + GP + g];
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        if (complete) {
            const float sc = inv * unit_out_scale(p, hkv);
            if (out)
                store_out4(p, out, D, s, hkv * G + g, q4,
                           make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc));
        } else {
            const size_t row = (static_cast<size_t>(c) * 2 + slot) * G + g;
            reinterpret_cast<float4 *>(p.part_o + row * D)[q4] =
                make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            if (q4 == 0) {
                p.part_ml[2 * row] = mx;
                p.part_ml[2 * row + 1] = lsum;
            }
        }
    }
}

// kMulti = false: the form for single-layer calls (layer logic compiled out).
template <class Pol, bool kMulti>
__global__ void __launch_bounds__(kThreads, 2)
    decode_streamk_kernel(const __grid_constant__ DecodeParams p)
{
    constexpr int D = Pol::kDim;
    constexpr int R = Pol::R;
    constexpr int kScratchFloats = scratch_floats(Pol::GP, D);
    static_assert(kScratchFloats % 4 == 0 && Pol::kExtraBytes % 16 == 0,
                  "merge scratch rows must stay 16-byte aligned");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ long long s_red[kWarps];
    __shared__ int s_start[4];  // start unit: s, hkv, L (in its layer); found flag
    __shared__ long long s_start_off;
    __shared__ int s_abort;
    __shared__ int s_last;
    __shared__ int s_w[kWriteBatch][5];  // fused write list: s, hkv, L, physical page, layer
    __shared__ int s_wn, s_wmore;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int Hkv = p.num_kv_heads;
    unsigned char *ring = smem + warp * Pol::kRingBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kWarps * Pol::kRingBytes) + warp * R;
    unsigned char *extra = smem + kWarps * Pol::kRingBytes + kWarps * R * sizeof(uint64_t);
    float *scratch = reinterpret_cast<float *>(extra + Pol::kExtraBytes);

    // ---------------------------------------------- this CTA's page range
    long long T1 = 0;  // pages of one layer
    for (int b0 = 0; b0 < p.num_seqs; b0 += kThreads) {
        long long v = 0;
        if (b0 + threadIdx.x < p.num_seqs)
            v = static_cast<long long>(Hkv) *
                unit_pages(seq_len_of(p, b0 + threadIdx.x));
        T1 += block_sum(v, s_red);
    }
    const long long T = T1 * (kMulti ? p.num_layers : 1);
    const int C = static_cast<int>(T < gridDim.x ? T : static_cast<long long>(gridDim.x));
    const int cta = blockIdx.x;
    if (cta >= C)
        return;  // uniform
    const long long a = range_start(cta, T, C), b = range_start(cta + 1, T, C);
    const int a_layer = kMulti ? static_cast<int>(a / T1) : 0;
    const long long a1 = a - a_layer * T1;  // page a inside its layer

    // Unit holding page a: scan the per-sequence page counts.
    if (threadIdx.x == 0)
        s_start[3] = 0;
    long long run = 0;
    for (int b0 = 0; b0 < p.num_seqs; b0 += kThreads) {
        const int sq = b0 + threadIdx.x;
        int Ls = 0;
        long long v = 0;
        if (sq < p.num_seqs) {
            Ls = seq_len_of(p, sq);
            v = static_cast<long long>(Hkv) * unit_pages(Ls);
        }
        // Block-wide inclusive scan of v (warp scans + warp offsets).
        long long incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long t = __shfl_up_sync(kFullMask, incl, off);
            if (lane >= off)
                incl += t;
        }
        __syncthreads();
        if (lane == 31)
            s_red[warp] = incl;
        __syncthreads();
        long long before = run;
        for (int w = 0; w < warp; ++w)
            before += s_red[w];
        const long long lo = before + incl - v, hi = before + incl;
        if (sq < p.num_seqs && lo <= a1 && a1 < hi) {
            const int np = unit_pages(Ls);
            const long long r = a1 - lo;
            s_start[0] = sq;
            s_start[1] = static_cast<int>(r / np);
            s_start[2] = Ls;
            s_start_off = a_layer * T1 + lo + (r / np) * np;
            s_start[3] = 1;
        }
        for (int w = 0; w < kWarps; ++w)
            run += s_red[w];
        __syncthreads();
        if (s_start[3])
            break;
    }

    if (!s_start[3]) {  // uniform; cannot happen for a < T, kept as a guard
        if (threadIdx.x == 0)
            set_status(p.status, PKV_ERR_OUT_OF_RANGE);
        return;
    }

    if (lane == 0)
        for (int st = 0; st < R; ++st)
            mbar_init(&bars[st], 1);
    if (threadIdx.x == 0)
        s_abort = 0;
    fence_mbar_init();
    __syncthreads();

    Unit start;
    start.layer = a_layer;
    start.s = s_start[0];
    start.hkv = s_start[1];
    start.L = s_start[2];
    start.np = unit_pages(start.L);
    start.off = s_start_off;

    const size_t tile_stride = static_cast<size_t>(Pol::kTileBytes);
    const size_t block_stride = static_cast<size_t>(Hkv) * tile_stride;

    // ---------------------------------------------- issue side (per warp)
    // This warp's pages are global pages a + warp + 4i, ring position i.
    Unit iu = start;
    int id_reg = -1, id_base = -1;
    // Cache bases of the issue unit's layer (a skipped layer copies nothing).
    int i_layer = -1;
    bool i_ok = false;
    const unsigned char *ikc = nullptr, *ivc = nullptr;
    uint32_t pos_i = 0, pos_c = 0;
    const uint32_t n_mine = (b - a > warp) ? static_cast<uint32_t>((b - a - warp + kWarps - 1) / kWarps) : 0u;
    uint32_t okmask = 0;

    auto issue_next = [&]() {
        const long long g = a + warp + static_cast<long long>(kWarps) * pos_i;
        while (g >= iu.off + iu.np) {
            unit_next<kMulti>(p, iu);
            id_base = -1;
        }
        const int pg = static_cast<int>(g - iu.off);
        // Cached ids cover pages id_base, id_base+4, ..., id_base+124 of the unit.
        if (id_base < 0 || pg < id_base || pg - id_base >= 4 * 32 || ((pg - id_base) & 3)) {
            id_base = pg;
            const int q = pg + 4 * lane;
            id_reg = (iu.L > 0 && q < iu.np)
                         ? __ldg(p.block_tables + static_cast<size_t>(iu.s) * p.max_blocks + q)
                         : -1;
        }
        const int phys = __shfl_sync(kFullMask, id_reg, (pg - id_base) >> 2);
        if (iu.layer != i_layer) {
            i_layer = iu.layer;
            const LayerPtrs lt = layer_ptrs<kMulti>(p, i_layer);
            i_ok = layer_usable<kMulti>(p, lt);
            ikc = static_cast<const unsigned char *>(lt.k_cache);
            ivc = static_cast<const unsigned char *>(lt.v_cache);
        }
        const int stg = pos_i % R;
        // A virtual page of an empty sequence, or a page of a skipped layer,
        // copies nothing.
        const bool real = iu.L > 0 && i_ok;
        const bool ok = real && phys >= 0 && phys < p.num_blocks;
        okmask = ok ? (okmask | (1u << stg)) : (okmask & ~(1u << stg));
        if (lane == 0) {
            uint64_t *bar = &bars[stg];
            if (!ok) {
                if (real)
                    set_status(p.status, PKV_ERR_OUT_OF_RANGE);
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, 2 * Pol::kTileBytes);
                const bool drop = p.drop_first_copy && cta == 0 && warp == 0 && pos_i == 0;
                if (!drop) {
                    const size_t off = static_cast<size_t>(phys) * block_stride +
                                       static_cast<size_t>(iu.hkv) * tile_stride;
                    unsigned char *dst = ring + stg * Pol::kStageBytes;
                    bulk_g2s(dst, ikc + off, Pol::kTileBytes, bar);
                    bulk_g2s(dst + Pol::kTileBytes, ivc + off, Pol::kTileBytes, bar);
                }
            }
        }
        ++pos_i;
    };
    auto refill = [&]() {
        while (pos_i < n_mine && pos_i < pos_c + R)
            issue_next();
    };

    // Fused cache write: the new tokens of the units whose last page lies in
    // this CTA's range are written before any page copy is issued, while HBM
    // is still idle.  Lane 0 of warp 0 lists them (with their physical page,
    // kWriteBatch at a time); all four warps then write the rows and fence
    // them against the copies the barrier releases.  (Writing them per warp,
    // where the page is copied, serialised several dependent loads of the
    // same warp under full memory load: about 7 us per token.)
    if (p.append) {
        Unit wu = start;
        for (;;) {
            if (threadIdx.x == 0) {
                int n = 0;
                while (wu.off < b && n < kWriteBatch) {
                    const long long g_last = wu.off + wu.np - 1;
                    const LayerPtrs wl = layer_ptrs<kMulti>(p, wu.layer);
                    if (wu.L > 0 && g_last >= a && g_last < b && wl.new_k != nullptr &&
                        layer_usable<kMulti>(p, wl)) {
                        const int phys = __ldg(p.block_tables +
                                               static_cast<size_t>(wu.s) * p.max_blocks + wu.np - 1);
                        if (phys >= 0 && phys < p.num_blocks) {
                            s_w[n][0] = wu.s;
                            s_w[n][1] = wu.hkv;
                            s_w[n][2] = wu.L;
                            s_w[n][3] = phys;
                            s_w[n][4] = wu.layer;
                            ++n;
                        }
                    }
                    unit_next<kMulti>(p, wu);
                }
                s_wn = n;
                s_wmore = (wu.off < b) ? 1 : 0;
            }
            __syncthreads();
            const int n = s_wn;
            write_token_rows<kMulti>(p, s_w, warp, n, kWarps, D, lane);
            fence_proxy_async_all();
            const int more = s_wmore;
            __syncthreads();  // the list is reused; every write is fenced
            if (!more)
                break;
        }
    }
    refill();

    // ---------------------------------------------- segments (all warps)
    Unit su = start;
    bool aborted = false;
    typename Pol::State st;
    // The query of a unit (null for a skipped layer or sequence: a zero
    // query) and its row of q.
    auto unit_q = [&](const Unit &u) -> const void * {
        const LayerPtrs lt = layer_ptrs<kMulti>(p, u.layer);
        if (!layer_usable<kMulti>(p, lt)) {
            if (threadIdx.x == 0)
                set_status(p.status, PKV_ERR_INVALID_ARG);
            return nullptr;
        }
        return unit_row(p, u.s) >= 0 ? lt.q : nullptr;
    };
    auto q_row = [&](const Unit &u) -> int {
        const int r = unit_row(p, u.s);
        return r >= 0 ? r : 0;
    };
    Pol::begin(st, p, unit_q(su), q_row(su), su.hkv, lane, extra);
    __syncthreads();  // policy shared data (SIMT query) is ready
    for (int k = 0;; ++k) {
        const float c = unit_score_scale(p, su.hkv);
        const long long lo = su.off > a ? su.off : a;
        const long long hi = (su.off + su.np < b) ? su.off + su.np : b;
        const bool complete = (lo == su.off) && (hi == su.off + su.np);
        const bool last = hi >= b;

        // This warp's pages of the segment: g in [lo, hi), g == a + warp (mod 4).
        long long g = lo + ((warp - ((lo - a) & 3)) & 3);
        for (; g < hi && !aborted; g += kWarps) {
            const int stg = pos_c % R;
            const uint32_t parity = (pos_c / R) & 1u;
            const bool ok = mbar_wait_bounded(&bars[stg], parity, kWaitLimitNs);
            if (!__all_sync(kFullMask, ok)) {
                if (lane == 0) {
                    set_status(p.status, PKV_ERR_TIMEOUT);
                    atomicExch(&s_abort, 1);
                }
                for (uint32_t q = pos_c + 1; q < pos_i; ++q)
                    mbar_wait_bounded(&bars[q % R], (q / R) & 1u, kWaitLimitNs);
                aborted = true;
                break;
            }
            const bool have = (okmask >> stg) & 1u;
            const int pg = static_cast<int>(g - su.off);
            const int valid = min(kBlockSize, su.L - pg * kBlockSize);
            const unsigned char *sk = ring + stg * Pol::kStageBytes;
            typename Pol::Frags fr;
            if (have) {
                if constexpr (Pol::kStaged)
                    Pol::load(fr, sk, sk + Pol::kTileBytes, lane);
                else
                    Pol::page(st, sk, sk + Pol::kTileBytes, valid, lane, warp, extra, c);
            }
            ++pos_c;
            // The stage is free: reads are ordered before the next bulk copy.
            fence_proxy_async();
            __syncwarp();
            refill();
            if constexpr (Pol::kStaged)
                if (have)
                    Pol::compute(st, fr, valid, lane, c);
        }

        // ------------------------------------------ merge the segment
        float *mine = scratch + warp * kScratchFloats;
        Pol::finish(st, mine, mine + Pol::GP * D, mine + Pol::GP * D + Pol::GP, lane);
        Unit nu = su;
        if (!last)
            unit_next<kMulti>(p, nu);
        // Register-only policies start the next segment's query loads now, so
        // their latency overlaps the merge below.
        if constexpr (!Pol::kSharedBegin)
            if (!last)
                Pol::begin(st, p, unit_q(nu), q_row(nu), nu.hkv, lane, extra);
        __syncthreads();
        const int slot = (k == 0) ? 0 : 1;
        const LayerPtrs sl = layer_ptrs<kMulti>(p, su.layer);
        void *sout = layer_usable<kMulti>(p, sl) ? sl.out : nullptr;
        merge_segment<D, Pol::GP>(p, sout, scratch, su.s, su.hkv, complete, cta, slot);
        if (!complete) {
            // Publish this partial; the CTA writing the unit's last partial
            // merges them all.  The barrier orders every thread's partial
            // writes before thread 0's gpu-scope fence and arrival.
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();
                const int n_ch =
                    owner_cta(su.off + su.np - 1, T, C) - owner_cta(su.off, T, C) + 1;
                const size_t gs = static_cast<size_t>(su.layer) * p.num_seqs + su.s;
                const unsigned old = atomicAdd(p.arrive + gs * Hkv + su.hkv, 1u);
                s_last = (old == static_cast<unsigned>(n_ch - 1)) ? 1 : 0;
            }
            __syncthreads();
            if (s_last && sout) {
                __threadfence();
                merge_streamk_partials<D>(p, sout, su.s, su.hkv, su.off, su.np, T, C);
            }
        }
        __syncthreads();  // scratch is free again
        if (*static_cast<volatile int *>(&s_abort) || aborted) {
            if (!aborted)
                for (uint32_t q = pos_c; q < pos_i; ++q)
                    mbar_wait_bounded(&bars[q % R], (q / R) & 1u, kWaitLimitNs);
            break;
        }
        if (last)
            break;
        su = nu;
        if constexpr (Pol::kSharedBegin) {
            Pol::begin(st, p, unit_q(su), q_row(su), su.hkv, lane, extra);
            __syncthreads();  // policy shared data (SIMT query) is ready
        }
    }
}

template <class Pol, bool kMulti>
pkv_status launch_streamk(const DecodeParams &p, cudaStream_t stream)
{
    constexpr int smem = kWarps * Pol::kRingBytes + kWarps * Pol::R * 8 + Pol::kExtraBytes +
                         scratch_bytes(Pol::GP, Pol::kDim);
    // Resident CTAs per SM, once the shared-memory attribute is set (per context).
    static ContextCache cache;
    int occ = 1;
    const pkv_status rc = cache.get(&occ, [](int *v) -> pkv_status {
        if (cudaFuncSetAttribute(decode_streamk_kernel<Pol, kMulti>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        int o = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, decode_streamk_kernel<Pol, kMulti>, kThreads,
                                                          smem) != cudaSuccess)
            return PKV_ERR_CUDA;
        *v = o > 0 ? o : 1;
        return PKV_OK;
    });
    if (rc != PKV_OK)
        return rc;
    long grid = static_cast<long>(occ) * device_sm_count();
    if (grid > p.streamk_max_ctas)
        grid = p.streamk_max_ctas;
    if (grid <= 0 || p.num_seqs <= 0)
        return PKV_OK;
    decode_streamk_kernel<Pol, kMulti><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// The schedule the call asked for: stream-K, or items (one per (sequence,
// KV head), or fixed partitions).
template <class Pol>
pkv_status launch_any(const DecodeParams &p, cudaStream_t stream)
{
    // Single-layer calls of the tensor-core policies run the form with the
    // layer logic compiled out.
    if constexpr (Pol::kSingleForm)
        if (p.layers == nullptr)
            return p.streamk ? launch_streamk<typename Pol::StreamK, false>(p, stream)
                             : launch_policy<Pol, false>(p, stream);
    return p.streamk ? launch_streamk<typename Pol::StreamK, true>(p, stream)
                     : launch_policy<Pol, true>(p, stream);
}

}  // namespace pkv
