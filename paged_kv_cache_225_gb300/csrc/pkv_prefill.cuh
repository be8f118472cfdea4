// Work items of the several-queries kernels (pkv_prefill.cu, the mma.sync
// form, and pkv_prefill_tc.cu, the tcgen05 form): a sequence's n queries x G
// grouped heads are its rows; an item is (sequence, KV head, partition of
// the context, block of RB rows).
#pragma once

#include "pkv_decode.cuh"

namespace pkv {

struct SeqInfo {
    int L;   // cached tokens (the queries included)
    int q0;  // first query row in q
    int nq;  // queries (0 when the sequence's arguments are invalid)
};

__device__ __forceinline__ SeqInfo seq_info(const PrefillParams &p, int s)
{
    SeqInfo si;
    int L = __ldg(p.seq_lens + s);
    if (L < 0 || L > p.max_len) {
        set_status(p.status, PKV_ERR_OUT_OF_RANGE);
        L = L < 0 ? 0 : p.max_len;
    }
    const int a = __ldg(p.q_start + s), b = __ldg(p.q_start + s + 1);
    si.L = L;
    si.q0 = a;
    si.nq = b - a;
    if (a < 0 || b > p.num_tokens || b < a || b - a > L || b - a > p.max_q_len) {
        set_status(p.status, PKV_ERR_OUT_OF_RANGE);
        si.q0 = 0;
        si.nq = 0;
    }
    return si;
}

__device__ __forceinline__ int seq_parts(const PrefillParams &p, int L)
{
    return p.max_parts > 1 ? parts_of(L, p.partition) : 1;
}

// Items of sequence s: KV heads x partitions x row blocks of RB rows.
template <int RB>
__device__ __forceinline__ int seq_item_count(const PrefillParams &p, const SeqInfo &si)
{
    if (p.skip_single && si.nq == 1)
        return 0;  // served by the decode kernels
    const int blocks = (si.nq * p.group + RB - 1) / RB;
    return p.num_kv_heads * seq_parts(p, si.L) * blocks;
}

struct PrefillItem {
    int s, hkv, part, rb, L, q0, nq;
};

// Warp-collective: maps item index u to its (sequence, KV head, partition,
// row block of RB rows).  (cur_s, cur_base) keep the scan position between
// calls; u only grows.  Returns false past the last item.
template <int RB>
__device__ bool find_prefill_item(const PrefillParams &p, int u, int &cur_s, int &cur_base,
                                  int lane, PrefillItem &it)
{
    const int S = p.num_seqs;
    for (;;) {
        const int sl = cur_s + lane;
        int n = 0;
        SeqInfo si = {0, 0, 0};
        if (sl < S) {
            si = seq_info(p, sl);
            n = seq_item_count<RB>(p, si);
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
            it.s = cur_s + ln;
            it.L = __shfl_sync(kFullMask, si.L, ln);
            it.q0 = __shfl_sync(kFullMask, si.q0, ln);
            it.nq = __shfl_sync(kFullMask, si.nq, ln);
            const int k = u - cur_base - excl;
            const int blocks = (it.nq * p.group + RB - 1) / RB;
            const int parts = seq_parts(p, it.L);
            it.rb = k % blocks;
            it.part = (k / blocks) % parts;
            it.hkv = k / (blocks * parts);
            return true;
        }
        if (cur_s + 32 >= S)
            return false;
        cur_base += tot;
        cur_s += 32;
    }
}


// Phases of the items for the tcgen05 kernel: every partition of a sequence
// but its last first, then the last partitions in three size classes,
// largest first (size relative to the partition length, or to max_len when
// contexts are not split), so that the grid ends on short items.
constexpr int kPrefillPhases = 4;
__device__ __forceinline__ int prefill_phase_parts(const PrefillParams &p, int L, int ph)
{
    const int parts = seq_parts(p, L);
    if (ph == 0)
        return parts - 1;
    const bool split = p.max_parts > 1;
    const int span = split ? p.partition : (p.max_len > 0 ? p.max_len : 1);
    const int rem = split ? L - (parts - 1) * p.partition : L;  // in [0, span]
    constexpr int nc = kPrefillPhases - 1;
    int cls = 1 + (nc - 1) - static_cast<int>((static_cast<long long>(rem) * nc) / span);
    cls = cls < 1 ? 1 : (cls > nc ? nc : cls);
    return cls == ph ? 1 : 0;
}

// Items of sequence si in phase ph: KV heads x its partitions of the phase x
// row blocks of RB rows.
template <int RB>
__device__ __forceinline__ int seq_phase_items(const PrefillParams &p, const SeqInfo &si, int ph)
{
    if (p.skip_single && si.nq == 1)
        return 0;  // served by the decode kernels
    const int blocks = (si.nq * p.group + RB - 1) / RB;
    return p.num_kv_heads * prefill_phase_parts(p, si.L, ph) * blocks;
}

// Items of each phase over all sequences (warp-collective).
template <int RB>
__device__ __forceinline__ void count_prefill_phases(const PrefillParams &p, int lane,
                                                     int (&n)[kPrefillPhases])
{
#pragma unroll
    for (int ph = 0; ph < kPrefillPhases; ++ph)
        n[ph] = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
        SeqInfo si = {0, 0, 0};
        if (s0 + lane < p.num_seqs)
            si = seq_info(p, s0 + lane);
#pragma unroll
        for (int ph = 0; ph < kPrefillPhases; ++ph) {
            int c = seq_phase_items<RB>(p, si, ph);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                c += __shfl_xor_sync(kFullMask, c, off);
            n[ph] += c;
        }
    }
}

// Warp-collective: maps item u of phase ph to its (sequence, KV head,
// partition, row block), with that phase's scan position (cur_s, cur_base);
// u only grows within a phase.  Returns false past the phase's last item.
template <int RB>
__device__ bool find_prefill_item_phase(const PrefillParams &p, int u, int ph, int &cur_s,
                                        int &cur_base, int lane, PrefillItem &it)
{
    const int S = p.num_seqs;
    for (;;) {
        const int sl = cur_s + lane;
        int n = 0;
        SeqInfo si = {0, 0, 0};
        if (sl < S) {
            si = seq_info(p, sl);
            n = seq_phase_items<RB>(p, si, ph);
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
            it.s = cur_s + ln;
            it.L = __shfl_sync(kFullMask, si.L, ln);
            it.q0 = __shfl_sync(kFullMask, si.q0, ln);
            it.nq = __shfl_sync(kFullMask, si.nq, ln);
            const int k = u - cur_base - excl;
            const int blocks = (it.nq * p.group + RB - 1) / RB;
            const int parts = seq_parts(p, it.L);
            it.rb = k % blocks;
            if (ph == 0) {
                it.part = (k / blocks) % (parts - 1);
                it.hkv = k / (blocks * (parts - 1));
            } else {
                it.part = parts - 1;
                it.hkv = k / blocks;
            }
            return true;
        }
        if (cur_s + 32 >= S)
            return false;
        cur_base += tot;
        cur_s += 32;
    }
}

// Pages of an item: the context partition [t0, t1) cut at the last position
// any of its rows sees.  pg0 is the first page's index in the block table.
__device__ __forceinline__ void item_pages(const PrefillParams &p, int L, int nq, int row0,
                                           int nrows, int part, int &pg0, int &npages)
{
    const int pos_max = (L - nq) + (row0 + nrows - 1) / p.group;
    const int t0 = part * p.partition;
    int t1 = t0 + p.partition < L ? t0 + p.partition : L;
    t1 = t1 < pos_max + 1 ? t1 : pos_max + 1;
    pg0 = t0 / kBlockSize;
    npages = t1 > t0 ? (t1 - t0 + kBlockSize - 1) / kBlockSize : 0;
}

// Log-sum-exp merge of the rows whose context spans several partitions
// (pkv_prefill.cu).
pkv_status launch_prefill_merge(const PrefillParams &p, cudaStream_t stream);

}  // namespace pkv
