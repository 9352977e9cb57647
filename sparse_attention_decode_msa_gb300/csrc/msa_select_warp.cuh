// msa_select_warp.cuh -- the warp select of one row of block scores (rows of
// up to 2048 blocks): the per-token select kernel and the prefill select
// tile use it.
//
// Contract ("MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2
// for Blackwell", section "The TP4 decode target"): the k blocks with the
// largest block score, ties toward the smaller block index, for any tie
// width; ascending, -1 padded ("Add Rubin (sm_107) MiniMax-M3.1 low-latency
// decode targets", q8kv4 indexer commit).  Lane l holds the order-preserving
// keys of blocks l, l + 32, ... in registers; a threshold search finds the
// k-th largest key theta (warp_select_keys).  The selection pass walks the
// blocks in index order 32 at a time; ballots give each tie its rank and each
// selected block its output slot, so the table comes out ascending.
// Comparisons only: bit-exact.
#pragma once

#include "msa_internal.cuh"

namespace msa {

constexpr int kWarpSelMaxN = 2048; // longest row of the warp select

// The k largest of a warp's row of keys (lane holds keys of blocks lane,
// lane + 32, ...; 0 for blocks past the row, below every key of a block of
// the row, which are all >= 1), ties to the smaller block: out[0..k)
// ascending.  Requires more than k candidate blocks.
//
// theta, the k-th largest key, is built from the top: a bit is kept while
// at least k keys are >= the candidate.  Bits that every key of the row has
// are set from the start and bits that none has are never tried: with
// them in place the count of keys >= a candidate is the one the plain
// bit-by-bit search sees (a key that matches theta above the tried bit and
// has it set also has every common bit below it).  The other bits are
// decided two at a time from three independent warp-wide counts.
template <int S>
__device__ __forceinline__ void warp_select_keys(const uint32_t (&key)[S], int k, int32_t *out)
{
    const int lane = threadIdx.x & 31;
    uint32_t k_or = 0u, k_and = 0xFFFFFFFFu;
#pragma unroll
    for (int s = 0; s < S; ++s) {
        k_or |= key[s];
        k_and &= key[s] ? key[s] : 0xFFFFFFFFu; // blocks past the row do not count
    }
    k_or = __reduce_or_sync(0xffffffffu, k_or);
    k_and = __reduce_and_sync(0xffffffffu, k_and);
    uint32_t theta = k_and;
    uint32_t open = k_or & ~k_and; // bits in which the row's keys differ
    auto count_ge = [&](uint32_t cand) {
        int c0 = 0, c1 = 0;
#pragma unroll
        for (int s = 0; s < S; s += 2) {
            c0 += key[s] >= cand;
            c1 += key[s + 1] >= cand;
        }
        return c0 + c1;
    };
#pragma unroll 1
    while (open) {
        const uint32_t hb = 1u << (31 - __clz(open)); // highest open bit
        open &= ~hb;
        if (!open) {
            if ((int)__reduce_add_sync(0xffffffffu, (unsigned)count_ge(theta | hb)) >= k)
                theta |= hb;
            break;
        }
        const uint32_t lb = 1u << (31 - __clz(open)); // the next one
        open &= ~lb;
        const int n_h = (int)__reduce_add_sync(0xffffffffu, (unsigned)count_ge(theta | hb));
        const int n_hl = (int)__reduce_add_sync(0xffffffffu, (unsigned)count_ge(theta | hb | lb));
        const int n_l = (int)__reduce_add_sync(0xffffffffu, (unsigned)count_ge(theta | lb));
        if (n_h >= k)
            theta |= hb | (n_hl >= k ? lb : 0u);
        else if (n_l >= k)
            theta |= lb;
    }
    int gt = 0;
#pragma unroll
    for (int s = 0; s < S; ++s)
        gt += key[s] > theta;
    // blocks equal to theta still needed, taken in index order
    const int need = k - (int)__reduce_add_sync(0xffffffffu, (unsigned)gt);
    const uint32_t below = (1u << lane) - 1u;
    int ties = 0, slot = 0;
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const bool eq = key[s] == theta;
        const uint32_t em = __ballot_sync(0xffffffffu, eq);
        const bool sel = key[s] > theta || (eq && ties + __popc(em & below) < need);
        ties += __popc(em);
        const uint32_t sm = __ballot_sync(0xffffffffu, sel);
        if (sel)
            out[slot + __popc(sm & below)] = lane + 32 * s;
        slot += __popc(sm);
    }
}

// Row x (token t = x / Hs, selection head gs = x % Hs) by one warp: its keys
// are the largest order-preserving key of block b over the selection head's
// index heads, forced blocks (the first `init` and the last `local` visible
// blocks) the largest key of all.  grid_wait: the block scores come from the
// previous kernel of the step (a programmatic dependent launch).  The row is
// read from L2.
template <int S>
__device__ __forceinline__ void warp_select_row(const SelectParams &p, int x, bool grid_wait)
{
    const int lane = threadIdx.x & 31;
    const int t = x / p.Hs, gs = x - t * p.Hs;
    const int r = t / p.nq, j = t - r * p.nq;
    int32_t *out = p.selected + (size_t)x * p.k;
    const int seq_len = p.seq_lens[r];
    const long long nb_req = ((long long)seq_len + p.nq - 1 + kPage - 1) / kPage;
    if (seq_len < 1 || nb_req > p.maxB) {
        if (lane == 0)
            set_error(p.err, kErrSeqLen);
        for (int i = lane; i < p.k; i += 32)
            out[i] = -1;
        return;
    }
    const int n = ceil_div(seq_len + j, kPage);
    if (n <= p.k) {
        for (int i = lane; i < p.k; i += 32)
            out[i] = i < n ? i : -1;
        return;
    }
    if (grid_wait)
        grid_dependency_wait(); // block_scores come from the previous kernel of the step
    const float *row = p.block_scores + ((size_t)t * p.Hi + (size_t)gs * p.r) * p.maxB;
    // every load of the row first, then the group maximum, then the forcing
    float v[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int b = lane + 32 * s;
        v[s] = b < n ? __ldcg(row + b) : 0.f;
    }
    uint32_t key[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int b = lane + 32 * s;
        // blocks past n take key 0, below every candidate tried (all >= 1)
        key[s] = b < n ? order_key(v[s]) : 0u;
    }
    for (int i = 1; i < p.r; ++i) { // the selection head's other index heads
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int b = lane + 32 * s;
            v[s] = b < n ? __ldcg(row + (size_t)i * p.maxB + b) : 0.f;
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int b = lane + 32 * s;
            const uint32_t k2 = b < n ? order_key(v[s]) : 0u;
            key[s] = k2 > key[s] ? k2 : key[s];
        }
    }
    if (p.init > 0 || p.local > 0) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int b = lane + 32 * s;
            if (b < n && (b < p.init || b >= n - p.local))
                key[s] = 0xFFFFFFFFu; // forced: above every score
        }
    }
    warp_select_keys<S>(key, p.k, out);
}

// The same select by the W warps of a CTA for rows longer than a warp
// handles quickly: warp w holds blocks w * 32 SW + lane + 32 s (s < SW), a
// contiguous range.  The threshold search is the one above with the counts
// summed over the warps through shared memory (red: 2 * W * 4 words, one
// barrier a step; the two halves alternate, so a warp writes a half again
// only after every warp has read it at the previous barrier).  The selection
// pass needs, per warp, the keys above theta and equal to theta in the warps
// before it: with those each warp walks its range in index order as above.
template <int SW, int W>
__device__ __forceinline__ void cta_select_keys(const uint32_t (&key)[SW], int k, int32_t *out,
                                                uint32_t *red)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t k_or = 0u, k_and = 0xFFFFFFFFu;
#pragma unroll
    for (int s = 0; s < SW; ++s) {
        k_or |= key[s];
        k_and &= key[s] ? key[s] : 0xFFFFFFFFu; // blocks past the row do not count
    }
    k_or = __reduce_or_sync(0xffffffffu, k_or);
    k_and = __reduce_and_sync(0xffffffffu, k_and);
    if (lane == 0) {
        red[4 * w] = k_or;
        red[4 * w + 1] = k_and;
    }
    __syncthreads();
    k_or = 0u;
    k_and = 0xFFFFFFFFu;
#pragma unroll
    for (int v = 0; v < W; ++v) {
        k_or |= red[4 * v];
        k_and &= red[4 * v + 1];
    }
    uint32_t theta = k_and;
    uint32_t open = k_or & ~k_and; // bits in which the row's keys differ
    auto count_ge = [&](uint32_t cand) {
        int c0 = 0;
#pragma unroll
        for (int s = 0; s < SW; ++s)
            c0 += key[s] >= cand;
        return (uint32_t)c0;
    };
    int half = 1; // red[0 .. 4W) held the common bits: start in the other half
#pragma unroll 1
    while (open) {
        uint32_t *rd = red + half * 4 * W;
        const uint32_t hb = 1u << (31 - __clz(open)); // highest open bit
        open &= ~hb;
        const uint32_t lb = open ? 1u << (31 - __clz(open)) : 0u; // the next one, if any
        open &= ~lb;
        const uint32_t c_h = __reduce_add_sync(0xffffffffu, count_ge(theta | hb));
        const uint32_t c_hl = lb ? __reduce_add_sync(0xffffffffu, count_ge(theta | hb | lb)) : 0u;
        const uint32_t c_l = lb ? __reduce_add_sync(0xffffffffu, count_ge(theta | lb)) : 0u;
        if (lane == 0) {
            rd[4 * w] = c_h;
            rd[4 * w + 1] = c_hl;
            rd[4 * w + 2] = c_l;
        }
        __syncthreads();
        int n_h = 0, n_hl = 0, n_l = 0;
#pragma unroll
        for (int v = 0; v < W; ++v) {
            n_h += (int)rd[4 * v];
            n_hl += (int)rd[4 * v + 1];
            n_l += (int)rd[4 * v + 2];
        }
        if (n_h >= k)
            theta |= hb | (lb && n_hl >= k ? lb : 0u);
        else if (lb && n_l >= k)
            theta |= lb;
        half ^= 1;
    }
    int gt = 0, eq = 0;
#pragma unroll
    for (int s = 0; s < SW; ++s) {
        gt += key[s] > theta;
        eq += key[s] == theta;
    }
    gt = (int)__reduce_add_sync(0xffffffffu, (unsigned)gt);
    eq = (int)__reduce_add_sync(0xffffffffu, (unsigned)eq);
    uint32_t *rd = red + half * 4 * W;
    if (lane == 0) {
        rd[4 * w] = (uint32_t)gt;
        rd[4 * w + 1] = (uint32_t)eq;
    }
    __syncthreads();
    int gt_all = 0;
#pragma unroll
    for (int v = 0; v < W; ++v)
        gt_all += (int)rd[4 * v];
    // blocks equal to theta still needed, taken in index order over the warps
    const int need = k - gt_all;
    int ties = 0, slot = 0;
    for (int v = 0; v < w; ++v) {
        const int eq_v = (int)rd[4 * v + 1];
        const int take = min(eq_v, max(0, need - ties));
        slot += (int)rd[4 * v] + take;
        ties += eq_v;
    }
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int s = 0; s < SW; ++s) {
        const bool e = key[s] == theta;
        const uint32_t em = __ballot_sync(0xffffffffu, e);
        const bool sel = key[s] > theta || (e && ties + __popc(em & below) < need);
        ties += __popc(em);
        const uint32_t sm = __ballot_sync(0xffffffffu, sel);
        if (sel)
            out[slot + __popc(sm & below)] = w * 32 * SW + lane + 32 * s;
        slot += __popc(sm);
    }
}

// Row x by the W warps of a CTA (warp_select_row's contract and steps, with
// warp w holding blocks w * 32 SW + lane + 32 s).  Every early exit depends
// on the row only, so the CTA's threads take it together.
template <int SW, int W>
__device__ __forceinline__ void cta_select_row(const SelectParams &p, int x, uint32_t *red)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int t = x / p.Hs, gs = x - t * p.Hs;
    const int r = t / p.nq, j = t - r * p.nq;
    int32_t *out = p.selected + (size_t)x * p.k;
    const int seq_len = p.seq_lens[r];
    const long long nb_req = ((long long)seq_len + p.nq - 1 + kPage - 1) / kPage;
    if (seq_len < 1 || nb_req > p.maxB) {
        if (threadIdx.x == 0)
            set_error(p.err, kErrSeqLen);
        for (int i = threadIdx.x; i < p.k; i += 32 * W)
            out[i] = -1;
        return;
    }
    const int n = ceil_div(seq_len + j, kPage);
    if (n <= p.k) {
        for (int i = threadIdx.x; i < p.k; i += 32 * W)
            out[i] = i < n ? i : -1;
        return;
    }
    grid_dependency_wait(); // block_scores come from the previous kernel of the step
    const float *row = p.block_scores + ((size_t)t * p.Hi + (size_t)gs * p.r) * p.maxB;
    const int b0 = w * 32 * SW + lane;
    float v[SW];
#pragma unroll
    for (int s = 0; s < SW; ++s) {
        const int b = b0 + 32 * s;
        v[s] = b < n ? __ldcg(row + b) : 0.f;
    }
    uint32_t key[SW];
#pragma unroll
    for (int s = 0; s < SW; ++s) {
        const int b = b0 + 32 * s;
        key[s] = b < n ? order_key(v[s]) : 0u; // 0: below every candidate tried
    }
    for (int i = 1; i < p.r; ++i) { // the selection head's other index heads
#pragma unroll
        for (int s = 0; s < SW; ++s) {
            const int b = b0 + 32 * s;
            v[s] = b < n ? __ldcg(row + (size_t)i * p.maxB + b) : 0.f;
        }
#pragma unroll
        for (int s = 0; s < SW; ++s) {
            const int b = b0 + 32 * s;
            const uint32_t k2 = b < n ? order_key(v[s]) : 0u;
            key[s] = k2 > key[s] ? k2 : key[s];
        }
    }
    if (p.init > 0 || p.local > 0) {
#pragma unroll
        for (int s = 0; s < SW; ++s) {
            const int b = b0 + 32 * s;
            if (b < n && (b < p.init || b >= n - p.local))
                key[s] = 0xFFFFFFFFu; // forced: above every score
        }
    }
    cta_select_keys<SW, W>(key, p.k, out, red);
}

} // namespace msa
