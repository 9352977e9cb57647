// msa_select_warp.cuh -- the warp select of one row of block scores (rows of
// up to 2048 blocks): the per-token select kernel and the prefill select
// tile use it.
//
// Contract ("MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2
// for Blackwell", section "The TP4 decode target"): the k blocks with the
// largest block score, ties toward the smaller block index, for any tie
// width; ascending, -1 padded ("Add Rubin (sm_107) MiniMax-M3.1 low-latency
// decode targets", q8kv4 indexer commit).  Lane l holds the order-preserving
// keys of blocks l, l + 32, ... in registers.  theta, the k-th largest key, is
// built bit by bit from the top: a bit is kept while at least k keys are >=
// the candidate (a warp-wide sum per bit).  The selection pass walks the
// blocks in index order 32 at a time; ballots give each tie its rank and each
// selected block its output slot, so the table comes out ascending.
// Comparisons only: bit-exact.
#pragma once

#include "msa_internal.cuh"

namespace msa {

constexpr int kWarpSelMaxN = 2048; // longest row of the warp select

// The k largest of a warp's row of keys (lane holds keys of blocks lane,
// lane + 32, ...; 0 below every candidate), ties to the smaller block:
// out[0..k) ascending.  Requires more than k candidate blocks.
template <int S>
__device__ __forceinline__ void warp_select_keys(const uint32_t (&key)[S], int k, int32_t *out)
{
    const int lane = threadIdx.x & 31;
    uint32_t theta = 0;
#pragma unroll 1
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = theta | (1u << bit);
        int c0 = 0, c1 = 0;
#pragma unroll
        for (int s = 0; s < S; s += 2) {
            c0 += key[s] >= cand;
            c1 += key[s + 1] >= cand;
        }
        if ((int)__reduce_add_sync(0xffffffffu, (unsigned)(c0 + c1)) >= k)
            theta = cand;
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

} // namespace msa
