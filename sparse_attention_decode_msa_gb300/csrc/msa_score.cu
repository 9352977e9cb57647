// msa_score.cu -- stage (a): index scores and the per-block max.
//
// "MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2 for
// Blackwell", section "The TP4 decode target": an index scorer streams the
// index-K pages; the prefill-select commit of "Add Rubin (sm_107) MiniMax-M3.1
// low-latency decode targets" keeps one max score per 128-token block.  Here
// the per-token scores never reach memory: each page is scored and reduced to
// its block max in registers.
//
// The dot products run on the tensor cores (mma.sync m16n8k16) with the page's
// 16-token row tiles as M and the request's query tokens as N.  Inputs are
// integer-valued (bf16) or NVFP4 with power-of-two scales, so every product
// and partial sum is exact in fp32 and the result equals the plain dot product
// bit for bit, whatever the summation order.  Because the K dimension is a
// pure sum, each thread may take its index-key dimensions in whatever order
// makes its global loads coalesced, provided the query fragment follows the
// same order.
//
// Work decomposition: one item = PPI consecutive pages of one request, one CTA
// of 4 warps per item in a grid-stride loop; each warp owns 2 row tiles of
// every page of the item and issues all of its 16-byte loads before the first
// mma, so a CTA keeps PPI * 32 KiB (bf16) of index keys in flight.
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kScoreThreads = 128;

// items of request r = ceil(nb_r / PPI); invalid requests get 0 items.
template <int PPI>
__device__ void build_item_prefix(const ScoreParams &p, int *prefix)
{
    // warp 0 scans R values, 32 at a time
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base < p.R; base += 32) {
            const int r = base + lane;
            int items = 0;
            if (r < p.R) {
                const int sl = p.seq_lens[r];
                const long long cached = (long long)sl + p.nq - 1;
                const long long nb = (cached + kPage - 1) / kPage;
                if (sl < 1 || nb > p.maxB) {
                    if (blockIdx.x == 0)
                        set_error(p.err, kErrSeqLen);
                } else {
                    items = (int)((nb + PPI - 1) / PPI);
                }
            }
            int incl = items;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (r < p.R)
                prefix[r] = carry + incl - items;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            prefix[p.R] = carry;
    }
    __syncthreads();
}

// Score kernel.  NVFP4 selects the index-key format; NT = n-tiles of 8 query
// tokens; PPI = pages per item.
template <bool NVFP4, int NT, int PPI>
__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(const ScoreParams p)
{
    extern __shared__ int item_prefix[]; // [R + 1]
    __shared__ float red[4][PPI][NT * 8];

    launch_dependents(); // the select may start its prologue while pages are scored
    build_item_prefix<PPI>(p, item_prefix);
    const int total = item_prefix[p.R];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2; // row within an 8-row group; query (n) index in B
    const int q = lane & 3;
    constexpr int MT = 2 * PPI; // row tiles per warp

    for (int item = blockIdx.x; item < total; item += gridDim.x) {
        // request of this item: largest r with prefix[r] <= item
        int lo = 0, hi = p.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (item_prefix[mid] <= item)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int r = lo;
        const int b0 = (item - item_prefix[r]) * PPI;
        const int seq_len = p.seq_lens[r];
        const int nb = ceil_div(seq_len + p.nq - 1, kPage);
        const int t0 = r * p.nq;

        // ---- issue every load of the item ----
        // row tile i of this warp: mt = i * 4 + warp; page pg = mt / 8; rows (mt % 8) * 16 + g (+8)
        uint4 raw[MT][2][NVFP4 ? 1 : 4];
        uint32_t sraw[MT][2];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int mt = i * 4 + warp; // warp < 4, so mt >> 3 == i >> 1
            const int pg = i >> 1;
            const int b = b0 + pg;
            int page = 0;
            const bool live = b < nb;
            if (live) {
                page = p.block_table[(size_t)r * p.maxB + b];
                if (page < 0 || page >= p.num_pages) {
                    set_error(p.err, kErrPage);
                    page = 0; // stay in bounds; the call's outputs are void
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = (mt & 7) * 16 + g + 8 * h;
                const size_t grow = (size_t)page * kPage + row;
                if (!NVFP4) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.idxk + grow * (kDim * 2));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        raw[i][h][c] = live ? __ldg(src + c * 4 + q) : make_uint4(0, 0, 0, 0);
                } else {
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.idxk + grow * (kDim / 2));
                    raw[i][h][0] = live ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
                    const uint16_t *s16 =
                        reinterpret_cast<const uint16_t *>(p.scales + grow * (kDim / 16));
                    sraw[i][h] = live ? (uint32_t)__ldg(s16 + q) : 0u;
                }
            }
        }

        float rmax[PPI][NT][2];
#pragma unroll
        for (int pg = 0; pg < PPI; ++pg)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                rmax[pg][nt][0] = rmax[pg][nt][1] = -INFINITY;

#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // B fragments of query tokens nt*8 + g, in this thread's dimension order
            const int j = nt * 8 + g;
            uint32_t bq[8][2];
            const uint16_t *qrow = p.q_idx + (size_t)(t0 + (j < p.nq ? j : 0)) * kDim;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                // bf16: k-step s = 2c + hh covers dims 32c + 8q + 4hh .. +3
                // nvfp4: k-step s covers dims 32q + 4s .. +3
                const int d0 = NVFP4 ? (32 * q + 4 * s) : (32 * (s >> 1) + 8 * q + 4 * (s & 1));
                uint2 v = make_uint2(0, 0);
                if (j < p.nq)
                    v = __ldg(reinterpret_cast<const uint2 *>(qrow + d0));
                if (NVFP4) {
                    bq[s][0] = bf16x2_to_f16x2(v.x);
                    bq[s][1] = bf16x2_to_f16x2(v.y);
                } else {
                    bq[s][0] = v.x;
                    bq[s][1] = v.y;
                }
            }

#pragma unroll
            for (int i = 0; i < MT; ++i) {
                const int mt = i * 4 + warp;
                const int pg = i >> 1;
                const int b = b0 + pg;
                if (b >= nb)
                    continue;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    uint32_t a[4];
                    if (!NVFP4) {
                        const uint4 &r0 = raw[i][0][s >> 1];
                        const uint4 &r1 = raw[i][1][s >> 1];
                        a[0] = (s & 1) ? r0.z : r0.x;
                        a[1] = (s & 1) ? r1.z : r1.x;
                        a[2] = (s & 1) ? r0.w : r0.y;
                        a[3] = (s & 1) ? r1.w : r1.y;
                        mma_bf16(acc, a, bq[s][0], bq[s][1]);
                    } else {
                        // byte 2s -> dims 32q+4s, +1; byte 2s+1 -> dims +2, +3
                        const uint32_t w0 = (&raw[i][0][0].x)[s >> 1];
                        const uint32_t w1 = (&raw[i][1][0].x)[s >> 1];
                        const int sh = (s & 1) * 16;
                        // scale byte: dims 32q..32q+15 -> byte 0, 32q+16.. -> byte 1
                        const int ssh = (s >> 2) * 8;
                        const uint32_t sc0 = (sraw[i][0] >> ssh) & 0xFFu;
                        const uint32_t sc1 = (sraw[i][1] >> ssh) & 0xFFu;
                        const uint32_t f0 = e4m3x2_to_f16x2(sc0 | (sc0 << 8));
                        const uint32_t f1 = e4m3x2_to_f16x2(sc1 | (sc1 << 8));
                        a[0] = hmul2_u32(e2m1x2_to_f16x2((w0 >> sh) & 0xFFu), f0);
                        a[1] = hmul2_u32(e2m1x2_to_f16x2((w1 >> sh) & 0xFFu), f1);
                        a[2] = hmul2_u32(e2m1x2_to_f16x2((w0 >> (sh + 8)) & 0xFFu), f0);
                        a[3] = hmul2_u32(e2m1x2_to_f16x2((w1 >> (sh + 8)) & 0xFFu), f1);
                        mma_f16(acc, a, bq[s][0], bq[s][1]);
                    }
                }
                // acc: (row g, cols 2q, 2q+1), (row g+8, cols 2q, 2q+1); col = query token
                const int pos_g = b * kPage + (mt & 7) * 16 + g;
                const bool need_mask = (b + 1) * kPage > seq_len;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int jj = nt * 8 + 2 * q + c;
                    float v0 = acc[c], v1 = acc[2 + c];
                    if (need_mask) {
                        const int L = seq_len + jj;
                        if (pos_g >= L)
                            v0 = -INFINITY;
                        if (pos_g + 8 >= L)
                            v1 = -INFINITY;
                    }
                    rmax[pg][nt][c] = fmaxf(rmax[pg][nt][c], fmaxf(v0, v1));
                }
            }
        }

        // ---- reduce over the warp's rows, then over the 4 warps ----
#pragma unroll
        for (int pg = 0; pg < PPI; ++pg)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float v = rmax[pg][nt][c];
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                    if (g == 0)
                        red[warp][pg][nt * 8 + 2 * q + c] = v;
                }
        __syncthreads();
        for (int e = threadIdx.x; e < PPI * p.nq; e += kScoreThreads) {
            const int pg = e / p.nq, jj = e - pg * p.nq;
            const int b = b0 + pg;
            if (b < nb) {
                const float v = fmaxf(fmaxf(red[0][pg][jj], red[1][pg][jj]),
                                      fmaxf(red[2][pg][jj], red[3][pg][jj]));
                p.block_scores[(size_t)(t0 + jj) * p.maxB + b] = v;
            }
        }
        __syncthreads();
    }
}

template <bool NVFP4, int NT, int PPI>
cudaError_t launch_t(const ScoreParams &p, int num_sms, cudaStream_t stream)
{
    auto kern = index_score_kernel<NVFP4, NT, PPI>;
    const size_t smem = sizeof(int) * (size_t)(p.R + 1);
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kScoreThreads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        per_sm = 1;
    // upper bound on items: every request at max_blocks
    const long long max_items = (long long)p.R * ((p.maxB + PPI - 1) / PPI);
    long long grid = (long long)num_sms * per_sm;
    if (grid > max_items)
        grid = max_items;
    if (grid < 1)
        grid = 1;
    kern<<<(unsigned)grid, kScoreThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_index_score(const ScoreParams &p, int index_dtype, int num_sms,
                               cudaStream_t stream)
{
    const int nt = (p.nq + 7) / 8;
    if (index_dtype == MSA_NVFP4) {
        switch (nt) {
        case 1: return launch_t<true, 1, 4>(p, num_sms, stream);
        case 2: return launch_t<true, 2, 2>(p, num_sms, stream);
        case 3:
        case 4: return launch_t<true, 4, 1>(p, num_sms, stream);
        case 5:
        case 6: return launch_t<true, 6, 1>(p, num_sms, stream);
        default: return launch_t<true, 8, 1>(p, num_sms, stream);
        }
    }
    switch (nt) {
    case 1: return launch_t<false, 1, 1>(p, num_sms, stream);
    case 2: return launch_t<false, 2, 1>(p, num_sms, stream);
    case 3:
    case 4: return launch_t<false, 4, 1>(p, num_sms, stream);
    case 5:
    case 6: return launch_t<false, 6, 1>(p, num_sms, stream);
    default: return launch_t<false, 8, 1>(p, num_sms, stream);
    }
}

} // namespace msa
