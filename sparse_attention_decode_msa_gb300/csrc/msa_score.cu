// msa_score.cu -- stage (a): index scores and the per-block max.
//
// "MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2 for
// Blackwell", section "The TP4 decode target": an index scorer streams the
// index-K pages; the prefill-select commit of "Add Rubin (sm_107) MiniMax-M3.1
// low-latency decode targets" keeps one max score per 128-token block.  Here
// the per-token scores never reach memory: each page is scored and reduced to
// its block max in registers.
//
// The dot products run on the tensor cores with the page's 16-token row tiles
// (or the whole 128-token page) as M and the request's query tokens as N.
// Inputs are integer-valued (bf16) or NVFP4 with power-of-two scales, so every
// product and partial sum is exact in fp32 and the result equals the plain
// dot product bit for bit, whatever the summation order.
//
// Four scorers, by index-key format and query tokens a request:
//   bf16, <= 8:   TMA page ring, ldmatrix + mma.sync (index_score_ring_kernel)
//   bf16, > 8:    TMA page ring, tcgen05 (index_score_umma_kernel)
//   NVFP4, <= 16: bulk-copy page ring, mma.sync (index_score_fp4_kernel)
//   NVFP4, > 16:  register-staged grid-stride items (index_score_kernel)
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

// Register-staged NVFP4 scorer for many query tokens a request.  NT = n-tiles
// of 8 query tokens; PPI = pages per item.  One item = PPI consecutive pages
// of one request, one CTA of 4 warps per item in a grid-stride loop; each
// warp owns 2 row tiles of every page of the item and issues all of its
// 16-byte loads before the first mma.  Because the K dimension is a pure sum,
// each thread takes its index-key dimensions in the order that makes its
// loads coalesced (32 q + 4 s .. + 3 at k-step s), and the query fragment
// follows the same order.
template <int NT, int PPI>
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
        uint4 raw[MT][2];
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
                const size_t grow = ((size_t)page * p.heads + p.head) * kPage + row;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.idxk + grow * (kDim / 2));
                raw[i][h] = live ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
                const uint16_t *s16 = reinterpret_cast<const uint16_t *>(p.scales + grow * (kDim / 16));
                sraw[i][h] = live ? (uint32_t)__ldg(s16 + q) : 0u;
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
            const uint16_t *qrow = p.q_idx + ((size_t)(t0 + (j < p.nq ? j : 0)) * p.heads + p.head) * kDim;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                // k-step s covers dims 32q + 4s .. +3
                uint2 v = make_uint2(0, 0);
                if (j < p.nq)
                    v = __ldg(reinterpret_cast<const uint2 *>(qrow + 32 * q + 4 * s));
                bq[s][0] = bf16x2_to_f16x2(v.x);
                bq[s][1] = bf16x2_to_f16x2(v.y);
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
                    // byte 2s -> dims 32q+4s, +1; byte 2s+1 -> dims +2, +3
                    const uint32_t w0 = (&raw[i][0].x)[s >> 1];
                    const uint32_t w1 = (&raw[i][1].x)[s >> 1];
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
                p.block_scores[((size_t)(t0 + jj) * p.heads + p.head) * p.maxB + b] = v;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// tcgen05 scorer (bf16 index keys, many query tokens per request).  The pages
// of the call, (request, block) in request-major order, are split into one
// contiguous range per persistent CTA.  Per page: the producer warp brings
// the 128 x 128 index-key tile into a shared-memory ring (TMA, 128-byte
// swizzle); the MMA warp computes S = K_idx Q_idx^T for the request's query
// tokens (M = 128 page tokens, N = q_per_req rounded up to 16) into one of
// kSAcc TMEM accumulators; four epilogue warps read the 128 x N scores (one
// token per TMEM lane), apply the causal limit and reduce each column to its
// maximum (redux.sync.max.f32, then across the four warps).  Integer-valued
// inputs make every product and partial sum exact in fp32, as in the
// mma.sync path.
constexpr int kSTile = kPage * kDim * 2; // bf16 tile
constexpr int kSAcc = 4;                 // TMEM accumulators (pages whose scores are in flight)
constexpr int kSThreads = 32 * 6;        // producer, MMA, 4 epilogue warps
constexpr int kSMaxSmem = 232448;

struct SLayout {
    size_t ring, qbuf, bars, red, prefix, misc, total;
};

__host__ __device__ inline SLayout score_layout(int npad, int stages, int R)
{
    SLayout L{};
    size_t off = 0;
    L.ring = off; // 1024-aligned (swizzle atoms)
    off += (size_t)stages * kSTile;
    L.qbuf = off = align_to(off, 1024); // [2] query tiles of npad rows
    off += 2 * (size_t)npad * kDim * 2;
    // full[S], empty[S], qfull[2], qempty[2], acc_full[kSAcc], acc_empty[kSAcc], esync, done
    L.bars = off = align_to(off, 8);
    off += (size_t)(2 * stages + 4 + 2 * kSAcc + 2) * 8;
    L.red = off = align_to(off, 16); // [2][4][npad] column maxima of the epilogue warps
    off += 2 * 4 * (size_t)npad * 4;
    L.prefix = off = align_to(off, 16); // [R + 1] pages before request r
    off += (size_t)(R + 1) * 4;
    L.misc = off = align_to(off, 16); // TMEM base, abort flag
    off += 16;
    L.total = off + 1024; // slack for aligning the dynamic base
    return L;
}

template <int NPAD>
constexpr uint32_t score_tmem_cols()
{
    return kSAcc * NPAD <= 32 ? 32 : kSAcc * NPAD <= 64 ? 64 : kSAcc * NPAD <= 128 ? 128
           : kSAcc * NPAD <= 256 ? 256 : 512;
}

template <int NPAD, int STAGES>
__global__ void __launch_bounds__(kSThreads, 1)
    index_score_umma_kernel(const __grid_constant__ CUtensorMap k_map,
                            const __grid_constant__ CUtensorMap q_map, const ScoreParams p)
{
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 64, "N of the MMA");
    constexpr int kQTile = NPAD * kDim * 2;
    constexpr uint32_t kCols = score_tmem_cols<NPAD>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SLayout lay = score_layout(NPAD, STAGES, p.R);
    uint8_t *ring = base + lay.ring;
    uint8_t *qbuf = base + lay.qbuf;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + lay.bars);
    uint64_t *empty = full + STAGES;
    uint64_t *qfull = empty + STAGES;
    uint64_t *qempty = qfull + 2;
    uint64_t *acc_full = qempty + 2;        // [kSAcc] scores of a page in TMEM (MMA commit)
    uint64_t *acc_empty = acc_full + kSAcc; // [kSAcc] TMEM accumulator read (4 epilogue warps)
    uint64_t *esync = acc_empty + kSAcc;    // epilogue warps: column maxima written (4 warps)
    uint64_t *done_bar = esync + 1;         // epilogue warps finished with TMEM (4 warps)
    float *red = reinterpret_cast<float *>(base + lay.red);
    int *prefix = reinterpret_cast<int *>(base + lay.prefix);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + lay.misc);
    volatile int *abort_flag = reinterpret_cast<int *>(base + lay.misc) + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    launch_dependents(); // the select may start its prologue while pages are scored

    if (threadIdx.x == 0) {
        prefetch_tensormap(&k_map);
        prefetch_tensormap(&q_map);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&qfull[b]), 1);
            mbar_init(smem_u32(&qempty[b]), 1);
        }
        for (int b = 0; b < kSAcc; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);
        }
        mbar_init(smem_u32(esync), 4);
        mbar_init(smem_u32(done_bar), 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(smem_u32(tmem_slot), kCols);
    build_item_prefix<1>(p, prefix); // ends with __syncthreads
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int P = prefix[p.R];
    const int x_begin = (int)((long long)blockIdx.x * P / gridDim.x);
    const int n = (int)((long long)(blockIdx.x + 1) * P / gridDim.x) - x_begin;

    // (request, block) of page x: the largest r with prefix[r] <= x has pages
    auto request_of = [&](int x) {
        int lo = 0, hi = p.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };
    int cur_r = 0, cur_b = 0; // cursor of each role over its pages
    if (n > 0) {
        cur_r = request_of(x_begin);
        cur_b = x_begin - prefix[cur_r];
    }
    auto advance = [&](int &r, int &b) {
        if (++b >= prefix[r + 1] - prefix[r]) {
            b = 0;
            do
                ++r;
            while (r < p.R && prefix[r + 1] == prefix[r]);
        }
    };

    if (warp == 0) {
        // =================== producer ===================
        const uint64_t k_policy = l2_evict_first_policy(); // index-key pages are streamed
        bool ok = true;
        int units = 0, last_r = -1, issued = 0, q_issued = 0;
        for (int l0 = 0; l0 < n && ok; l0 += 32) {
            // page ids of the next 32 pages, one block-table read per lane
            int page = 0, rr = 0;
            if (l0 + lane < n) {
                const int x = x_begin + l0 + lane;
                rr = request_of(x);
                const int bb = x - prefix[rr];
                page = p.block_table[(size_t)rr * p.maxB + bb];
                if (page < 0 || page >= p.num_pages) {
                    set_error(p.err, kErrPage);
                    page = 0; // stay in bounds; the call's outputs are void
                }
            }
            const int cnt = n - l0 < 32 ? n - l0 : 32;
            for (int i = 0; i < cnt; ++i) {
                const int l = l0 + i;
                const int pg = __shfl_sync(0xffffffffu, page, i);
                const int ri = __shfl_sync(0xffffffffu, rr, i);
                if (lane == 0) {
                    const int slot = l % STAGES;
                    if (l >= STAGES)
                        ok = mbar_wait_or_abort(smem_u32(&empty[slot]), ((l / STAGES) - 1) & 1, abort_flag);
                    if (ok && ri != last_r) {
                        last_r = ri;
                        const int qb = units & 1;
                        if (units >= 2)
                            ok = mbar_wait_or_abort(smem_u32(&qempty[qb]), ((units >> 1) - 1) & 1, abort_flag);
                        if (ok) {
                            const uint32_t qbar = smem_u32(&qfull[qb]);
                            const uint32_t dst = smem_u32(qbuf + qb * kQTile);
                            mbar_arrive_expect_tx(qbar, kQTile);
                            tma_load_2d(dst, &q_map, 0, ri * p.nq, qbar);
                            tma_load_2d(dst + kQTile / 2, &q_map, 64, ri * p.nq, qbar);
                            q_issued = units + 1;
                        }
                        ++units;
                    }
                    if (ok) {
                        const uint32_t bar = smem_u32(&full[slot]);
                        const uint32_t dst = smem_u32(ring + (size_t)slot * kSTile);
                        mbar_arrive_expect_tx(bar, kSTile);
                        const int krow = (pg * p.heads + p.head) * kPage;
                        tma_load_2d_hint(dst, &k_map, 0, krow, bar, k_policy);
                        tma_load_2d_hint(dst + kSTile / 2, &k_map, 64, krow, bar, k_policy);
                        issued = l + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
            }
        }
        if (!ok && lane == 0) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            // let the copies in flight land before the CTA's shared memory goes away
            for (int z = issued - STAGES < 0 ? 0 : issued - STAGES; z < issued; ++z)
                (void)mbar_wait_bounded(smem_u32(&full[z % STAGES]), (z / STAGES) & 1);
            for (int u = q_issued - 2 < 0 ? 0 : q_issued - 2; u < q_issued; ++u)
                (void)mbar_wait_bounded(smem_u32(&qfull[u & 1]), (u >> 1) & 1);
        }
        return;
    }

    if (warp == 1) {
        // =================== MMA issuer (lane 0) ===================
        constexpr uint32_t kIdesc = umma_idesc_bf16(128, NPAD, 0, 0); // both K-major
        if (lane == 0 && n > 0) {
            bool ok = true;
            int units = 0, mma_r = -1, r = cur_r, b = cur_b;
            for (int l = 0; l < n && ok; ++l) {
                const int slot = l % STAGES, ab = l % kSAcc;
                ok = mbar_wait_or_abort(smem_u32(&full[slot]), (l / STAGES) & 1, abort_flag);
                if (ok && r != mma_r) {
                    ok = mbar_wait_or_abort(smem_u32(&qfull[units & 1]), (units >> 1) & 1, abort_flag);
                    mma_r = r;
                    ++units;
                }
                if (ok && l >= kSAcc)
                    ok = mbar_wait_or_abort(smem_u32(&acc_empty[ab]), ((l / kSAcc) - 1) & 1, abort_flag);
                if (!ok)
                    break;
                tcgen05_after_sync();
                const int qb = (units - 1) & 1;
                const uint32_t tile = smem_u32(ring + (size_t)slot * kSTile);
                const uint32_t qtile = smem_u32(qbuf + qb * kQTile);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = umma_desc_sw128(tile + (ks >> 2) * (kSTile / 2) + (ks & 3) * 32, 16, 1024);
                    const uint64_t bq = umma_desc_sw128(qtile + (ks >> 2) * (kQTile / 2) + (ks & 3) * 32, 16, 1024);
                    umma_bf16(tmem + ab * NPAD, a, bq, kIdesc, ks > 0);
                }
                umma_commit(smem_u32(&acc_full[ab]));
                umma_commit(smem_u32(&empty[slot])); // tile read
                const int r_prev = r;
                advance(r, b);
                if (l + 1 == n || r != r_prev)
                    umma_commit(smem_u32(&qempty[qb])); // last page of the request here
            }
            if (!ok) {
                set_error(p.err, kErrTimeout);
                *abort_flag = 1;
            }
        }
        __syncwarp();
        // free TMEM once the epilogue warps are done with it (they always
        // arrive, also after an abort; the wait is bounded)
        if (lane == 0)
            (void)mbar_wait_bounded(smem_u32(done_bar), 0);
        __syncwarp();
        tcgen05_after_sync();
        tmem_dealloc(tmem, kCols);
        return;
    }

    // =================== epilogue warps 2..5 ===================
    const int quarter = warp & 3;   // TMEM lanes 32 * quarter ..: page tokens
    const int e = threadIdx.x - 64; // 0..127
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16);
    bool ok = true;
    int r = cur_r, b = cur_b, seq_r = -1, seq_len = 0;
    for (int l = 0; l < n && ok; ++l) {
        const int ab = l % kSAcc, rb2 = l & 1; // accumulator, red buffer
        ok = mbar_wait_or_abort(smem_u32(&acc_full[ab]), (l / kSAcc) & 1, abort_flag);
        if (!ok)
            break;
        tcgen05_after_sync();
        float v[NPAD];
#pragma unroll
        for (int c16 = 0; c16 < NPAD / 16; ++c16)
            tmem_ld16(lane_base + ab * NPAD + 16 * c16, *reinterpret_cast<float(*)[16]>(v + 16 * c16));
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&acc_empty[ab]));
        if (r != seq_r) {
            seq_r = r;
            seq_len = p.seq_lens[r];
        }
        // token j of the request sees positions < seq_len + j
        const int lim = seq_len - (b * kPage + 32 * quarter + lane); // visible iff j + lim > 0
        float *rw = red + (rb2 * 4 + quarter) * NPAD;
        float mine = -INFINITY; // maximum of column j, kept by lane j % 32
#pragma unroll
        for (int j = 0; j < NPAD; ++j) {
            if (j < p.nq) {
                const float m = warp_max_f32(j + lim > 0 ? v[j] : -INFINITY);
                if (lane == (j & 31))
                    mine = m;
            }
            if ((j & 31) == 31 || j == NPAD - 1) {
                if (lane + (j & ~31) < p.nq && lane <= (j & 31))
                    rw[lane + (j & ~31)] = mine;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(esync));
        if (!mbar_wait_or_abort(smem_u32(esync), l & 1, abort_flag)) {
            ok = false;
            break;
        }
        if (e < p.nq) {
            const float *rb = red + rb2 * 4 * NPAD;
            const float m = fmaxf(fmaxf(rb[e], rb[NPAD + e]), fmaxf(rb[2 * NPAD + e], rb[3 * NPAD + e]));
            p.block_scores[((size_t)(r * p.nq + e) * p.heads + p.head) * p.maxB + b] = m;
        }
        advance(r, b);
    }
    if (!ok) {
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
    }
    tcgen05_before_sync();
    __syncwarp();
    if (lane == 0)
        mbar_arrive(smem_u32(done_bar));
}

template <int NPAD, int STAGES>
cudaError_t launch_umma_t(const ScoreParams &p, const CUtensorMap &kmap, const CUtensorMap &qmap,
                          int num_sms, cudaStream_t stream)
{
    auto kern = index_score_umma_kernel<NPAD, STAGES>;
    const size_t smem = score_layout(NPAD, STAGES, p.R).total;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    long long grid = num_sms;
    const long long max_pages = (long long)p.R * p.maxB;
    if (grid > max_pages)
        grid = max_pages;
    if (grid < 1)
        grid = 1;
    kern<<<(unsigned)grid, kSThreads, smem, stream>>>(kmap, qmap, p);
    return cudaGetLastError();
}

// The deepest ring that fits next to the request prefix (R + 1 ints).
template <int NPAD>
cudaError_t launch_umma_fit(const ScoreParams &p, const CUtensorMap &kmap, const CUtensorMap &qmap,
                            int num_sms, cudaStream_t stream)
{
    if (score_layout(NPAD, 5, p.R).total <= (size_t)kSMaxSmem)
        return launch_umma_t<NPAD, 5>(p, kmap, qmap, num_sms, stream);
    if (score_layout(NPAD, 3, p.R).total > (size_t)kSMaxSmem)
        return cudaErrorInvalidConfiguration; // not reached within the shape limits
    return launch_umma_t<NPAD, 3>(p, kmap, qmap, num_sms, stream);
}

// ---------------------------------------------------------------------------
// NVFP4 scorer with a bulk-copy page ring (up to 16 query tokens a request).
// One persistent CTA per SM takes a contiguous range of the call's pages
// (request-major).  Two producer warps stream the pages' packed E2M1 codes
// (8 KiB) and E4M3 scales (1 KiB) into a ring of shared-memory stages with
// two 1-D bulk copies each, warp w the pages w, w + 2, ... (one warp alone
// issues bulk copies of this size at about one per 340 ns, 4 TB/s over the
// GPU; two reach the HBM rate); consumer warp c scores pages c, c + 12, ... of
// the range on its own:
// 16-byte loads of 32 codes per row and thread, widened in registers
// (cvt.rn.f16x2.e2m1x2 times the power-of-two f16 scale: exact), mma.sync
// m16n8k16 against the request's query tokens kept as f16 fragments in
// registers, causal mask, maximum over the page's 128 rows in registers and
// shuffles, one write per (query token, block).  No global load waits in the
// consumers' path and no cross-warp reduction.
constexpr int kF4Producers = 2;
constexpr int kF4Consumers = 12;
constexpr int kF4Threads = 32 * (kF4Producers + kF4Consumers);
constexpr int kF4Codes = kPage * kDim / 2;      // 8 KiB
constexpr int kF4Scales = kPage * kDim / 16;    // 1 KiB
constexpr int kF4Stage = kF4Codes + kF4Scales;  // 9 KiB
// ring depths: 24 stages, or 12 when the request prefix of a call with many
// requests leaves no room for 24
constexpr int kF4StagesDeep = 24, kF4StagesShallow = 12;
// a slot's successive pages belong to one producer warp and one consumer warp
static_assert(kF4StagesDeep % kF4Producers == 0 && kF4StagesDeep % kF4Consumers == 0 &&
                  kF4StagesShallow % kF4Producers == 0 && kF4StagesShallow % kF4Consumers == 0,
              "ring / warp split");

__host__ __device__ constexpr size_t fp4_smem_bytes(int R, int stages)
{
    // ring, full[S], empty[S], abort flag, request prefix [R + 1]
    return align_to((size_t)stages * kF4Stage, 16) + 2 * (size_t)stages * 8 + 16 + (size_t)(R + 1) * 4 + 128;
}

template <int NT, int kF4Stages>
__global__ void __launch_bounds__(kF4Threads, 1) index_score_fp4_kernel(const ScoreParams p)
{
    extern __shared__ __align__(128) uint8_t smem_f4[];
    uint8_t *ring = smem_f4;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_f4 + align_to((size_t)kF4Stages * kF4Stage, 16));
    uint64_t *empty = full + kF4Stages;
    volatile int *abort_flag = reinterpret_cast<int *>(empty + kF4Stages);
    int *prefix = reinterpret_cast<int *>(empty + kF4Stages) + 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    launch_dependents(); // the select may start its prologue while pages are scored
    if (threadIdx.x == 0) {
        for (int s = 0; s < kF4Stages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    build_item_prefix<1>(p, prefix); // ends with __syncthreads

    const int P = prefix[p.R];
    const int x_begin = (int)((long long)blockIdx.x * P / gridDim.x);
    const int n = (int)((long long)(blockIdx.x + 1) * P / gridDim.x) - x_begin;
    auto request_of = [&](int x) { // largest r with prefix[r] <= x (a request with pages)
        int lo = 0, hi = p.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };

    if (warp < kF4Producers) {
        // =================== producers: pages warp, warp + kF4Producers, ... ===================
        const uint64_t k_policy = l2_evict_first_policy(); // index-key pages are streamed
        bool ok = true;
        int issued = 0; // one past this warp's last issued page
        for (int l0 = warp; l0 < n && ok; l0 += 32 * kF4Producers) {
            int page = 0;
            if (l0 + kF4Producers * lane < n) {
                const int x = x_begin + l0 + kF4Producers * lane;
                const int rr = request_of(x);
                page = p.block_table[(size_t)rr * p.maxB + (x - prefix[rr])];
                if (page < 0 || page >= p.num_pages) {
                    set_error(p.err, kErrPage);
                    page = 0; // stay in bounds; the call's outputs are void
                }
            }
            const int left = (n - l0 + kF4Producers - 1) / kF4Producers; // this warp's pages from l0 on
            const int cnt = left < 32 ? left : 32;
            for (int i = 0; i < cnt; ++i) {
                const int l = l0 + kF4Producers * i;
                const int pg = __shfl_sync(0xffffffffu, page, i);
                if (lane == 0) {
                    const int slot = l % kF4Stages;
                    if (l >= kF4Stages)
                        ok = mbar_wait_or_abort(smem_u32(&empty[slot]), ((l / kF4Stages) - 1) & 1, abort_flag);
                    if (ok) {
                        const uint32_t bar = smem_u32(&full[slot]);
                        const uint32_t dst = smem_u32(ring + (size_t)slot * kF4Stage);
                        mbar_arrive_expect_tx(bar, kF4Stage);
                        const size_t prow = (size_t)pg * p.heads + p.head;
                        bulk_load_hint(dst, p.idxk + prow * kF4Codes, kF4Codes, bar, k_policy);
                        bulk_load_hint(dst + kF4Codes, p.scales + prow * kF4Scales, kF4Scales, bar, k_policy);
                        issued = l + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
            }
        }
        if (!ok && lane == 0) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            // this warp's copies that may still be in flight: its pages among
            // the last kF4Stages before its next one (older ones were consumed)
            for (int z = issued - kF4Stages < 0 ? 0 : issued - kF4Stages; z < issued; ++z)
                if (z % kF4Producers == warp)
                    (void)mbar_wait_bounded(smem_u32(&full[z % kF4Stages]), (z / kF4Stages) & 1);
        }
        return;
    }

    // =================== consumer warps ===================
    const int cw = warp - kF4Producers;
    const int g = lane >> 2, q = lane & 3;
    uint32_t bq[NT][8][2]; // query fragments of the current request, f16
    int frag_r = -1, seq_len = 0;
    bool ok = true;
    for (int l = cw; l < n && ok; l += kF4Consumers) {
        const int slot = l % kF4Stages;
        const int x = x_begin + l;
        const int r = request_of(x), b = x - prefix[r];
        if (r != frag_r) {
            frag_r = r;
            seq_len = p.seq_lens[r];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int j = nt * 8 + g;
                const uint16_t *qrow = p.q_idx + ((size_t)(r * p.nq + (j < p.nq ? j : 0)) * p.heads + p.head) * kDim;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    // k-step s covers dims 32 q + 4 s .. + 3 (the codes' order below)
                    uint2 v = make_uint2(0, 0);
                    if (j < p.nq)
                        v = __ldg(reinterpret_cast<const uint2 *>(qrow + 32 * q + 4 * s));
                    bq[nt][s][0] = bf16x2_to_f16x2(v.x);
                    bq[nt][s][1] = bf16x2_to_f16x2(v.y);
                }
            }
        }
        if (!mbar_wait_or_abort(smem_u32(&full[slot]), (l / kF4Stages) & 1, abort_flag)) {
            ok = false;
            break;
        }
        const uint8_t *codes = ring + (size_t)slot * kF4Stage;
        const uint8_t *scl = codes + kF4Codes;
        float rmax[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            rmax[nt][0] = rmax[nt][1] = -INFINITY;
        const bool need_mask = (b + 1) * kPage > seq_len;
#pragma unroll 2
        for (int mt = 0; mt < kPage / 16; ++mt) {
            const int row0 = 16 * mt + g;
            const uint4 c0 = *reinterpret_cast<const uint4 *>(codes + row0 * 64 + 16 * q);
            const uint4 c1 = *reinterpret_cast<const uint4 *>(codes + (row0 + 8) * 64 + 16 * q);
            const uint32_t s0 = *reinterpret_cast<const uint16_t *>(scl + row0 * 8 + 2 * q);
            const uint32_t s1 = *reinterpret_cast<const uint16_t *>(scl + (row0 + 8) * 8 + 2 * q);
            // the two scales of each row (dims 32q .. +15 and +16 .. +31), as f16 pairs
            const uint32_t f0[2] = {e4m3x2_to_f16x2((s0 & 0xFFu) * 0x101u), e4m3x2_to_f16x2((s0 >> 8) * 0x101u)};
            const uint32_t f1[2] = {e4m3x2_to_f16x2((s1 & 0xFFu) * 0x101u), e4m3x2_to_f16x2((s1 >> 8) * 0x101u)};
            uint32_t a[8][4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // word w of the 16 bytes: k-steps 2w (bytes 0, 1) and 2w + 1 (bytes 2, 3),
                // dims 32q + 8w .. + 7; scale byte w / 2
                uint32_t r0[4], r1[4];
                e2m1x8_scaled_f16x2((&c0.x)[w], f0[w >> 1], r0);
                e2m1x8_scaled_f16x2((&c1.x)[w], f1[w >> 1], r1);
                a[2 * w][0] = r0[0];
                a[2 * w][2] = r0[1];
                a[2 * w + 1][0] = r0[2];
                a[2 * w + 1][2] = r0[3];
                a[2 * w][1] = r1[0];
                a[2 * w][3] = r1[1];
                a[2 * w + 1][1] = r1[2];
                a[2 * w + 1][3] = r1[3];
            }
            const int pos_g = b * kPage + row0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // two accumulators (even and odd k-steps) halve the dependent
                // chain; the scores are exact in fp32 in any order
                float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int s = 0; s < 8; s += 2) {
                    mma_f16(acc, a[s], bq[nt][s][0], bq[nt][s][1]);
                    mma_f16(acc2, a[s + 1], bq[nt][s + 1][0], bq[nt][s + 1][1]);
                }
                // acc: (row g, cols 2q, 2q+1), (row g + 8, cols 2q, 2q+1); col = query token
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float v0 = acc[c] + acc2[c], v1 = acc[2 + c] + acc2[2 + c];
                    if (need_mask) {
                        const int L = seq_len + nt * 8 + 2 * q + c;
                        if (pos_g >= L)
                            v0 = -INFINITY;
                        if (pos_g + 8 >= L)
                            v1 = -INFINITY;
                    }
                    rmax[nt][c] = fmaxf(rmax[nt][c], fmaxf(v0, v1));
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty[slot])); // the page's codes are in registers
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v = rmax[nt][c];
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                const int jj = nt * 8 + 2 * q + c;
                if (g == 0 && jj < p.nq)
                    p.block_scores[((size_t)(r * p.nq + jj) * p.heads + p.head) * p.maxB + b] = v;
            }
    }
    if (!ok) {
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
    }
}

template <int NT, int STAGES>
cudaError_t launch_fp4_t(const ScoreParams &p, int num_sms, cudaStream_t stream)
{
    const size_t smem = fp4_smem_bytes(p.R, STAGES);
    cudaError_t e = cudaFuncSetAttribute(index_score_fp4_kernel<NT, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    long long grid = num_sms;
    const long long max_pages = (long long)p.R * p.maxB;
    if (grid > max_pages)
        grid = max_pages;
    if (grid < 1)
        grid = 1;
    index_score_fp4_kernel<NT, STAGES><<<(unsigned)grid, kF4Threads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int NT>
cudaError_t launch_fp4_fit(const ScoreParams &p, int num_sms, cudaStream_t stream)
{
    if (fp4_smem_bytes(p.R, kF4StagesDeep) <= (size_t)kSMaxSmem)
        return launch_fp4_t<NT, kF4StagesDeep>(p, num_sms, stream);
    return launch_fp4_t<NT, kF4StagesShallow>(p, num_sms, stream);
}

// ---------------------------------------------------------------------------
// bf16 scorer with a TMA page ring (up to 8 query tokens a request).  One
// persistent CTA per SM takes a contiguous range of the call's pages
// (request-major).  Two producer warps bring each page's 128 x 128 index-key
// tile into a 6-stage ring (two 16 KiB TMA boxes, 128-byte swizzle), warp w
// the pages w, w + 2, ...; consumer warp c scores pages c, c + 6, ... on its
// own: ldmatrix of the swizzled rows (conflict-free), mma.sync m16n8k16
// against the request's query tokens kept in registers, causal mask, maximum
// over the page's 128 rows in registers and shuffles, one write per (query
// token, block).  With a few pages per SM (a short decode step), nearly a
// CTA's whole share of pages is in flight from the start.
constexpr int kRProducers = 2;
constexpr int kRConsumers = 6;
constexpr int kRThreads = 32 * (kRProducers + kRConsumers);
constexpr int kRStages = 6;
constexpr int kRTile = kPage * kDim * 2; // bf16 page tile, 32 KiB
// a slot's successive pages belong to one producer warp and one consumer warp
static_assert(kRStages % kRProducers == 0 && kRStages % kRConsumers == 0, "ring / warp split");

__host__ __device__ constexpr size_t ring_smem_bytes(int R)
{
    // alignment slack (swizzle atoms: 1024 B), ring, full[S], empty[S],
    // abort flag, request prefix [R + 1]
    return 1024 + (size_t)kRStages * kRTile + 2 * kRStages * 8 + 16 + (size_t)(R + 1) * 4 + 16;
}

__global__ void __launch_bounds__(kRThreads, 1)
    index_score_ring_kernel(const __grid_constant__ CUtensorMap k_map, const ScoreParams p)
{
    extern __shared__ uint8_t smem_rg[];
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_rg) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + (size_t)kRStages * kRTile);
    uint64_t *empty = full + kRStages;
    volatile int *abort_flag = reinterpret_cast<int *>(empty + kRStages);
    int *prefix = reinterpret_cast<int *>(empty + kRStages) + 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    launch_dependents(); // the select may start its prologue while pages are scored
    if (threadIdx.x == 0) {
        prefetch_tensormap(&k_map);
        for (int s = 0; s < kRStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    build_item_prefix<1>(p, prefix); // ends with __syncthreads

    const int P = prefix[p.R];
    const int x_begin = (int)((long long)blockIdx.x * P / gridDim.x);
    const int n = (int)((long long)(blockIdx.x + 1) * P / gridDim.x) - x_begin;
    auto request_of = [&](int x) { // largest r with prefix[r] <= x (a request with pages)
        int lo = 0, hi = p.R - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= x)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    };

    if (warp < kRProducers) {
        // =================== producers: pages warp, warp + kRProducers, ... ===================
        const uint64_t k_policy = l2_evict_first_policy(); // index-key pages are streamed
        bool ok = true;
        int issued = 0; // one past this warp's last issued page
        for (int l0 = warp; l0 < n && ok; l0 += 32 * kRProducers) {
            int page = 0;
            if (l0 + kRProducers * lane < n) {
                const int x = x_begin + l0 + kRProducers * lane;
                const int rr = request_of(x);
                page = p.block_table[(size_t)rr * p.maxB + (x - prefix[rr])];
                if (page < 0 || page >= p.num_pages) {
                    set_error(p.err, kErrPage);
                    page = 0; // stay in bounds; the call's outputs are void
                }
            }
            const int left = (n - l0 + kRProducers - 1) / kRProducers; // this warp's pages from l0 on
            const int cnt = left < 32 ? left : 32;
            for (int i = 0; i < cnt; ++i) {
                const int l = l0 + kRProducers * i;
                const int pg = __shfl_sync(0xffffffffu, page, i);
                if (lane == 0) {
                    const int slot = l % kRStages;
                    if (l >= kRStages)
                        ok = mbar_wait_or_abort(smem_u32(&empty[slot]), ((l / kRStages) - 1) & 1, abort_flag);
                    if (ok) {
                        const uint32_t bar = smem_u32(&full[slot]);
                        const uint32_t dst = smem_u32(ring + (size_t)slot * kRTile);
                        mbar_arrive_expect_tx(bar, kRTile);
                        const int krow = (pg * p.heads + p.head) * kPage;
                        tma_load_2d_hint(dst, &k_map, 0, krow, bar, k_policy);
                        tma_load_2d_hint(dst + kRTile / 2, &k_map, 64, krow, bar, k_policy);
                        issued = l + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
            }
        }
        if (!ok && lane == 0) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            // this warp's copies that may still be in flight: its pages among
            // the last kRStages before its next one (older ones were consumed)
            for (int z = issued - kRStages < 0 ? 0 : issued - kRStages; z < issued; ++z)
                if (z % kRProducers == warp)
                    (void)mbar_wait_bounded(smem_u32(&full[z % kRStages]), (z / kRStages) & 1);
        }
        return;
    }

    // =================== consumer warps ===================
    const int cw = warp - kRProducers;
    const int g = lane >> 2, q = lane & 3;
    // ldmatrix.x4 of a 16 x 16 A tile: lanes 8i .. 8i + 7 give the rows of
    // matrix i = (rows +0 / +8 for i even / odd, dims +0 / +8 for i < 2 / >= 2)
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int lchunk = lane >> 4;
    uint32_t bq[8][2]; // query fragments of the current request: k-step s, dims 16 s + 2 q (+8)
    int frag_r = -1, seq_len = 0;
    bool ok = true;
    for (int l = cw; l < n && ok; l += kRConsumers) {
        const int slot = l % kRStages;
        const int x = x_begin + l;
        const int r = request_of(x), b = x - prefix[r];
        if (r != frag_r) {
            frag_r = r;
            seq_len = p.seq_lens[r];
            const uint16_t *qrow = p.q_idx + ((size_t)(r * p.nq + (g < p.nq ? g : 0)) * p.heads + p.head) * kDim;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                uint32_t v0 = 0, v1 = 0;
                if (g < p.nq) {
                    v0 = __ldg(reinterpret_cast<const uint32_t *>(qrow + 16 * s + 2 * q));
                    v1 = __ldg(reinterpret_cast<const uint32_t *>(qrow + 16 * s + 8 + 2 * q));
                }
                bq[s][0] = v0;
                bq[s][1] = v1;
            }
        }
        if (!mbar_wait_or_abort(smem_u32(&full[slot]), (l / kRStages) & 1, abort_flag)) {
            ok = false;
            break;
        }
        const uint32_t tile = smem_u32(ring + (size_t)slot * kRTile);
        float rmax[2] = {-INFINITY, -INFINITY};
        const bool need_mask = (b + 1) * kPage > seq_len;
#pragma unroll 2
        for (int mt = 0; mt < kPage / 16; ++mt) {
            // rows are 128 B (64 dims) in each half of the tile; 16-byte chunk
            // c of row w sits at chunk c ^ (w % 8)
            const int row = 16 * mt + lrow;
            const uint32_t rbase = tile + row * 128;
            const int sw = row & 7;
            // two accumulators (even and odd k-steps) halve the dependent
            // chain; the scores are exact in fp32 in any order
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < 8; s += 2) {
                uint32_t a0[4], a1[4];
                ldsm_x4(a0, rbase + (s >> 2) * (kRTile / 2) + (((2 * (s & 3) + lchunk) ^ sw) << 4));
                ldsm_x4(a1, rbase + ((s + 1) >> 2) * (kRTile / 2) + (((2 * ((s + 1) & 3) + lchunk) ^ sw) << 4));
                mma_bf16(acc, a0, bq[s][0], bq[s][1]);
                mma_bf16(acc2, a1, bq[s + 1][0], bq[s + 1][1]);
            }
            // acc: (row g, cols 2q, 2q+1), (row g + 8, cols 2q, 2q+1); col = query token
            const int pos_g = b * kPage + 16 * mt + g;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v0 = acc[c] + acc2[c], v1 = acc[2 + c] + acc2[2 + c];
                if (need_mask) {
                    const int L = seq_len + 2 * q + c;
                    if (pos_g >= L)
                        v0 = -INFINITY;
                    if (pos_g + 8 >= L)
                        v1 = -INFINITY;
                }
                rmax[c] = fmaxf(rmax[c], fmaxf(v0, v1));
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty[slot])); // the page's rows are read
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float v = rmax[c];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
            const int jj = 2 * q + c;
            if (g == 0 && jj < p.nq)
                p.block_scores[((size_t)(r * p.nq + jj) * p.heads + p.head) * p.maxB + b] = v;
        }
    }
    if (!ok) {
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
    }
}

cudaError_t launch_ring(const ScoreParams &p, const CUtensorMap &kmap, int num_sms, cudaStream_t stream)
{
    const size_t smem = ring_smem_bytes(p.R);
    cudaError_t e = cudaFuncSetAttribute(index_score_ring_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    long long grid = num_sms;
    const long long max_pages = (long long)p.R * p.maxB;
    if (grid > max_pages)
        grid = max_pages;
    if (grid < 1)
        grid = 1;
    index_score_ring_kernel<<<(unsigned)grid, kRThreads, smem, stream>>>(kmap, p);
    return cudaGetLastError();
}

template <int NT, int PPI>
cudaError_t launch_t(const ScoreParams &p, int num_sms, cudaStream_t stream)
{
    auto kern = index_score_kernel<NT, PPI>;
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
    // The rings leave room for the request prefix of the largest call.
    static_assert(ring_smem_bytes(kMaxRequests) <= (size_t)kSMaxSmem, "bf16 ring and request prefix");
    static_assert(fp4_smem_bytes(kMaxRequests, kF4StagesShallow) <= (size_t)kSMaxSmem,
                  "NVFP4 ring and request prefix");
    if (index_dtype == MSA_BF16) {
        CUtensorMap kmap; // every page row of the index-key pool, 64-dim boxes of 128 rows
        if (!encode_2d_sw128(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.idxk, kDim,
                             (uint64_t)p.num_pages * p.heads * kPage, kDim * 2, 64, kPage))
            return cudaErrorInvalidValue;
        // up to 8 query tokens a request (one n-tile of mma.sync): the
        // TMA-ring mma.sync scorer; more: tcgen05, one MMA per page for all
        if (p.nq <= 8)
            return launch_ring(p, kmap, num_sms, stream);
        const int T = p.R * p.nq;
        const int npad = (p.nq + 15) / 16 * 16;
        CUtensorMap qmap; // this head's query rows: T rows, heads * Di apart
        if (!encode_2d_sw128(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q_idx + (size_t)p.head * kDim, kDim, T,
                             (uint64_t)p.heads * kDim * 2, 64, npad))
            return cudaErrorInvalidValue;
        switch (npad) {
        case 16: return launch_umma_fit<16>(p, kmap, qmap, num_sms, stream);
        case 32: return launch_umma_fit<32>(p, kmap, qmap, num_sms, stream);
        case 48: return launch_umma_fit<48>(p, kmap, qmap, num_sms, stream);
        default: return launch_umma_fit<64>(p, kmap, qmap, num_sms, stream);
        }
    }
    // NVFP4: up to 16 query tokens a request, the bulk-copy ring (the
    // widening of the codes in registers keeps up with HBM there); more, the
    // register-staged scorer with several n-tiles
    const int nt = (p.nq + 7) / 8;
    switch (nt) {
    case 1: return launch_fp4_fit<1>(p, num_sms, stream);
    case 2: return launch_fp4_fit<2>(p, num_sms, stream);
    case 3:
    case 4: return launch_t<4, 1>(p, num_sms, stream);
    case 5:
    case 6: return launch_t<6, 1>(p, num_sms, stream);
    default: return launch_t<8, 1>(p, num_sms, stream);
    }
}

} // namespace msa
