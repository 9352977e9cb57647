// msa_select.cu -- stage (b): top-k block selection.
//
// Contract ("MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2
// for Blackwell", section "The TP4 decode target"): the k blocks with the
// largest block score, score ties broken toward the smaller block index, for
// any tie width.  Output ("Add Rubin (sm_107) MiniMax-M3.1 low-latency decode
// targets", q8kv4 indexer commit): ascending block ids, -1 padded to k.
//
// With several index heads a row is (token, KV head) and its score per block
// is the maximum over the KV head's group of index heads (the maximum of the
// order-preserving keys).  Forced blocks (the first `init` and the last
// `local` visible blocks) take the largest key, above every score, so they
// are always kept and the remaining places go to the best scores.
//
// Scores map to order-preserving 32-bit keys.  Rows of up to 2048 blocks take
// one warp per token (below); longer rows one CTA per token, where an
// MSB-first radix select (four 8-bit digits) finds the k-th largest key theta
// and how many of the blocks equal to theta are still needed.  A block is selected if
// its key is above theta, or equal to theta and among the first `need` such
// blocks in index order.  Two CTA-wide exclusive scans over blocks in index
// order give each tie its rank and each selected block its output slot, so
// the table comes out ascending with no sort.  Comparisons only: bit-exact.
#include "msa_internal.cuh"
#include "msa_select_warp.cuh"

namespace msa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;

// CTA-wide exclusive scan of one int per thread; returns the prefix and
// writes the total to *total.  Uses `tmp` (kSelWarps + 1 ints).
__device__ int cta_exclusive_scan(int v, int *tmp, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += u;
    }
    if (lane == 31)
        tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < kSelWarps ? tmp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += u;
        }
        if (lane < kSelWarps)
            tmp[lane] = wi - w;
        if (lane == kSelWarps - 1)
            tmp[kSelWarps] = wi;
    }
    __syncthreads();
    const int res = tmp[warp] + incl - v;
    *total = tmp[kSelWarps];
    __syncthreads();
    return res;
}

// Key of block b of row (t, gs): forced -> the largest key, else the largest
// key over the group's index heads.
__device__ __forceinline__ uint32_t row_key(const SelectParams &p, const float *row, int b, int n)
{
    if (b < p.init || b >= n - p.local)
        return 0xFFFFFFFFu;
    uint32_t k = order_key(row[b]);
    for (int i = 1; i < p.r; ++i) {
        const uint32_t v = order_key(row[(size_t)i * p.maxB + b]);
        k = v > k ? v : k;
    }
    return k;
}

__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(const SelectParams p)
{
    extern __shared__ uint32_t keys[]; // [maxB]
    __shared__ int hist[256];
    __shared__ int scan_tmp[kSelWarps + 1];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;

    launch_dependents(); // the decode may start its prologue while tokens are selected
    const int x = blockIdx.x; // row: token t, selection head gs
    const int t = x / p.Hs, gs = x - t * p.Hs;
    const int r = t / p.nq, j = t - r * p.nq;
    int32_t *out = p.selected + (size_t)x * p.k;
    const int seq_len = p.seq_lens[r];
    const long long nb_req = ((long long)seq_len + p.nq - 1 + kPage - 1) / kPage;
    if (seq_len < 1 || nb_req > p.maxB) {
        if (threadIdx.x == 0)
            set_error(p.err, kErrSeqLen);
        for (int i = threadIdx.x; i < p.k; i += kSelThreads)
            out[i] = -1;
        return;
    }
    const int n = ceil_div(seq_len + j, kPage); // blocks with a visible position
    if (n <= p.k) {
        for (int i = threadIdx.x; i < p.k; i += kSelThreads)
            out[i] = i < n ? i : -1;
        return;
    }

    // block_scores come from the previous kernel of the step
    grid_dependency_wait();
    const float *row = p.block_scores + ((size_t)t * p.Hi + (size_t)gs * p.r) * p.maxB;
    for (int b = threadIdx.x; b < n; b += kSelThreads)
        keys[b] = row_key(p, row, b, n);
    if (threadIdx.x == 0) {
        s_prefix = 0u;
        s_need = p.k;
    }
    __syncthreads();

    // ---- radix select of the k-th largest key ----
    uint32_t pmask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kSelThreads)
            hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int b0 = 0; b0 < n; b0 += kSelThreads) {
            const int b = b0 + threadIdx.x;
            const bool cand = b < n && (keys[b] & pmask) == prefix;
            const uint32_t digit = cand ? (keys[b] >> shift) & 0xFFu : 0xFFFFFFFFu;
            // aggregate equal digits within the warp: one atomic per distinct digit
            const uint32_t peers = __match_any_sync(0xffffffffu, digit);
            const int leader = __ffs(peers) - 1;
            if (cand && (threadIdx.x & 31) == leader)
                atomicAdd(&hist[digit], __popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            const int lane = threadIdx.x;
            int c[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                sum += c[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += u;
            }
            const int above = incl - sum; // keys with a larger digit
            const int need = s_need;
            if (above < need && need <= incl) {
                int acc = above;
                for (int i = 0; i < 8; ++i) {
                    if (acc + c[i] >= need) {
                        s_prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
                        s_need = need - acc;
                        break;
                    }
                    acc += c[i];
                }
            }
        }
        pmask |= 0xFFu << shift;
        __syncthreads();
    }
    const uint32_t theta = s_prefix;
    const int need = s_need; // ties at theta to take, counted in index order

    // ---- ordered compaction: thread i owns blocks [i*chunk, (i+1)*chunk) ----
    const int chunk = ceil_div(n, kSelThreads);
    const int lo = min(n, threadIdx.x * chunk), hi = min(n, lo + chunk);
    int ties = 0;
    for (int b = lo; b < hi; ++b)
        ties += keys[b] == theta;
    int dummy;
    int tie_rank = cta_exclusive_scan(ties, scan_tmp, &dummy);
    int chosen = 0;
    for (int b = lo; b < hi; ++b) {
        const uint32_t kb = keys[b];
        const bool eq = kb == theta;
        chosen += (kb > theta) || (eq && tie_rank < need);
        tie_rank += eq;
    }
    int total;
    int slot = cta_exclusive_scan(chosen, scan_tmp, &total);
    tie_rank -= ties;
    for (int b = lo; b < hi; ++b) {
        const uint32_t kb = keys[b];
        const bool eq = kb == theta;
        if (((kb > theta) || (eq && tie_rank < need)) && slot < p.k)
            out[slot++] = b;
        tie_rank += eq;
    }
    for (int i = total + threadIdx.x; i < p.k; i += kSelThreads)
        out[i] = -1;
}

// ---------------------------------------------------------------------------
// Rows of up to 2048 blocks: one warp per token (msa_select_warp.cuh).
// One warp per CTA: the rows spread over more SMs and a small CTA leaves room
// next to it for the decode CTA that follows in the step (measured 0.5-1 us
// faster fused steps than 4-warp CTAs on every workload).
constexpr int kWarpSelWarps = 1;

template <int S> // key slots per lane: rows of up to 32 * S blocks
__global__ void __launch_bounds__(32 * kWarpSelWarps) select_topk_warp_kernel(const SelectParams p)
{
    launch_dependents();
    const int rows = p.R * p.nq * p.Hs;
    const int x = blockIdx.x * kWarpSelWarps + (threadIdx.x >> 5); // row: token t, selection head gs
    if (x >= rows)
        return;
    warp_select_row<S>(p, x, true);
}

// Rows of 257 to 2048 blocks: four warps per token row, one row per CTA
// (msa_select_warp.cuh, cta_select_row): the threshold search's counts over a
// warp's keys shrink fourfold for one shared-memory sum a step.
constexpr int kCtaSelWarps = 4;

template <int SW, int W> // key slots per lane, warps: rows of up to 32 * W * SW blocks
__global__ void __launch_bounds__(32 * W) select_topk_cta_kernel(const SelectParams p)
{
    launch_dependents();
    __shared__ uint32_t red[2 * 4 * W];
    cta_select_row<SW, W>(p, blockIdx.x, red);
}

// ---- many query rows from a head-major score buffer -------------------------
//
// "Add Rubin (sm_107) MiniMax-M3.1 low-latency decode targets", prefill-select
// commit: context rows take a tile select, one CTA per KV head and 8 queries
// over a [heads, max_k_tiles, tokens] max-score block, each score sector read
// once, with the same table bit for bit as the per-token select (tie order,
// init / local forcing).  Here: block_scores is [Hs][maxB][T] (row index
// innermost), row t = r * nq + j sees ceil((seq_len + j) / 128) blocks.  The
// CTA's threads read the 32-byte sector of block b (8 rows' scores) once,
// transpose the keys into shared memory, and each warp selects its row.
constexpr int kTileRows = 8;

template <int S>
__global__ void __launch_bounds__(32 * kTileRows) select_tile_kernel(const SelectParams p)
{
    extern __shared__ uint32_t tkeys[]; // [kTileRows][32 * S]
    __shared__ int s_n[kTileRows];
    constexpr int W = 32 * S;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int T = p.R * p.nq;
    const int t0 = blockIdx.x * kTileRows, gs = blockIdx.y;
    if (threadIdx.x < kTileRows) {
        const int t = t0 + threadIdx.x;
        int n = 0; // rows past T: none
        if (t < T) {
            const int r = t / p.nq, j = t - r * p.nq;
            const int seq_len = p.seq_lens[r];
            const long long nb_req = ((long long)seq_len + p.nq - 1 + kPage - 1) / kPage;
            n = (seq_len < 1 || nb_req > p.maxB) ? -1 : ceil_div(seq_len + j, kPage);
        }
        s_n[threadIdx.x] = n;
    }
    __syncthreads();
    int n_max = 0;
#pragma unroll
    for (int i = 0; i < kTileRows; ++i)
        n_max = max(n_max, s_n[i]);
    const float *tile = p.block_scores + (size_t)gs * p.maxB * T + t0;
    const bool full = t0 + kTileRows <= T && (T & 3) == 0; // two aligned float4 per sector
    for (int b = threadIdx.x; b < n_max; b += 32 * kTileRows) {
        const float *src = tile + (size_t)b * T;
        float v[kTileRows];
        if (full) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
            const float4 c = __ldg(reinterpret_cast<const float4 *>(src) + 1);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
        } else {
#pragma unroll
            for (int i = 0; i < kTileRows; ++i)
                v[i] = t0 + i < T ? __ldg(src + i) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kTileRows; ++i) {
            const int n = s_n[i];
            uint32_t k = 0u; // past the row's visible blocks: below every candidate
            if (b < n)
                k = (b < p.init || b >= n - p.local) ? 0xFFFFFFFFu : order_key(v[i]);
            tkeys[i * W + b] = k;
        }
    }
    __syncthreads();
    const int t = t0 + w;
    if (t >= T)
        return;
    int32_t *out = p.selected + ((size_t)t * p.Hs + gs) * p.k;
    const int n = s_n[w];
    if (n < 0) {
        if (lane == 0)
            set_error(p.err, kErrSeqLen);
        for (int i = lane; i < p.k; i += 32)
            out[i] = -1;
        return;
    }
    if (n <= p.k) {
        for (int i = lane; i < p.k; i += 32)
            out[i] = i < n ? i : -1;
        return;
    }
    uint32_t key[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int b = lane + 32 * s;
        key[s] = b < n ? tkeys[w * W + b] : 0u;
    }
    warp_select_keys<S>(key, p.k, out);
}

template <int S>
cudaError_t launch_tile_t(const SelectParams &p, cudaStream_t stream)
{
    const size_t smem = sizeof(uint32_t) * kTileRows * 32 * S;
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(select_tile_kernel<S>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int T = p.R * p.nq;
    const dim3 grid((T + kTileRows - 1) / kTileRows, p.Hs), block(32 * kTileRows);
    const cudaError_t e = launch_kernel(select_tile_kernel<S>, grid, block, smem, stream, false, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream, bool pdl)
{
    if (p.maxB <= kWarpSelMaxN) {
        const int rows = p.R * p.nq * p.Hs;
        cudaError_t e;
        if (p.maxB <= 256) {
            const dim3 grid((rows + kWarpSelWarps - 1) / kWarpSelWarps), block(32 * kWarpSelWarps);
            e = launch_kernel(select_topk_warp_kernel<8>, grid, block, 0, stream, pdl, p);
        } else {
            const dim3 grid(rows);
            static_assert(32 * kCtaSelWarps * 16 == kWarpSelMaxN, "CTA select capacity");
            if (p.maxB <= 512)
                e = launch_kernel(select_topk_cta_kernel<4, kCtaSelWarps>, grid, dim3(32 * kCtaSelWarps), 0,
                                  stream, pdl, p);
            else if (p.maxB <= 1024)
                e = launch_kernel(select_topk_cta_kernel<8, kCtaSelWarps>, grid, dim3(32 * kCtaSelWarps), 0,
                                  stream, pdl, p);
            else
                e = launch_kernel(select_topk_cta_kernel<16, kCtaSelWarps>, grid, dim3(32 * kCtaSelWarps), 0,
                                  stream, pdl, p);
        }
        if (e != cudaSuccess)
            return e;
        return cudaGetLastError();
    }
    const size_t smem = sizeof(uint32_t) * (size_t)p.maxB;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int rows = p.R * p.nq * p.Hs;
    cudaError_t e = launch_kernel(select_topk_kernel, dim3(rows), dim3(kSelThreads), smem, stream, pdl, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace msa

namespace msa {

cudaError_t launch_select_rows(const SelectParams &p, cudaStream_t stream)
{
    if (p.maxB <= 256)
        return launch_tile_t<8>(p, stream);
    if (p.maxB <= 512)
        return launch_tile_t<16>(p, stream);
    if (p.maxB <= 1024)
        return launch_tile_t<32>(p, stream);
    return launch_tile_t<64>(p, stream);
}

} // namespace msa
