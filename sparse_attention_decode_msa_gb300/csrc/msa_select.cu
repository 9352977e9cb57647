// msa_select.cu -- stage (b): top-k block selection.
//
// Contract ("MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2
// for Blackwell", section "The TP4 decode target"): the k blocks with the
// largest block score, score ties broken toward the smaller block index, for
// any tie width.  Output ("Add Rubin (sm_107) MiniMax-M3.1 low-latency decode
// targets", q8kv4 indexer commit): ascending block ids, -1 padded to k.
//
// One CTA per token.  Scores map to order-preserving 32-bit keys; an MSB-first
// radix select (four 8-bit digits) finds the k-th largest key theta and how
// many of the blocks equal to theta are still needed.  A block is selected if
// its key is above theta, or equal to theta and among the first `need` such
// blocks in index order.  Two CTA-wide exclusive scans over blocks in index
// order give each tie its rank and each selected block its output slot, so
// the table comes out ascending with no sort.  Comparisons only: bit-exact.
#include "msa_internal.cuh"

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

__global__ void __launch_bounds__(kSelThreads) select_topk_kernel(const SelectParams p)
{
    extern __shared__ uint32_t keys[]; // [maxB]
    __shared__ int hist[256];
    __shared__ int scan_tmp[kSelWarps + 1];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;

    launch_dependents(); // the decode may start its prologue while tokens are selected
    const int t = blockIdx.x;
    const int r = t / p.nq, j = t - r * p.nq;
    int32_t *out = p.selected + (size_t)t * p.k;
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
    const float *row = p.block_scores + (size_t)t * p.maxB;
    for (int b = threadIdx.x; b < n; b += kSelThreads)
        keys[b] = order_key(row[b]);
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

} // namespace

cudaError_t launch_select(const SelectParams &p, cudaStream_t stream, bool pdl)
{
    const size_t smem = sizeof(uint32_t) * (size_t)p.maxB;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_topk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
    }
    const int T = p.R * p.nq;
    cudaError_t e = launch_kernel(select_topk_kernel, dim3(T), dim3(kSelThreads), smem, stream, pdl, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace msa
