// msa_decode.cu -- stage (c): GQA attention over the selected P128 pages.
//
// "MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2 for
// Blackwell", section "The TP4 decode target" (long-context sparse decode)
// and "Add Rubin (sm_107) MiniMax-M3.1 low-latency decode targets", section
// "Items and numerics" (split-K merge: fixed order, no atomics on the data,
// one divide per output) describe the stage; this is its GB300 design:
//
// * Work.  A unit is (token t, KV head g): 16 query heads against the
//   visible positions of the token's selected blocks.  Unit u = g * T + t
//   holds n_t = min(k, ceil((seq_len + j) / 128)) page tasks, so tokens of one
//   request that share a KV head sit next to each other and their common pages
//   are served from L2.  All tasks of all units are laid end to end and cut
//   into equal contiguous ranges, one per persistent CTA ("stream-K"), so
//   every SM streams the same number of pages whatever the unit sizes.
// * Merge.  A CTA that covers a whole unit writes its output directly.
//   Otherwise each CTA of the unit writes an unnormalised partial (o, m, l)
//   to its slot and bumps the unit's arrival counter; the CTA that arrives
//   last combines the slots in slot order (so the result does not depend on
//   which CTA is last), writes O and LSE, and resets the counter to zero.
// * Data movement.  Each CTA first gathers its task table (block id and page
//   of every task, through `selected` and the block table) into shared memory
//   with all threads at once, so no page lookup sits on the copy path.  Per
//   task the K and the V tile of KV head g (32 KiB each in bf16, 16 KiB in
//   FP8) are fetched by TMA (cp.async.bulk.tensor, 128-byte swizzle) into a
//   ring of shared-memory stages guarded by mbarriers; one thread keeps
//   kAhead tasks in flight.  The 16 query rows of each unit (4 KiB) arrive by
//   a 1-D bulk copy ahead of the unit.  Page offsets are 64-bit.
// * Math.  Each of the 4 warps owns 32 of the page's 128 tokens and keeps its
//   own online-softmax state for the 16 query heads; S = Q K^T and O += P V
//   are mma.sync m16n8k16 tiles fed by ldmatrix from the swizzled stages
//   (bf16), or by ldmatrix plus in-register E4M3 -> f16 converts (FP8: keys and
//   values are exact in f16; k_scale is folded into the logit scale and
//   v_scale into the output).  Logits are kept in base 2.  The 4 warps' states
//   are combined in a fixed order.
#include <cmath>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kDecThreads = 128;
constexpr int kQBufs = 4;     // query-row buffers (>= tasks in flight)
constexpr int kWin = 256;     // task-table window (two windows resident)
constexpr int kQBytes = kGroup * kDim * 2;

template <bool FP8>
struct Cfg {
    static constexpr int kTileBytes = FP8 ? 16384 : 32768;
    static constexpr int kStages = FP8 ? 8 : 4; // two stages (K, V) per task
    static constexpr int kAhead = kStages / 2;  // tasks in flight
    static constexpr int kRingBytes = kTileBytes * kStages;
    static_assert(kAhead <= kQBufs, "a unit's query buffer must outlive the tasks in flight");
    static_assert(kAhead < kWin, "the task table must hold the tasks in flight");
};

struct Task {
    int t, g, i;
};

// qt[t] = sum_{t' < t} n_t' (the tasks of one KV head before token t); qt[T] = total.
__device__ void build_token_prefix(const DecodeParams &p, int *qt)
{
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base < p.T; base += 32) {
            const int t = base + lane;
            int n = 0;
            if (t < p.T) {
                const int r = t / p.nq, j = t - r * p.nq;
                const int sl = p.seq_lens[r];
                const long long nb = ((long long)sl + p.nq - 1 + kPage - 1) / kPage;
                if (sl >= 1 && nb <= p.maxB) {
                    n = ceil_div(sl + j, kPage);
                    n = n < p.k ? n : p.k;
                }
            }
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o)
                    incl += v;
            }
            if (t < p.T)
                qt[t] = carry + incl - n;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0)
            qt[p.T] = carry;
    }
}

__device__ __forceinline__ Task task_of(long long x, const int *qt, int T)
{
    const int PT = qt[T];
    Task tk;
    tk.g = (int)(x / PT);
    const int rem = (int)(x - (long long)tk.g * PT);
    int lo = 0, hi = T - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (qt[mid] <= rem)
            lo = mid;
        else
            hi = mid - 1;
    }
    tk.t = lo;
    tk.i = rem - qt[lo];
    return tk;
}

// CTA that owns task x when P tasks are cut into G equal ranges:
// range(c) = [floor(c P / G), floor((c+1) P / G)).
__device__ __forceinline__ int owner_of(long long x, long long P, int G)
{
    return (int)(((x + 1) * G + P - 1) / P) - 1;
}

__device__ __forceinline__ bool range_empty(int c, long long P, int G)
{
    return (long long)c * P / G == (long long)(c + 1) * P / G;
}

// Table entry of task x: {K-tile row in the KV tensor map or -1, block id, t, g}.
__device__ int4 make_entry(const DecodeParams &p, long long x, const int *qt)
{
    const Task tk = task_of(x, qt, p.T);
    const int r = tk.t / p.nq, j = tk.t - r * p.nq;
    const int n_vis = ceil_div(p.seq_lens[r] + j, kPage);
    const int b = p.selected[(size_t)tk.t * p.k + tk.i];
    int row = -1;
    if (b < 0 || b >= n_vis) {
        set_error(p.err, kErrSelection);
    } else {
        const long long page = p.block_table[(size_t)r * p.maxB + b];
        if (page < 0 || page >= p.num_pages)
            set_error(p.err, kErrPage);
        else
            row = (int)(((page * 2) * p.Hkv + tk.g) * kPage);
    }
    return make_int4(row, b, tk.t, tk.g);
}

// Output dimension of accumulator column `col` (0..7) of n-tile nt.
template <bool FP8>
__device__ __forceinline__ int o_dim(int nt, int col)
{
    // bf16: n-tile nt = dims 8nt..8nt+7.  FP8: virtual n-tile nt = (chunk C,
    // parity) covers dims 16C + 2n + parity.
    return FP8 ? (nt >> 1) * 16 + 2 * col + (nt & 1) : nt * 8 + col;
}

template <bool FP8>
__global__ void __launch_bounds__(kDecThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p)
{
    using C = Cfg<FP8>;
    extern __shared__ uint8_t smem_raw[];
    // ring at a 1024-byte boundary (128-byte swizzle atoms)
    uint8_t *ring = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *qbuf = ring + C::kRingBytes;                                  // [kQBufs][16][128] bf16
    uint64_t *bars = reinterpret_cast<uint64_t *>(qbuf + kQBufs * kQBytes); // [kStages]
    uint64_t *qbars = bars + C::kStages;                                   // [kQBufs]
    int4 *table = reinterpret_cast<int4 *>(qbars + kQBufs);               // [2][kWin]
    float *comb_o = reinterpret_cast<float *>(table + 2 * kWin);          // [16][128]
    float *comb_m = comb_o + kGroup * kDim;                               // [4][16]
    float *comb_l = comb_m + 4 * kGroup;                                  // [4][16]
    int *s_flag = reinterpret_cast<int *>(comb_l + 4 * kGroup);           // [4]
    int *qt = s_flag + 4;                                                  // [T + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g8 = lane >> 2, q4 = lane & 3;

    // ---- prologue: everything that does not read the previous kernel's output ----
    if (threadIdx.x == 0) {
        prefetch_tensormap(&kv_map);
        for (int s = 0; s < C::kStages; ++s)
            mbar_init(smem_u32(&bars[s]), 1);
        for (int s = 0; s < kQBufs; ++s)
            mbar_init(smem_u32(&qbars[s]), 1);
        fence_mbar_init();
    }
    build_token_prefix(p, qt);
    __syncthreads();

    const long long P = (long long)p.Hkv * qt[p.T];
    const int G = gridDim.x, c = blockIdx.x;
    const long long x_begin = (long long)c * P / G, x_end = (long long)(c + 1) * P / G;
    const int ntasks = (int)(x_end - x_begin);

    // `selected` comes from the previous kernel of the step
    grid_dependency_wait();
    if (ntasks == 0)
        return;

    auto fill_window = [&](int w) {
        const int l0 = w * kWin;
        int4 *dst = table + (w & 1) * kWin;
        for (int i = threadIdx.x; i < kWin && l0 + i < ntasks; i += kDecThreads)
            dst[i] = make_entry(p, x_begin + l0 + i, qt);
    };
    fill_window(0);
    if (ntasks > kWin)
        fill_window(1);
    __syncthreads();

    auto entry = [&](int l) -> int4 { return table[((l / kWin) & 1) * kWin + (l % kWin)]; };

    // ---- producer (thread 0): K and V tiles of task l into stages 2l, 2l+1 mod S,
    // and the query rows of every new unit into qbuf[unit index mod kQBufs] ----
    int issued_tiles = 0;   // thread 0 only
    int prod_units = 0;     // thread 0 only
    int prod_last = -1;     // thread 0 only: unit of the last issued task
    auto issue = [&](int l) {
        const int4 e = entry(l);
        const int u = e.w * p.T + e.z;
        if (u != prod_last) {
            prod_last = u;
            const int qb = prod_units % kQBufs;
            ++prod_units;
            const uint32_t qbar = smem_u32(&qbars[qb]);
            mbar_arrive_expect_tx(qbar, kQBytes);
            bulk_load(smem_u32(qbuf + qb * kQBytes),
                      p.q + ((size_t)e.z * p.Hkv * kGroup + (size_t)e.w * kGroup) * kDim, kQBytes,
                      qbar);
        }
        issued_tiles = 2 * l + 2;
        for (int kv = 0; kv < 2; ++kv) {
            const int z = 2 * l + kv;
            const uint32_t bar = smem_u32(&bars[z % C::kStages]);
            const uint32_t dst = smem_u32(ring + (size_t)(z % C::kStages) * C::kTileBytes);
            if (e.x < 0) {
                mbar_arrive(bar); // completes the phase with no data; consumers skip the task
                continue;
            }
            const int row = e.x + kv * p.Hkv * kPage;
            mbar_arrive_expect_tx(bar, C::kTileBytes);
            tma_load_2d(dst, &kv_map, 0, row, bar);
            if (!FP8)
                tma_load_2d(dst + 16384, &kv_map, 64, row, bar);
        }
    };
    if (threadIdx.x == 0) {
        const int pre = ntasks < C::kAhead ? ntasks : C::kAhead;
        for (int l = 0; l < pre; ++l)
            issue(l);
    }

    // ---- consumer state (every warp) ----
    float o[16][4];
    float m_run[2], l_run[2];
    uint32_t qa[8][4];
    int cur_unit = -1, cons_units = 0;
    int cur_t = 0, cur_g = 0;
    bool abort = false;
    int abort_task = 0;
    const int tb = warp * 32; // this warp's tokens within a page

    auto reset_state = [&]() {
#pragma unroll
        for (int n = 0; n < 16; ++n)
            o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
    };

    // query fragments of the current unit from its shared-memory buffer
    auto load_q = [&](int qb) {
        const uint8_t *qs = qbuf + qb * kQBytes;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint8_t *r0 = qs + g8 * (kDim * 2);
            const uint8_t *r1 = qs + (g8 + 8) * (kDim * 2);
            if (!FP8) {
                qa[s][0] = *reinterpret_cast<const uint32_t *>(r0 + (16 * s + 2 * q4) * 2);
                qa[s][1] = *reinterpret_cast<const uint32_t *>(r1 + (16 * s + 2 * q4) * 2);
                qa[s][2] = *reinterpret_cast<const uint32_t *>(r0 + (16 * s + 8 + 2 * q4) * 2);
                qa[s][3] = *reinterpret_cast<const uint32_t *>(r1 + (16 * s + 8 + 2 * q4) * 2);
            } else {
                // permuted k order matching the FP8 key fragments: k-step s covers
                // dims 16s + 4q4 .. +3 (slots 2q4,2q4+1 <- +0,+1; 2q4+8,+9 <- +2,+3)
                const uint2 v0 = *reinterpret_cast<const uint2 *>(r0 + (16 * s + 4 * q4) * 2);
                const uint2 v1 = *reinterpret_cast<const uint2 *>(r1 + (16 * s + 4 * q4) * 2);
                qa[s][0] = bf16x2_to_f16x2(v0.x);
                qa[s][1] = bf16x2_to_f16x2(v1.x);
                qa[s][2] = bf16x2_to_f16x2(v0.y);
                qa[s][3] = bf16x2_to_f16x2(v1.y);
            }
        }
    };

    // O and LSE rows of unit (t, g) from a combined (o, M, L): o is unnormalised.
    auto store_final = [&](int t, int g, int row, int d0, const float (&v)[8], float M, float L) {
        const float inv = L > 0.f ? 1.f / L : 0.f; // one reciprocal per row
        uint4 packed;
        packed.x = pack_bf16(v[0] * inv, v[1] * inv);
        packed.y = pack_bf16(v[2] * inv, v[3] * inv);
        packed.z = pack_bf16(v[4] * inv, v[5] * inv);
        packed.w = pack_bf16(v[6] * inv, v[7] * inv);
        const size_t h = (size_t)t * p.Hkv * kGroup + (size_t)g * kGroup + row;
        *reinterpret_cast<uint4 *>(p.out + h * kDim + d0) = packed;
        if (d0 == 0)
            p.lse[h] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * 0.69314718055994531f;
    };

    // Combine the 4 warps' states of unit (t, g); write its output, or its
    // partial and, if this CTA is the last of the unit to arrive, the merge.
    auto finalize = [&](int t, int g) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
        }
        if (q4 == 0) {
            comb_m[warp * kGroup + g8] = m_run[0];
            comb_m[warp * kGroup + g8 + 8] = m_run[1];
            comb_l[warp * kGroup + g8] = l_run[0];
            comb_l[warp * kGroup + g8 + 8] = l_run[1];
        }
        __syncthreads();
        float fac[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = g8 + 8 * h;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                M = fmaxf(M, comb_m[w * kGroup + row]);
            fac[h] = (M == -INFINITY) ? 0.f : ex2(m_run[h] - M);
        }
        // fixed order (warp 0, 1, 2, 3): bitwise reproducible
        for (int w = 0; w < 4; ++w) {
            if (warp == w) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const int d = o_dim<FP8>(n, 2 * q4 + cc);
                        float *a = &comb_o[g8 * kDim + d];
                        float *b = &comb_o[(g8 + 8) * kDim + d];
                        const float va = o[n][cc] * fac[0], vb = o[n][2 + cc] * fac[1];
                        *a = w == 0 ? va : *a + va;
                        *b = w == 0 ? vb : *b + vb;
                    }
                }
            }
            __syncthreads();
        }
        const long long Pt = qt[p.T];
        const long long u_first = (long long)g * Pt + qt[t];
        const int n_u = qt[t + 1] - qt[t];
        const int c_first = owner_of(u_first, P, G);
        const int c_last = owner_of(u_first + n_u - 1, P, G);
        const int u = g * p.T + t;
        const bool whole = c_first == c_last;
        float *slot = p.partial + (size_t)(c + u) * kPartialFloats;
        for (int e = threadIdx.x; e < kGroup * kDim / 8; e += kDecThreads) {
            const int row = e >> 4, d0 = (e & 15) * 8;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                M = fmaxf(M, comb_m[w * kGroup + row]);
            float L = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                L += (M == -INFINITY) ? 0.f : comb_l[w * kGroup + row] * ex2(comb_m[w * kGroup + row] - M);
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                v[i] = comb_o[row * kDim + d0 + i] * p.v_scale;
            if (whole) {
                store_final(t, g, row, d0, v, M, L);
            } else {
                float4 *dst = reinterpret_cast<float4 *>(slot + row * kDim + d0);
                dst[0] = make_float4(v[0], v[1], v[2], v[3]);
                dst[1] = make_float4(v[4], v[5], v[6], v[7]);
                if (d0 == 0) {
                    slot[kGroup * kDim + row] = M;
                    slot[kGroup * kDim + kGroup + row] = L;
                }
            }
        }
        if (!whole) {
            __threadfence(); // publish this CTA's slot before counting in
            __syncthreads();
            if (threadIdx.x == 0) {
                int arrivals = 0;
                for (int cc = c_first; cc <= c_last; ++cc)
                    arrivals += !range_empty(cc, P, G);
                const int before = atomicAdd(&p.counters[u], 1);
                s_flag[0] = before == arrivals - 1;
            }
            __syncthreads();
            if (s_flag[0]) {
                __threadfence();
                // merge every slot of the unit, in slot order
                const float *base = p.partial + (size_t)(c_first + u) * kPartialFloats;
                const int nslots = c_last - c_first + 1;
                for (int e = threadIdx.x; e < kGroup * kDim / 8; e += kDecThreads) {
                    const int row = e >> 4, d0 = (e & 15) * 8;
                    float M = -INFINITY;
                    for (int s = 0; s < nslots; ++s)
                        if (!range_empty(c_first + s, P, G))
                            M = fmaxf(M, __ldcg(base + (size_t)s * kPartialFloats + kGroup * kDim + row));
                    float L = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                    for (int s = 0; s < nslots; ++s) {
                        if (range_empty(c_first + s, P, G))
                            continue;
                        const float *sl = base + (size_t)s * kPartialFloats;
                        const float ms = __ldcg(sl + kGroup * kDim + row);
                        const float wgt = (M == -INFINITY) ? 0.f : ex2(ms - M);
                        L += wgt * __ldcg(sl + kGroup * kDim + kGroup + row);
                        const float4 a = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0));
                        const float4 b = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0 + 4));
                        acc[0] += wgt * a.x; acc[1] += wgt * a.y; acc[2] += wgt * a.z; acc[3] += wgt * a.w;
                        acc[4] += wgt * b.x; acc[5] += wgt * b.y; acc[6] += wgt * b.z; acc[7] += wgt * b.w;
                    }
                    store_final(t, g, row, d0, acc, M, L);
                }
                if (threadIdx.x == 0)
                    p.counters[u] = 0; // ready for the next call
            }
        }
        __syncthreads();
    };

    for (int l = 0; l < ntasks; ++l) {
        const int4 e = entry(l);
        const int u = e.w * p.T + e.z;
        if (u != cur_unit) {
            if (cur_unit >= 0)
                finalize(cur_t, cur_g);
            cur_unit = u;
            cur_t = e.z;
            cur_g = e.w;
            reset_state();
            const int qb = cons_units % kQBufs;
            if (!mbar_wait_bounded(smem_u32(&qbars[qb]), (cons_units / kQBufs) & 1))
                abort = true;
            ++cons_units;
            load_q(qb);
        }
        const int r = e.z / p.nq, j = e.z - r * p.nq;
        const int L = p.seq_lens[r] + j;
        const int zk = 2 * l, zv = 2 * l + 1;
        const uint32_t tileK = smem_u32(ring + (size_t)(zk % C::kStages) * C::kTileBytes);
        const uint32_t tileV = smem_u32(ring + (size_t)(zv % C::kStages) * C::kTileBytes);

        bool ok = mbar_wait_bounded(smem_u32(&bars[zk % C::kStages]), (zk / C::kStages) & 1);
        ok = mbar_wait_bounded(smem_u32(&bars[zv % C::kStages]), (zv / C::kStages) & 1) && ok;
        if (!ok)
            abort = true;

        if (e.x >= 0 && !abort) {
            // ---- S = Q K^T over this warp's 32 tokens: 4 n-tiles of 8 tokens ----
            float s[4][4];
#pragma unroll
            for (int n = 0; n < 4; ++n)
                s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
            if (!FP8) {
#pragma unroll
                for (int n2 = 0; n2 < 2; ++n2) {
                    const int mi = lane >> 3;
                    const int tok = tb + 16 * n2 + ((mi >> 1) << 3) + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int chunk = 2 * ks + (mi & 1);
                        const uint32_t addr = tileK + (chunk >> 3) * 16384 + tok * 128 +
                                              (((chunk & 7) ^ (tok & 7)) << 4);
                        uint32_t b[4];
                        ldsm_x4(b, addr);
                        mma_bf16(s[2 * n2], qa[ks], b[0], b[1]);
                        mma_bf16(s[2 * n2 + 1], qa[ks], b[2], b[3]);
                    }
                }
            } else {
#pragma unroll
                for (int n2 = 0; n2 < 2; ++n2) {
                    const int mi = lane >> 3;
                    const int tok = tb + 16 * n2 + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int ks = 0; ks < 8; ks += 2) {
                        const int chunk = ks + (mi >> 1);
                        const uint32_t addr = tileK + tok * 128 + ((chunk ^ (tok & 7)) << 4);
                        uint32_t b[4];
                        ldsm_x4(b, addr);
                        // b[0]: (n-tile 2n2, k-step ks), b[1]: (2n2+1, ks), b[2]: (2n2, ks+1), b[3]: (2n2+1, ks+1)
                        mma_f16(s[2 * n2], qa[ks], e4m3x2_to_f16x2(b[0] & 0xFFFFu),
                                e4m3x2_to_f16x2(b[0] >> 16));
                        mma_f16(s[2 * n2 + 1], qa[ks], e4m3x2_to_f16x2(b[1] & 0xFFFFu),
                                e4m3x2_to_f16x2(b[1] >> 16));
                        mma_f16(s[2 * n2], qa[ks + 1], e4m3x2_to_f16x2(b[2] & 0xFFFFu),
                                e4m3x2_to_f16x2(b[2] >> 16));
                        mma_f16(s[2 * n2 + 1], qa[ks + 1], e4m3x2_to_f16x2(b[3] & 0xFFFFu),
                                e4m3x2_to_f16x2(b[3] >> 16));
                    }
                }
            }

            // ---- scale, causal mask, online softmax (base 2) ----
            const int pos0 = e.y * kPage + tb; // position of this warp's token 0
            const bool need_mask = pos0 + 32 > L;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int n = 0; n < 4; ++n) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v = s[n][k] * p.scale_log2;
                    if (need_mask && pos0 + 8 * n + 2 * q4 + (k & 1) >= L)
                        v = -INFINITY;
                    s[n][k] = v;
                    mx[k >> 1] = fmaxf(mx[k >> 1], v);
                }
            }
            float ref[2], alpha[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                const float m_new = fmaxf(m_run[h], mx[h]);
                ref[h] = (m_new == -INFINITY) ? 0.f : m_new;
                alpha[h] = ex2(m_run[h] - ref[h]); // 0 when m_run is -inf
                m_run[h] = m_new;
                l_run[h] *= alpha[h];
            }
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o[n][0] *= alpha[0];
                o[n][1] *= alpha[0];
                o[n][2] *= alpha[1];
                o[n][3] *= alpha[1];
            }
            uint32_t pa[2][4];
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const float p0 = ex2(s[n][0] - ref[0]), p1 = ex2(s[n][1] - ref[0]);
                const float p2 = ex2(s[n][2] - ref[1]), p3 = ex2(s[n][3] - ref[1]);
                l_run[0] += p0 + p1;
                l_run[1] += p2 + p3;
                // A fragment of P for k-step n/2: n-tile 2kk -> regs 0,1; 2kk+1 -> regs 2,3
                const int kk = n >> 1, hi = (n & 1) * 2;
                pa[kk][hi + 0] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
                pa[kk][hi + 1] = FP8 ? pack_f16(p2, p3) : pack_bf16(p2, p3);
            }

            // ---- O += P V over this warp's 32 tokens ----
            if (!FP8) {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int mi = lane >> 3;
                    const int tok = tb + 16 * kk + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int nd2 = 0; nd2 < 8; ++nd2) {
                        const int chunk = 2 * nd2 + (mi >> 1);
                        const uint32_t addr = tileV + (chunk >> 3) * 16384 + tok * 128 +
                                              (((chunk & 7) ^ (tok & 7)) << 4);
                        uint32_t b[4];
                        ldsm_x4_t(b, addr);
                        mma_bf16(o[2 * nd2], pa[kk], b[0], b[1]);
                        mma_bf16(o[2 * nd2 + 1], pa[kk], b[2], b[3]);
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const int mi = lane >> 3;
                    const int tok = tb + 16 * kk + ((mi & 1) << 3) + (lane & 7);
#pragma unroll
                    for (int C2 = 0; C2 < 8; C2 += 2) {
                        const int chunk = C2 + (mi >> 1);
                        const uint32_t addr = tileV + tok * 128 + ((chunk ^ (tok & 7)) << 4);
                        uint32_t b[4];
                        ldsm_x4_t(b, addr);
                        // b[0]: tokens 0-7 of the k-step, chunk C2; b[1]: tokens 8-15, C2;
                        // b[2], b[3]: chunk C2+1.  Bytes: {V[2q][2g], V[2q][2g+1], V[2q+1][2g], V[2q+1][2g+1]}
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t lo = __byte_perm(b[2 * h], 0, 0x3120);
                            const uint32_t hi = __byte_perm(b[2 * h + 1], 0, 0x3120);
                            const int vn = 2 * (C2 + h); // even-dim virtual n-tile of chunk C2+h
                            mma_f16(o[vn], pa[kk], e4m3x2_to_f16x2(lo & 0xFFFFu), e4m3x2_to_f16x2(hi & 0xFFFFu));
                            mma_f16(o[vn + 1], pa[kk], e4m3x2_to_f16x2(lo >> 16), e4m3x2_to_f16x2(hi >> 16));
                        }
                    }
                }
            }
        }

        // every warp is done with both stages of task l
        abort = __syncthreads_or(abort);
        if (abort) {
            abort_task = l;
            break;
        }
        // refill the table window that task l closed
        if ((l + 1) % kWin == 0 && l + 1 + kWin < ntasks) {
            fill_window((l + 1) / kWin + 1);
            __syncthreads();
        }
        if (threadIdx.x == 0 && l + C::kAhead < ntasks)
            issue(l + C::kAhead);
    }

    if (abort) {
        if (threadIdx.x == 0) {
            set_error(p.err, kErrTimeout);
            // Wait (bounded) for every copy issued and not yet consumed, so none
            // lands in shared memory after the CTA has exited.
            for (int z = 2 * abort_task; z < issued_tiles; ++z)
                (void)mbar_wait_bounded(smem_u32(&bars[z % C::kStages]), (z / C::kStages) & 1);
            for (int u = cons_units; u < prod_units; ++u)
                (void)mbar_wait_bounded(smem_u32(&qbars[u % kQBufs]), (u / kQBufs) & 1);
        }
        return;
    }
    finalize(cur_t, cur_g);
}

// ---- tensor map of the KV pool: rows of 128 elements, [pages*2*Hkv*128] rows ----

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn load_encode()
{
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<EncodeFn>(ptr);
    return nullptr;
}

EncodeFn get_encode()
{
    static const EncodeFn fn = load_encode(); // thread-safe one-time lookup
    return fn;
}

bool encode_kv_map(CUtensorMap *map, const void *kv_pool, int kv_dtype, int num_pages, int Hkv)
{
    EncodeFn enc = get_encode();
    if (!enc)
        return false;
    const bool fp8 = kv_dtype == MSA_FP8_E4M3;
    const cuuint64_t rows = (cuuint64_t)num_pages * 2 * Hkv * kPage;
    const cuuint64_t dims[2] = {(cuuint64_t)kDim, rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kDim * (fp8 ? 1 : 2)};
    const cuuint32_t box[2] = {fp8 ? 128u : 64u, (cuuint32_t)kPage};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                           const_cast<void *>(kv_pool), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <bool FP8>
size_t decode_smem_bytes(int T)
{
    using C = Cfg<FP8>;
    return 1024 + C::kRingBytes + kQBufs * kQBytes + (C::kStages + kQBufs) * sizeof(uint64_t) +
           2 * kWin * sizeof(int4) + sizeof(float) * (kGroup * kDim + 8 * kGroup) +
           sizeof(int) * (size_t)(4 + T + 1);
}

template <bool FP8>
cudaError_t launch_decode_t(const DecodeParams &p, const CUtensorMap &map, int ctas,
                            cudaStream_t stream, bool pdl)
{
    const size_t smem = decode_smem_bytes<FP8>(p.T);
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<FP8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = launch_kernel(sparse_decode_kernel<FP8>, dim3(ctas), dim3(kDecThreads), smem, stream, pdl,
                      map, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_sparse_decode(const DecodeParams &p, const void *kv_pool, int kv_dtype, int ctas,
                                 cudaStream_t stream, bool pdl)
{
    CUtensorMap map;
    if (!encode_kv_map(&map, kv_pool, kv_dtype, p.num_pages, p.Hkv))
        return cudaErrorInvalidValue;
    if (kv_dtype == MSA_FP8_E4M3)
        return launch_decode_t<true>(p, map, ctas, stream, pdl);
    return launch_decode_t<false>(p, map, ctas, stream, pdl);
}

} // namespace msa
