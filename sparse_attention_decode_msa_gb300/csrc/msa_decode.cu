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
// * Data movement.  One producer warp gathers the CTA's task table (block id
//   and page of every task, through `selected` and the block table) into
//   shared memory ahead of use, and issues the copies: per task the K and the
//   V tile of KV head g (32 KiB each in bf16, 16 KiB in FP8) by TMA
//   (cp.async.bulk.tensor, 128-byte swizzle) into a ring of shared-memory
//   stages, each guarded by a "full" mbarrier (bytes landed) and an "empty"
//   mbarrier (all consumer warps done), and the 16 query rows of each unit
//   (4 KiB) by a 1-D bulk copy.  Consumers hand a K stage back as soon as
//   Q K^T has read it.  Page offsets are 64-bit.
// * Math.  Each of the 8 consumer warps owns 16 of the page's 128 tokens and
//   keeps its own online-softmax state for the 16 query heads; S = Q K^T and
//   O += P V are mma.sync m16n8k16 tiles fed by ldmatrix from the swizzled
//   stages (bf16), or by ldmatrix plus in-register E4M3 -> f16 converts (FP8:
//   keys and values are exact in f16; k_scale is folded into the logit scale
//   and v_scale into the output).  Logits are kept in base 2.  The warps'
//   states are combined in a fixed order.
// * Every wait is bounded; a timeout sets MSA_ERR_TIMEOUT, raises a CTA abort
//   flag that ends every other wait, and the producer waits (bounded) for its
//   copies in flight before the CTA exits.
#include <cmath>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kConsumerWarps = 8;              // each owns kTPW tokens of every page
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kTPW = kPage / kConsumerWarps;   // tokens per consumer warp
constexpr int kNT = kTPW / 8;                  // S n-tiles (8 tokens) per warp
constexpr int kKK = kTPW / 16;                 // P.V k-steps (16 tokens) per warp
constexpr int kVPR = 64 / kConsumerWarps;      // accumulator values per lane per combine round
static_assert(kTPW % 16 == 0, "a warp's tokens must fill whole m16n8k16 k-steps");
constexpr int kDecThreads = kConsumers + 32; // + one producer warp
constexpr int kQBufs = 2;                    // query-row buffers
constexpr int kWin = 128;                    // task-table window (two windows resident)
constexpr int kQBytes = kGroup * kDim * 2;
constexpr int kMaxSmem = 232448;             // dynamic shared memory limit per CTA

template <bool FP8, int STAGES>
struct Cfg {
    static constexpr int kTileBytes = FP8 ? 16384 : 32768;
    static constexpr int kAhead = STAGES / 2;  // tasks the producer may run ahead
    static constexpr int kRingBytes = kTileBytes * STAGES;
    static_assert(STAGES % 2 == 0, "K and V of a task take two stages");
    static_assert(kAhead < kWin, "the task table must cover the tasks in flight");
};

// Shared-memory layout of the decode CTA (offsets from a 1024-byte aligned
// base); the host sizes the allocation with the same function.
struct SmemLayout {
    size_t ring, qbuf, bars, table, cbuf, comb, flags, qt, total;
};

__host__ __device__ constexpr size_t align_to(size_t v, size_t a)
{
    return (v + a - 1) / a * a;
}

__host__ __device__ inline SmemLayout decode_layout(int T, int stages, int tile_bytes)
{
    SmemLayout L{};
    size_t off = 0;
    L.ring = off;                                   // 1024-aligned: 128-byte swizzle atoms
    off += (size_t)stages * tile_bytes;
    L.qbuf = off = align_to(off, 128);             // bulk-copy destinations: 16-byte aligned
    off += (size_t)kQBufs * kQBytes;
    L.bars = off = align_to(off, 8);               // full[S], empty[S], qfull, qempty, consumer barrier
    off += (size_t)(2 * stages + 2 * kQBufs + 1) * 8;
    L.table = off = align_to(off, 16);             // int4 entries
    off += (size_t)2 * kWin * 16;
    L.cbuf = off = align_to(off, 16);              // [warps][kVPR][32] floats (8 KiB)
    off += (size_t)kConsumerWarps * kVPR * 32 * 4;
    L.comb = off = align_to(off, 16);              // comb_m[4][16], comb_l[4][16]
    off += (size_t)2 * kConsumerWarps * kGroup * 4;
    L.flags = off = align_to(off, 16);             // 4 ints
    off += 16;
    L.qt = off = align_to(off, 16);                // [T + 1] ints
    off += (size_t)(T + 1) * 4;
    L.total = align_to(off, 16) + 1024;            // + slack to align the base
    return L;
}

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

// Table entry of task x: {K-tile row in the KV tensor map or -1, visible
// tokens of the page (1..128: the causal limit cuts the last block), t, g}.
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
    const int nvis = min(kPage, p.seq_lens[r] + j - b * kPage);
    return make_int4(row, nvis, tk.t, tk.g);
}

// Output dimension of accumulator column `col` (0..7) of n-tile nt.
template <bool FP8>
__device__ __forceinline__ int o_dim(int nt, int col)
{
    // bf16: n-tile nt = dims 8nt..8nt+7.  FP8: virtual n-tile nt = (chunk C,
    // parity) covers dims 16C + 2n + parity.
    return FP8 ? (nt >> 1) * 16 + 2 * col + (nt & 1) : nt * 8 + col;
}

template <bool FP8, int STAGES>
__global__ void __launch_bounds__(kDecThreads, 1)
    sparse_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p)
{
    using C = Cfg<FP8, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemLayout lay = decode_layout(p.T, STAGES, C::kTileBytes);
    uint8_t *ring = base + lay.ring;                                    // [S] tiles
    uint8_t *qbuf = base + lay.qbuf;                                    // [kQBufs][16][128] bf16
    uint64_t *full = reinterpret_cast<uint64_t *>(base + lay.bars);    // [S] tile landed
    uint64_t *empty = full + STAGES;                                    // [S] tile consumed
    uint64_t *qfull = empty + STAGES;                                   // [kQBufs]
    uint64_t *qempty = qfull + kQBufs;                                  // [kQBufs]
    uint64_t *csync_bar = qempty + kQBufs;                              // consumer barrier
    int4 *table = reinterpret_cast<int4 *>(base + lay.table);          // [2][kWin]
    float *cbuf = reinterpret_cast<float *>(base + lay.cbuf);          // [warps][kVPR][32]
    float *comb_m = reinterpret_cast<float *>(base + lay.comb);        // [warps][16]
    float *comb_l = comb_m + kConsumerWarps * kGroup;                   // [warps][16]
    int *s_flag = reinterpret_cast<int *>(base + lay.flags);           // [0] last, [1] abort
    int *qt = reinterpret_cast<int *>(base + lay.qt);                  // [T + 1]
    volatile int *abort_flag = s_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- prologue: everything that does not read the previous kernel's output ----
    if (threadIdx.x == 0) {
        prefetch_tensormap(&kv_map);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        for (int s = 0; s < kQBufs; ++s) {
            mbar_init(smem_u32(&qfull[s]), 1);
            mbar_init(smem_u32(&qempty[s]), kConsumerWarps);
        }
        mbar_init(smem_u32(csync_bar), kConsumers);
        s_flag[0] = 0;
        s_flag[1] = 0;
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

    auto entry = [&](int l) -> int4 { return table[((l / kWin) & 1) * kWin + (l % kWin)]; };

    if (warp == kConsumerWarps) {
        // =================== producer warp ===================
        auto fill_window = [&](int w) {
            const int l0 = w * kWin;
            int4 *dst = table + (w & 1) * kWin;
            for (int i = lane; i < kWin && l0 + i < ntasks; i += 32)
                dst[i] = make_entry(p, x_begin + l0 + i, qt);
            __syncwarp();
        };
        fill_window(0);
        if (ntasks > kWin)
            fill_window(1);
        int issued = 0;        // tiles issued (lane 0)
        int q_issued = 0;      // query-row copies issued (lane 0)
        int prod_units = 0, prod_last = -1;
        bool ok = true;
        for (int l = 0; l < ntasks && ok; ++l) {
            // K stage of task l: wait until the consumers released its previous tile
            const int zk = 2 * l;
            if (lane == 0 && zk >= STAGES)
                ok = mbar_wait_or_abort(smem_u32(&empty[zk % STAGES]), ((zk / STAGES) - 1) & 1,
                                        abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            // the consumers have read every entry up to task l - S/2: the window
            // before this one can be replaced by the one after it
            if (l % kWin == C::kAhead && l >= kWin && (l / kWin + 1) * kWin < ntasks)
                fill_window(l / kWin + 1);
            if (lane == 0) {
                const int4 e = entry(l);
                const int u = e.w * p.T + e.z;
                if (u != prod_last) {
                    prod_last = u;
                    const int qb = prod_units % kQBufs;
                    if (prod_units >= kQBufs)
                        ok = mbar_wait_or_abort(smem_u32(&qempty[qb]),
                                                ((prod_units / kQBufs) - 1) & 1, abort_flag);
                    if (ok) {
                        const uint32_t qbar = smem_u32(&qfull[qb]);
                        mbar_arrive_expect_tx(qbar, kQBytes);
                        bulk_load(smem_u32(qbuf + qb * kQBytes),
                                  p.q + ((size_t)e.z * p.Hkv * kGroup + (size_t)e.w * kGroup) * kDim,
                                  kQBytes, qbar);
                        q_issued = prod_units + 1;
                    }
                    ++prod_units;
                }
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int z = zk + kv;
                    const int st = z % STAGES;
                    if (kv == 1 && z >= STAGES)
                        ok = mbar_wait_or_abort(smem_u32(&empty[st]), ((z / STAGES) - 1) & 1,
                                                abort_flag);
                    if (!ok)
                        break;
                    const uint32_t bar = smem_u32(&full[st]);
                    issued = z + 1;
                    if (e.x < 0) {
                        mbar_arrive(bar); // completes the phase with no data; consumers skip the task
                        continue;
                    }
                    const uint32_t dst = smem_u32(ring + (size_t)st * C::kTileBytes);
                    const int row = e.x + kv * p.Hkv * kPage;
                    mbar_arrive_expect_tx(bar, C::kTileBytes);
                    tma_load_2d(dst, &kv_map, 0, row, bar);
                    if (!FP8)
                        tma_load_2d(dst + 16384, &kv_map, 64, row, bar);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (!ok && lane == 0) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            // Wait (bounded) for every copy this warp issued, so none lands in
            // shared memory after the CTA has exited.
            for (int z = issued - STAGES < 0 ? 0 : issued - STAGES; z < issued; ++z)
                (void)mbar_wait_bounded(smem_u32(&full[z % STAGES]), (z / STAGES) & 1);
            for (int u = q_issued - kQBufs < 0 ? 0 : q_issued - kQBufs; u < q_issued; ++u)
                (void)mbar_wait_bounded(smem_u32(&qfull[u % kQBufs]), (u / kQBufs) & 1);
        }
        return;
    }

    // =================== consumer warps 0..3 ===================
    const int g8 = lane >> 2, q4 = lane & 3;
    float o[16][4];
    float m_run[2], l_run[2];
    uint32_t qa[8][4];
    int cur_unit = -1, cons_units = 0, cur_t = 0, cur_g = 0;
    int sync_phase = 0;
    bool ok = true;
    const int tb = warp * kTPW; // this warp's tokens within a page

    // bounded barrier of the 128 consumer threads
    auto csync = [&]() {
        mbar_arrive(smem_u32(csync_bar));
        if (!mbar_wait_or_abort(smem_u32(csync_bar), sync_phase & 1, abort_flag))
            ok = false;
        ++sync_phase;
    };

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

    // Combine the warps' states of unit (t, g); write its output, or its
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
        csync();
        // per row (g8, g8 + 8): combined max M, denominator L, this warp's factor
        float M[2], L[2], fac[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = g8 + 8 * h;
            M[h] = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                M[h] = fmaxf(M[h], comb_m[w * kGroup + row]);
            L[h] = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                L[h] += (M[h] == -INFINITY) ? 0.f
                                            : comb_l[w * kGroup + row] * ex2(comb_m[w * kGroup + row] - M[h]);
            fac[h] = (M[h] == -INFINITY) ? 0.f : ex2(m_run[h] - M[h]);
        }
        const long long Pt = qt[p.T];
        const long long u_first = (long long)g * Pt + qt[t];
        const int n_u = qt[t + 1] - qt[t];
        const int c_first = owner_of(u_first, P, G);
        const int c_last = owner_of(u_first + n_u - 1, P, G);
        const int u = g * p.T + t;
        const bool whole = c_first == c_last;
        float *slot = p.partial + (size_t)(c + u) * kPartialFloats;
        const size_t hbase = (size_t)t * p.Hkv * kGroup + (size_t)g * kGroup;
        // Sum the warps' accumulators in kConsumerWarps rounds of kVPR values per
        // lane through an 8 KiB buffer laid out [warp][value][lane] (conflict-free);
        // warp rr sums round rr in warp order (fixed, so bitwise reproducible)
        // and writes those dimensions.
#pragma unroll
        for (int rr = 0; rr < kConsumerWarps; ++rr) {
#pragma unroll
            for (int i = 0; i < kVPR; ++i) {
                const int n = rr * (kVPR / 4) + (i >> 2), e = i & 3;
                cbuf[(warp * kVPR + i) * 32 + lane] = o[n][e] * fac[e >> 1];
            }
            csync();
            if (warp == rr) {
#pragma unroll
                for (int i = 0; i < kVPR; i += 2) {
                    const int n = rr * (kVPR / 4) + (i >> 2), e = i & 3; // e in {0, 2}: cols 2q4, 2q4+1 of row e/2
                    float v0 = 0.f, v1 = 0.f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        v0 += cbuf[(w * kVPR + i) * 32 + lane];
                        v1 += cbuf[(w * kVPR + i + 1) * 32 + lane];
                    }
                    const int h = e >> 1, row = g8 + 8 * h;
                    v0 *= p.v_scale;
                    v1 *= p.v_scale;
                    const int d0 = o_dim<FP8>(n, 2 * q4), d1 = o_dim<FP8>(n, 2 * q4 + 1);
                    if (whole) {
                        const float inv = L[h] > 0.f ? 1.f / L[h] : 0.f;
                        const uint32_t pk = pack_bf16(v0 * inv, v1 * inv);
                        uint16_t *orow = p.out + (hbase + row) * kDim;
                        if (!FP8) {
                            *reinterpret_cast<uint32_t *>(orow + d0) = pk; // d1 == d0 + 1
                        } else {
                            orow[d0] = (uint16_t)(pk & 0xFFFFu);
                            orow[d1] = (uint16_t)(pk >> 16);
                        }
                    } else {
                        float *srow = slot + row * kDim;
                        if (!FP8) {
                            *reinterpret_cast<float2 *>(srow + d0) = make_float2(v0, v1);
                        } else {
                            srow[d0] = v0;
                            srow[d1] = v1;
                        }
                    }
                }
            }
            csync();
        }
        if (warp == 0 && q4 == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = g8 + 8 * h;
                if (whole) {
                    p.lse[hbase + row] =
                        (M[h] == -INFINITY) ? -INFINITY : (M[h] + log2f(L[h])) * 0.69314718055994531f;
                } else {
                    slot[kGroup * kDim + row] = M[h];
                    slot[kGroup * kDim + kGroup + row] = L[h];
                }
            }
        }
        if (whole)
            return;
        __threadfence(); // publish this CTA's slot before counting in
        csync();
        if (threadIdx.x == 0) {
            int arrivals = 0;
            for (int cc = c_first; cc <= c_last; ++cc)
                arrivals += !range_empty(cc, P, G);
            const int before = atomicAdd(&p.counters[u], 1);
            s_flag[0] = before == arrivals - 1;
        }
        csync();
        if (s_flag[0]) {
            __threadfence();
            // merge every slot of the unit, in slot order; one reciprocal per row
            const float *base = p.partial + (size_t)(c_first + u) * kPartialFloats;
            const int nslots = c_last - c_first + 1;
            for (int e = threadIdx.x; e < kGroup * kDim / 8; e += kConsumers) {
                const int row = e >> 4, d0 = (e & 15) * 8;
                float Mx = -INFINITY;
                for (int s = 0; s < nslots; ++s)
                    if (!range_empty(c_first + s, P, G))
                        Mx = fmaxf(Mx, __ldcg(base + (size_t)s * kPartialFloats + kGroup * kDim + row));
                float Lx = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int s = 0; s < nslots; ++s) {
                    if (range_empty(c_first + s, P, G))
                        continue;
                    const float *sl = base + (size_t)s * kPartialFloats;
                    const float ms = __ldcg(sl + kGroup * kDim + row);
                    const float wgt = (Mx == -INFINITY) ? 0.f : ex2(ms - Mx);
                    Lx += wgt * __ldcg(sl + kGroup * kDim + kGroup + row);
                    const float4 a = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0));
                    const float4 b = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0 + 4));
                    acc[0] += wgt * a.x; acc[1] += wgt * a.y; acc[2] += wgt * a.z; acc[3] += wgt * a.w;
                    acc[4] += wgt * b.x; acc[5] += wgt * b.y; acc[6] += wgt * b.z; acc[7] += wgt * b.w;
                }
                const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
                uint4 packed;
                packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
                packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
                packed.z = pack_bf16(acc[4] * inv, acc[5] * inv);
                packed.w = pack_bf16(acc[6] * inv, acc[7] * inv);
                *reinterpret_cast<uint4 *>(p.out + (hbase + row) * kDim + d0) = packed;
                if (d0 == 0)
                    p.lse[hbase + row] =
                        (Mx == -INFINITY) ? -INFINITY : (Mx + log2f(Lx)) * 0.69314718055994531f;
            }
            if (threadIdx.x == 0)
                p.counters[u] = 0; // ready for the next call
        }
        csync(); // s_flag and cbuf are reused by the next unit
    };

    for (int l = 0; l < ntasks && ok; ++l) {
        const int zk = 2 * l, zv = 2 * l + 1;
        const int sk = zk % STAGES, sv = zv % STAGES;
        if (!mbar_wait_or_abort(smem_u32(&full[sk]), (zk / STAGES) & 1, abort_flag)) {
            ok = false;
            break;
        }
        const int4 e = entry(l); // written before the producer armed full[sk]
        const int u = e.w * p.T + e.z;
        if (u != cur_unit) {
            if (cur_unit >= 0) {
                finalize(cur_t, cur_g);
                if (!ok)
                    break;
            }
            cur_unit = u;
            cur_t = e.z;
            cur_g = e.w;
            reset_state();
            const int qb = cons_units % kQBufs;
            if (!mbar_wait_or_abort(smem_u32(&qfull[qb]), (cons_units / kQBufs) & 1, abort_flag)) {
                ok = false;
                break;
            }
            load_q(qb);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&qempty[qb]));
            ++cons_units;
        }
        const int nvis = e.y; // visible tokens of this page
        const uint32_t tileK = smem_u32(ring + (size_t)sk * C::kTileBytes);
        const uint32_t tileV = smem_u32(ring + (size_t)sv * C::kTileBytes);
        const bool live = e.x >= 0;

        // ---- S = Q K^T over this warp's kTPW tokens: kNT n-tiles of 8 tokens ----
        float s[kNT][4];
#pragma unroll
        for (int n = 0; n < kNT; ++n)
            s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        if (live) {
            if (!FP8) {
#pragma unroll
                for (int n2 = 0; n2 < kNT / 2; ++n2) {
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
                for (int n2 = 0; n2 < kNT / 2; ++n2) {
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
        }
        // the K tile is no longer read: hand its stage back to the producer
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty[sk]));

        uint32_t pa[kKK][4];
        if (live) {
            // ---- scale, causal mask, online softmax (base 2) ----
            const bool need_mask = tb + kTPW > nvis;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v = s[n][k] * p.scale_log2;
                    if (need_mask && tb + 8 * n + 2 * q4 + (k & 1) >= nvis)
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
#pragma unroll
            for (int n = 0; n < kNT; ++n) {
                const float p0 = ex2(s[n][0] - ref[0]), p1 = ex2(s[n][1] - ref[0]);
                const float p2 = ex2(s[n][2] - ref[1]), p3 = ex2(s[n][3] - ref[1]);
                l_run[0] += p0 + p1;
                l_run[1] += p2 + p3;
                // A fragment of P for k-step n/2: n-tile 2kk -> regs 0,1; 2kk+1 -> regs 2,3
                const int kk = n >> 1, hi = (n & 1) * 2;
                pa[kk][hi + 0] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
                pa[kk][hi + 1] = FP8 ? pack_f16(p2, p3) : pack_bf16(p2, p3);
            }
        }

        if (!mbar_wait_or_abort(smem_u32(&full[sv]), (zv / STAGES) & 1, abort_flag)) {
            ok = false;
            break;
        }
        if (live) {
            // ---- O += P V over this warp's kTPW tokens ----
            if (!FP8) {
#pragma unroll
                for (int kk = 0; kk < kKK; ++kk) {
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
                for (int kk = 0; kk < kKK; ++kk) {
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
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&empty[sv]));
    }
    if (ok && cur_unit >= 0)
        finalize(cur_t, cur_g);
    if (!ok) {
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
    }
}

// ===========================================================================
// bf16 KV: tcgen05 UMMA with TMEM accumulators
// ===========================================================================
//
// Per page (task) of unit (t, g):
//   S^T[128 tok][16 heads] = K[128 tok][128 dim] . Q^T          (M=128, N=16, K=128)
//   O^T[128 dim][16 heads] = V^T[128 dim][128 tok] . P^T        (M=128, N=16, K=128)
// both issued by one thread as tcgen05.mma.kind::f16 (8 instructions of K=16
// each), fp32 accumulators in TMEM (double-buffered: S at columns 0/16, O at
// 32/48).  Operands: K tile and the unit's Q rows are K-major with the TMA's
// 128-byte swizzle; the V tile, as loaded, is the MN-major form of V^T; P^T is
// written by the softmax warps in the K-major 128-byte-swizzled form.
// Warps: 0 = TMA producer + task table, 1 = MMA issuer + TMEM owner,
// 2..5 = softmax (thread = one TMEM lane: a token for S^T, a dimension for
// O^T).  The softmax warps exchange per-head page maxima through shared memory,
// keep the running max / denominator per head, and fold each page's O^T into
// 16 registers (one per head) once the next page's P^T is written.

constexpr int kUSmxWarps = 8;              // softmax warps: two per TMEM lane quarter
constexpr int kUCvtWarps = 4;              // FP8 only: E4M3 -> f16 converter warps
constexpr int kUSoftmax = 32 * kUSmxWarps; // softmax threads
template <bool FP8>
constexpr int kUThreadsT = 32 * (2 + kUSmxWarps + (FP8 ? kUCvtWarps : 0)); // producer, MMA, softmax[, converters]
constexpr int kUHeads = 8;                 // heads per softmax thread (half of the group)
constexpr int kUTmemCols = 64;             // S[2] + O[2], 16 columns each
constexpr int kUTile = 32768;              // bf16 K or V tile of one (page, KV head)
constexpr int kUQTile = 4096;              // 16 query rows of one unit, two 64-dim boxes
constexpr int kUPTile = 4096;              // P^T of one page: [16 heads][128 tokens] bf16

struct USmem {
    size_t ring, stage, qbuf, pbuf, bars, table, xbuf, lbuf, misc, qt, total;
};

// bf16: the ring holds the MMA operands.  FP8: the ring holds E4M3 tiles
// (16 KiB) and one f16 staging tile each for K and V feeds the MMA.
__host__ __device__ inline USmem umma_layout(int T, int stages, bool fp8)
{
    USmem L{};
    size_t off = 0;
    L.ring = off;                          // 1024-aligned tiles
    off += (size_t)stages * (fp8 ? kUTile / 2 : kUTile);
    L.stage = off = align_to(off, 1024);   // FP8: K and V f16 tiles
    off += fp8 ? 2 * kUTile : 0;
    L.qbuf = off = align_to(off, 1024);    // [2] query tiles (swizzle atoms: 1024-aligned)
    off += 2 * kUQTile;
    L.pbuf = off = align_to(off, 1024);    // [2] P^T tiles
    off += 2 * kUPTile;
    // full[S], empty[S], qfull[2], qempty[2], s_full[2], s_free[2], p_full[2],
    // p_free[2], o_full[2], o_free[2], softmax sync, done, then FP8 only:
    // kst_full, kst_empty, vst_full, vst_empty, qconv[2]
    L.bars = off = align_to(off, 8);
    off += (size_t)(2 * stages + 16 + 2 + 6) * 8;
    L.table = off = align_to(off, 16);     // [2][kWin] int4
    off += (size_t)2 * kWin * 16;
    L.xbuf = off = align_to(off, 16);      // [2][4 quarters][16] page maxima
    off += 2 * 4 * 16 * 4;
    L.lbuf = off = align_to(off, 16);      // [4 quarters][16] denominators
    off += 4 * 16 * 4;
    L.misc = off = align_to(off, 16);      // tmem base, flags
    off += 16;
    L.qt = off = align_to(off, 16);        // [T + 1]
    off += (size_t)(T + 1) * 4;
    L.total = align_to(off, 16) + 1024;
    return L;
}

// 8 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}

template <bool FP8, int STAGES>
__global__ void __launch_bounds__(kUThreadsT<FP8>, 1)
    sparse_decode_umma_kernel(const __grid_constant__ CUtensorMap kv_map,
                              const __grid_constant__ CUtensorMap q_map, const DecodeParams p)
{
    constexpr int kRaw = FP8 ? kUTile / 2 : kUTile; // bytes of one ring tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const USmem lay = umma_layout(p.T, STAGES, FP8);
    uint8_t *ring = base + lay.ring;
    uint8_t *kst = base + lay.stage;        // FP8: f16 K tile
    uint8_t *vst = kst + kUTile;            // FP8: f16 V tile
    uint8_t *qbuf = base + lay.qbuf;
    uint8_t *pbuf = base + lay.pbuf;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + lay.bars);
    uint64_t *empty = full + STAGES;
    uint64_t *qfull = empty + STAGES;
    uint64_t *qempty = qfull + 2;
    uint64_t *s_full = qempty + 2;
    uint64_t *s_free = s_full + 2;
    uint64_t *p_full = s_free + 2;
    uint64_t *p_free = p_full + 2;
    uint64_t *o_full = p_free + 2;
    uint64_t *o_free = o_full + 2;
    uint64_t *smx_bar = o_free + 2;    // softmax-warps barrier (kUSoftmax arrivals)
    uint64_t *done_bar = smx_bar + 1;  // softmax warps finished with TMEM (kUSmxWarps arrivals)
    uint64_t *kst_full = done_bar + 1; // FP8: staging K converted (kUCvtWarps)
    uint64_t *kst_empty = kst_full + 1; // FP8: staging K read by the MMA (commit)
    uint64_t *vst_full = kst_empty + 1;
    uint64_t *vst_empty = vst_full + 1;
    uint64_t *qconv = vst_empty + 1;   // FP8: [2] query tile widened to f16 (kUCvtWarps)
    int4 *table = reinterpret_cast<int4 *>(base + lay.table);
    float *xbuf = reinterpret_cast<float *>(base + lay.xbuf);
    float *lbuf = reinterpret_cast<float *>(base + lay.lbuf);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + lay.misc);
    int *s_flag = reinterpret_cast<int *>(base + lay.misc) + 1; // [0] last arrival, [1] abort
    int *qt = reinterpret_cast<int *>(base + lay.qt);
    volatile int *abort_flag = s_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kv_map);
        prefetch_tensormap(&q_map);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), FP8 ? kUCvtWarps : 1);
        }
        mbar_init(smem_u32(kst_full), kUCvtWarps);
        mbar_init(smem_u32(kst_empty), 1);
        mbar_init(smem_u32(vst_full), kUCvtWarps);
        mbar_init(smem_u32(vst_empty), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&qconv[b]), kUCvtWarps);
            mbar_init(smem_u32(&qfull[b]), 1);
            mbar_init(smem_u32(&qempty[b]), 1);
            mbar_init(smem_u32(&s_full[b]), 1);
            mbar_init(smem_u32(&s_free[b]), kUSmxWarps);
            mbar_init(smem_u32(&p_full[b]), kUSmxWarps);
            mbar_init(smem_u32(&p_free[b]), 1);
            mbar_init(smem_u32(&o_full[b]), 1);
            mbar_init(smem_u32(&o_free[b]), kUSmxWarps);
        }
        mbar_init(smem_u32(smx_bar), kUSoftmax);
        mbar_init(smem_u32(done_bar), kUSmxWarps);
        s_flag[0] = 0;
        s_flag[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(smem_u32(tmem_slot), kUTmemCols);
    build_token_prefix(p, qt);
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = *tmem_slot;

    const long long P = (long long)p.Hkv * qt[p.T];
    const int G = gridDim.x, c = blockIdx.x;
    const long long x_begin = (long long)c * P / G, x_end = (long long)(c + 1) * P / G;
    const int ntasks = (int)(x_end - x_begin);

    grid_dependency_wait(); // `selected` comes from the previous kernel of the step

    auto entry = [&](int l) -> int4 { return table[((l / kWin) & 1) * kWin + (l % kWin)]; };
    auto unit_of = [&](const int4 &e) { return e.w * p.T + e.z; };
    auto fill_window = [&](int w) { // producer warp
        const int l0 = w * kWin;
        int4 *dst = table + (w & 1) * kWin;
        for (int i = lane; i < kWin && l0 + i < ntasks; i += 32)
            dst[i] = make_entry(p, x_begin + l0 + i, qt);
        __syncwarp();
    };
    // the first two table windows, visible to every warp before anything starts
    if (warp == 0) {
        if (ntasks > 0)
            fill_window(0);
        if (ntasks > kWin)
            fill_window(1);
    }
    __syncthreads();

    if (warp == 0) {
        // =================== producer ===================
        constexpr int kAhead = STAGES / 2;
        int issued = 0, q_issued = 0, prod_units = 0, prod_last = -1;
        bool ok = true;
        for (int l = 0; l < ntasks && ok; ++l) {
            const int zk = 2 * l;
            if (lane == 0 && zk >= STAGES)
                ok = mbar_wait_or_abort(smem_u32(&empty[zk % STAGES]), ((zk / STAGES) - 1) & 1,
                                        abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            // The softmax warps trail the MMA warp by up to two tasks and the MMA
            // warp trails this one by up to kAhead (kAhead + 1 with the FP8
            // converters between them): only kAhead + 3 (+ 1) tasks into a
            // window has every reader left the window before it.
            if (l % kWin == kAhead + 3 + (FP8 ? 1 : 0) && l >= kWin && (l / kWin + 1) * kWin < ntasks)
                fill_window(l / kWin + 1);
            if (lane == 0) {
                const int4 e = entry(l);
                const int u = unit_of(e);
                if (u != prod_last) {
                    prod_last = u;
                    const int qb = prod_units & 1;
                    if (prod_units >= 2)
                        ok = mbar_wait_or_abort(smem_u32(&qempty[qb]), ((prod_units >> 1) - 1) & 1,
                                                abort_flag);
                    if (ok) {
                        const uint32_t qbar = smem_u32(&qfull[qb]);
                        const uint32_t dst = smem_u32(qbuf + qb * kUQTile);
                        const int row = (e.z * p.Hkv + e.w) * kGroup;
                        mbar_arrive_expect_tx(qbar, kUQTile);
                        tma_load_2d(dst, &q_map, 0, row, qbar);
                        tma_load_2d(dst + kUQTile / 2, &q_map, 64, row, qbar);
                        q_issued = prod_units + 1;
                    }
                    ++prod_units;
                }
                for (int kv = 0; kv < 2 && ok; ++kv) {
                    const int z = zk + kv;
                    const int st = z % STAGES;
                    if (kv == 1 && z >= STAGES)
                        ok = mbar_wait_or_abort(smem_u32(&empty[st]), ((z / STAGES) - 1) & 1,
                                                abort_flag);
                    if (!ok)
                        break;
                    const uint32_t bar = smem_u32(&full[st]);
                    issued = z + 1;
                    if (e.x < 0) {
                        mbar_arrive(bar); // no data: consumers skip the task
                        continue;
                    }
                    const uint32_t dst = smem_u32(ring + (size_t)st * kRaw);
                    const int row = e.x + kv * p.Hkv * kPage;
                    mbar_arrive_expect_tx(bar, kRaw);
                    tma_load_2d(dst, &kv_map, 0, row, bar);
                    if (!FP8)
                        tma_load_2d(dst + kUTile / 2, &kv_map, 64, row, bar);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        if (!ok && lane == 0) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
            for (int z = issued - STAGES < 0 ? 0 : issued - STAGES; z < issued; ++z)
                (void)mbar_wait_bounded(smem_u32(&full[z % STAGES]), (z / STAGES) & 1);
            for (int u = q_issued - 2 < 0 ? 0 : q_issued - 2; u < q_issued; ++u)
                (void)mbar_wait_bounded(smem_u32(&qfull[u & 1]), (u >> 1) & 1);
        }
        return;
    }

    if (warp == 1) {
        // =================== MMA issuer (lane 0) ===================
        // S^T(l + 1) is issued before P^T(l) is awaited, so the tensor core
        // works on the next page while the softmax warps work on this one.
        // bf16 operands, or f16 for FP8 KV (widened E4M3, f16 Q and P)
        constexpr uint32_t kF16 = FP8 ? ~((7u << 7) | (7u << 10)) : ~0u;
        constexpr uint32_t kIdescS = umma_idesc_bf16(128, 16, 0, 0) & kF16; // K and Q^T both K-major
        constexpr uint32_t kIdescO = umma_idesc_bf16(128, 16, 1, 0) & kF16; // V^T MN-major, P^T K-major
        bool ok = true;
        if (lane == 0) {
            int s_units = 0, s_unit = -1;
            auto issue_s = [&](int l) -> bool {
                const int zk = 2 * l, b = l & 1;
                if (!FP8 && !mbar_wait_or_abort(smem_u32(&full[zk % STAGES]), (zk / STAGES) & 1, abort_flag))
                    return false;
                if (FP8 && !mbar_wait_or_abort(smem_u32(kst_full), l & 1, abort_flag))
                    return false;
                const int4 e = entry(l);
                const int u = unit_of(e);
                if (u != s_unit) {
                    uint64_t *qb_bar = FP8 ? qconv : qfull;
                    if (!mbar_wait_or_abort(smem_u32(&qb_bar[s_units & 1]), (s_units >> 1) & 1, abort_flag))
                        return false;
                    s_unit = u;
                    ++s_units;
                }
                const int qb = (s_units - 1) & 1;
                if (l >= 2 && !mbar_wait_or_abort(smem_u32(&s_free[b]), ((l >> 1) - 1) & 1, abort_flag))
                    return false;
                tcgen05_after_sync();
                if (e.x >= 0) {
                    const uint32_t tileK = FP8 ? smem_u32(kst) : smem_u32(ring + (size_t)(zk % STAGES) * kRaw);
                    const uint32_t qtile = smem_u32(qbuf + qb * kUQTile);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t a = umma_desc_sw128(tileK + (ks >> 2) * (kUTile / 2) + (ks & 3) * 32, 16, 1024);
                        const uint64_t bq = umma_desc_sw128(qtile + (ks >> 2) * (kUQTile / 2) + (ks & 3) * 32, 16, 1024);
                        umma_bf16(tmem + 16 * b, a, bq, kIdescS, ks > 0);
                    }
                }
                umma_commit(smem_u32(&s_full[b]));
                umma_commit(FP8 ? smem_u32(kst_empty) : smem_u32(&empty[zk % STAGES])); // K tile read
                // last task of its unit: the query tile can be replaced
                if (l + 1 == ntasks || unit_of(entry(l + 1)) != u)
                    umma_commit(smem_u32(&qempty[qb]));
                return true;
            };
            auto issue_pv = [&](int l) -> bool {
                const int zv = 2 * l + 1, b = l & 1;
                if (!FP8 && !mbar_wait_or_abort(smem_u32(&full[zv % STAGES]), (zv / STAGES) & 1, abort_flag))
                    return false;
                if (FP8 && !mbar_wait_or_abort(smem_u32(vst_full), l & 1, abort_flag))
                    return false;
                if (!mbar_wait_or_abort(smem_u32(&p_full[b]), (l >> 1) & 1, abort_flag))
                    return false;
                if (l >= 2 && !mbar_wait_or_abort(smem_u32(&o_free[b]), ((l >> 1) - 1) & 1, abort_flag))
                    return false;
                tcgen05_after_sync();
                if (entry(l).x >= 0) {
                    const uint32_t tileV = FP8 ? smem_u32(vst) : smem_u32(ring + (size_t)(zv % STAGES) * kRaw);
                    const uint32_t ptile = smem_u32(pbuf + b * kUPTile);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        // V^T, MN-major: 16 tokens per k-step = 16 rows of 128 bytes;
                        // the two 64-dim halves of a row are 16 KiB apart (LBO)
                        const uint64_t a = umma_desc_sw128(tileV + ks * 2048, kUTile / 2, 1024);
                        const uint64_t bp = umma_desc_sw128(ptile + (ks >> 2) * (kUPTile / 2) + (ks & 3) * 32, 16, 1024);
                        umma_bf16(tmem + 32 + 16 * b, a, bp, kIdescO, ks > 0);
                    }
                }
                umma_commit(smem_u32(&o_full[b]));
                umma_commit(smem_u32(&p_free[b]));
                umma_commit(FP8 ? smem_u32(vst_empty) : smem_u32(&empty[zv % STAGES])); // V tile read
                return true;
            };
            if (ntasks > 0)
                ok = issue_s(0);
            for (int l = 0; l < ntasks && ok; ++l) {
                if (l + 1 < ntasks)
                    ok = issue_s(l + 1);
                if (ok)
                    ok = issue_pv(l);
            }
            if (!ok) {
                set_error(p.err, kErrTimeout);
                *abort_flag = 1;
            }
        }
        __syncwarp();
        // free TMEM once the softmax warps are done with it (they always arrive,
        // also after an abort; the wait is bounded)
        if (lane == 0)
            (void)mbar_wait_bounded(smem_u32(done_bar), 0);
        __syncwarp();
        tcgen05_after_sync();
        tmem_dealloc(tmem, kUTmemCols);
        return;
    }

    if (FP8 && warp >= 2 + kUSmxWarps) {
        // =================== converter warps (FP8) ===================
        // E4M3 K / V tiles from the ring into the f16 staging tiles, in the
        // two-64-dim-box, 128-byte-swizzled layout the MMA descriptors read;
        // the query tile of each new unit is widened from bf16 to f16 in place.
        const int ct = threadIdx.x - 32 * (2 + kUSmxWarps); // 0..127
        bool ok = true;
        int units = 0, cur = -1;
        auto convert = [&](const uint8_t *raw, uint8_t *dst) {
#pragma unroll 2
            for (int item = ct; item < kPage * 8; item += 32 * kUCvtWarps) {
                const int r = item >> 3, c = item & 7; // row, 16-byte chunk of 16 E4M3 dims
                const uint4 w = *reinterpret_cast<const uint4 *>(raw + r * 128 + ((c ^ (r & 7)) << 4));
                uint4 lo, hi;
                lo.x = e4m3x2_to_f16x2(w.x & 0xFFFFu);
                lo.y = e4m3x2_to_f16x2(w.x >> 16);
                lo.z = e4m3x2_to_f16x2(w.y & 0xFFFFu);
                lo.w = e4m3x2_to_f16x2(w.y >> 16);
                hi.x = e4m3x2_to_f16x2(w.z & 0xFFFFu);
                hi.y = e4m3x2_to_f16x2(w.z >> 16);
                hi.z = e4m3x2_to_f16x2(w.w & 0xFFFFu);
                hi.w = e4m3x2_to_f16x2(w.w >> 16);
                const int h = c >> 2, c0 = 2 * (c & 3);  // box (64 dims), first 8-dim chunk
                uint8_t *row = dst + h * (kUTile / 2) + r * 128;
                *reinterpret_cast<uint4 *>(row + ((c0 ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(row + (((c0 + 1) ^ (r & 7)) << 4)) = hi;
            }
            fence_async_smem();
        };
        for (int l = 0; l < ntasks && ok; ++l) {
            const int zk = 2 * l, zv = zk + 1;
            ok = mbar_wait_or_abort(smem_u32(&full[zk % STAGES]), (zk / STAGES) & 1, abort_flag);
            if (!ok)
                break;
            const int4 e = entry(l);
            const int u = unit_of(e);
            if (u != cur) {
                const int qb = units & 1;
                ok = mbar_wait_or_abort(smem_u32(&qfull[qb]), (units >> 1) & 1, abort_flag);
                if (!ok)
                    break;
                uint8_t *q = qbuf + qb * kUQTile;
                for (int i = ct; i < kUQTile / 16; i += 32 * kUCvtWarps) {
                    uint4 v = reinterpret_cast<uint4 *>(q)[i];
                    v.x = bf16x2_to_f16x2(v.x);
                    v.y = bf16x2_to_f16x2(v.y);
                    v.z = bf16x2_to_f16x2(v.z);
                    v.w = bf16x2_to_f16x2(v.w);
                    reinterpret_cast<uint4 *>(q)[i] = v;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(smem_u32(&qconv[qb]));
                cur = u;
                ++units;
            }
            if (l >= 1)
                ok = mbar_wait_or_abort(smem_u32(kst_empty), (l - 1) & 1, abort_flag);
            if (!ok)
                break;
            if (e.x >= 0)
                convert(ring + (size_t)(zk % STAGES) * kRaw, kst);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(kst_full));
                mbar_arrive(smem_u32(&empty[zk % STAGES]));
            }
            ok = mbar_wait_or_abort(smem_u32(&full[zv % STAGES]), (zv / STAGES) & 1, abort_flag);
            if (ok && l >= 1)
                ok = mbar_wait_or_abort(smem_u32(vst_empty), (l - 1) & 1, abort_flag);
            if (!ok)
                break;
            if (e.x >= 0)
                convert(ring + (size_t)(zv % STAGES) * kRaw, vst);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(vst_full));
                mbar_arrive(smem_u32(&empty[zv % STAGES]));
            }
        }
        if (!ok) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
        }
        return;
    }

    // =================== softmax warps 2..9 ===================
    // Warps w and w + 4 share TMEM lanes 32*(w & 3) .. +31 and split the 16
    // heads into halves: each thread holds one token (of S^T) or one dimension
    // (of O^T) for kUHeads heads.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;      // heads 8*half .. 8*half + 7
    const int h0 = kUHeads * half;
    const int idx = 32 * quarter + lane;   // token of S^T / dimension of O^T
    const int sidx = threadIdx.x - 64;     // 0 .. kUSoftmax - 1
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + h0;
    int sync_phase = 0;
    bool ok = true;
    auto ssync = [&]() {
        mbar_arrive(smem_u32(smx_bar));
        if (!mbar_wait_or_abort(smem_u32(smx_bar), sync_phase & 1, abort_flag))
            ok = false;
        ++sync_phase;
    };

    float o[kUHeads], lsum[kUHeads], m_run[kUHeads], alpha_prev[kUHeads];
    bool pending = false; // a page's O^T waits to be folded in
    int cur_unit = -1, cur_t = 0, cur_g = 0;

    auto reset = [&]() {
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            o[h] = 0.f;
            lsum[h] = 0.f;
            m_run[h] = -INFINITY;
            alpha_prev[h] = 1.f;
        }
    };

    // fold the previous page's O^T (thread = dimension) into o[]
    auto fold = [&](int l_prev) {
        const int b = l_prev & 1;
        if (!mbar_wait_or_abort(smem_u32(&o_full[b]), (l_prev >> 1) & 1, abort_flag)) {
            ok = false;
            return;
        }
        tcgen05_after_sync();
        if (pending) {
            float v[kUHeads];
            tmem_ld8(lane_base + 32 + 16 * b, v);
#pragma unroll
            for (int h = 0; h < kUHeads; ++h)
                o[h] = o[h] * alpha_prev[h] + v[h];
        }
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&o_free[b]));
        pending = false;
    };

    auto finalize = [&](int t, int g) {
        // denominators: reduce lsum over the 128 token lanes
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            float v = lsum[h];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0)
                lbuf[quarter * 16 + h0 + h] = v;
        }
        ssync();
        float L[kUHeads];
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            L[h] = lbuf[h0 + h] + lbuf[16 + h0 + h] + lbuf[32 + h0 + h] + lbuf[48 + h0 + h];
        ssync(); // lbuf is reused by the next unit
        const long long Pt = qt[p.T];
        const long long u_first = (long long)g * Pt + qt[t];
        const int n_u = qt[t + 1] - qt[t];
        const int c_first = owner_of(u_first, P, G);
        const int c_last = owner_of(u_first + n_u - 1, P, G);
        const int u = g * p.T + t;
        const bool whole = c_first == c_last;
        const size_t hbase = (size_t)t * p.Hkv * kGroup + (size_t)g * kGroup + h0;
        float *slot = p.partial + (size_t)(c + u) * kPartialFloats;
        float Mi = -INFINITY, Li = 0.f; // head h0 + idx (idx < kUHeads)
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            if (h == idx) {
                Mi = m_run[h];
                Li = L[h];
            }
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            o[h] *= p.v_scale; // 1 for bf16 values
        if (whole) {
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                const float inv = L[h] > 0.f ? 1.f / L[h] : 0.f;
                p.out[(hbase + h) * kDim + idx] = (uint16_t)(pack_bf16(o[h] * inv, 0.f) & 0xFFFFu);
            }
            if (idx < kUHeads)
                p.lse[hbase + idx] = (Mi == -INFINITY) ? -INFINITY : (Mi + log2f(Li)) * 0.69314718055994531f;
            return;
        }
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            slot[(h0 + h) * kDim + idx] = o[h];
        if (idx < kUHeads) {
            slot[kGroup * kDim + h0 + idx] = Mi;
            slot[kGroup * kDim + kGroup + h0 + idx] = Li;
        }
        __threadfence(); // publish this CTA's slot before counting in
        ssync();
        if (sidx == 0) {
            int arrivals = 0;
            for (int cc = c_first; cc <= c_last; ++cc)
                arrivals += !range_empty(cc, P, G);
            const int before = atomicAdd(&p.counters[u], 1);
            s_flag[0] = before == arrivals - 1;
        }
        ssync();
        if (s_flag[0]) {
            __threadfence();
            const float *sbase = p.partial + (size_t)(c_first + u) * kPartialFloats;
            const int nslots = c_last - c_first + 1;
            const size_t obase = (size_t)t * p.Hkv * kGroup + (size_t)g * kGroup;
            for (int e = sidx; e < kGroup * kDim / 8; e += kUSoftmax) {
                const int row = e >> 4, d0 = (e & 15) * 8;
                float Mx = -INFINITY;
                for (int s = 0; s < nslots; ++s)
                    if (!range_empty(c_first + s, P, G))
                        Mx = fmaxf(Mx, __ldcg(sbase + (size_t)s * kPartialFloats + kGroup * kDim + row));
                float Lx = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                for (int s = 0; s < nslots; ++s) {
                    if (range_empty(c_first + s, P, G))
                        continue;
                    const float *sl = sbase + (size_t)s * kPartialFloats;
                    const float ms = __ldcg(sl + kGroup * kDim + row);
                    const float wgt = (Mx == -INFINITY) ? 0.f : ex2(ms - Mx);
                    Lx += wgt * __ldcg(sl + kGroup * kDim + kGroup + row);
                    const float4 a = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0));
                    const float4 bb = __ldcg(reinterpret_cast<const float4 *>(sl + row * kDim + d0 + 4));
                    acc[0] += wgt * a.x; acc[1] += wgt * a.y; acc[2] += wgt * a.z; acc[3] += wgt * a.w;
                    acc[4] += wgt * bb.x; acc[5] += wgt * bb.y; acc[6] += wgt * bb.z; acc[7] += wgt * bb.w;
                }
                const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
                uint4 packed;
                packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
                packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
                packed.z = pack_bf16(acc[4] * inv, acc[5] * inv);
                packed.w = pack_bf16(acc[6] * inv, acc[7] * inv);
                *reinterpret_cast<uint4 *>(p.out + (obase + row) * kDim + d0) = packed;
                if (d0 == 0)
                    p.lse[obase + row] = (Mx == -INFINITY) ? -INFINITY : (Mx + log2f(Lx)) * 0.69314718055994531f;
            }
            if (sidx == 0)
                p.counters[u] = 0; // ready for the next call
        }
        ssync(); // s_flag is reused by the next unit
    };

    int l_last = -1;
    for (int l = 0; l < ntasks && ok; ++l) {
        const int b = l & 1;
        if (!mbar_wait_or_abort(smem_u32(&s_full[b]), (l >> 1) & 1, abort_flag)) {
            ok = false;
            break;
        }
        tcgen05_after_sync();
        const int4 e = entry(l);
        const int u = unit_of(e);
        const bool live = e.x >= 0;
        float sv[kUHeads];
        if (live)
            tmem_ld8(lane_base + 16 * b, sv);
        tcgen05_before_sync();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&s_free[b]));

        if (u != cur_unit) {
            if (cur_unit >= 0) {
                if (l_last >= 0)
                    fold(l_last);
                if (!ok)
                    break;
                finalize(cur_t, cur_g);
                if (!ok)
                    break;
            }
            cur_unit = u;
            cur_t = e.z;
            cur_g = e.w;
            reset();
            l_last = -1;
        }

        // page maxima per head (log2 domain) across the 128 tokens
        const bool visible = live && idx < e.y;
        float wmax[kUHeads];
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            sv[h] = visible ? sv[h] * p.scale_log2 : -INFINITY;
            wmax[h] = warp_max_f32(sv[h]);
        }
        if (lane == 0) {
            float4 *xw = reinterpret_cast<float4 *>(xbuf + (b * 4 + quarter) * 16 + h0);
            xw[0] = make_float4(wmax[0], wmax[1], wmax[2], wmax[3]);
            xw[1] = make_float4(wmax[4], wmax[5], wmax[6], wmax[7]);
        }
        ssync();
        float alpha[kUHeads], pv[kUHeads];
#pragma unroll
        for (int h4 = 0; h4 < kUHeads / 4; ++h4) {
            float4 a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                a[q] = reinterpret_cast<const float4 *>(xbuf + (b * 4 + q) * 16 + h0)[h4];
            const float pm[4] = {fmaxf(fmaxf(a[0].x, a[1].x), fmaxf(a[2].x, a[3].x)),
                                 fmaxf(fmaxf(a[0].y, a[1].y), fmaxf(a[2].y, a[3].y)),
                                 fmaxf(fmaxf(a[0].z, a[1].z), fmaxf(a[2].z, a[3].z)),
                                 fmaxf(fmaxf(a[0].w, a[1].w), fmaxf(a[2].w, a[3].w))};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int h = 4 * h4 + k;
                const float m_new = fmaxf(m_run[h], pm[k]);
                const float ref = (m_new == -INFINITY) ? 0.f : m_new;
                alpha[h] = ex2(m_run[h] - ref); // 0 when m_run is -inf
                m_run[h] = m_new;
                pv[h] = ex2(sv[h] - ref);
                lsum[h] = lsum[h] * alpha[h] + pv[h];
            }
        }
        // P^T[h][token idx] into the K-major, 128-byte-swizzled B tile
        if (l >= 2 && !mbar_wait_or_abort(smem_u32(&p_free[b]), ((l >> 1) - 1) & 1, abort_flag)) {
            ok = false;
            break;
        }
        if (live) {
            uint8_t *pt = pbuf + b * kUPTile + (idx >> 6) * (kUPTile / 2);
            const int col = idx & 63;
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                const int hh = h0 + h;
                const uint32_t off = hh * 128 + ((((col >> 3) ^ (hh & 7))) << 4) + (col & 7) * 2;
                const uint32_t pk = FP8 ? pack_f16(pv[h], 0.f) : pack_bf16(pv[h], 0.f);
                *reinterpret_cast<uint16_t *>(pt + off) = (uint16_t)(pk & 0xFFFFu);
            }
            fence_async_smem();
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&p_full[b]));

        // fold the previous page of this unit, then this page becomes pending
        if (l_last >= 0) {
            fold(l_last);
            if (!ok)
                break;
        }
        // a page with no data contributes p = 0 and leaves the state unchanged
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            alpha_prev[h] = live ? alpha[h] : 1.f;
        pending = live;
        l_last = l;
    }
    if (ok && cur_unit >= 0) {
        if (l_last >= 0)
            fold(l_last);
        if (ok)
            finalize(cur_t, cur_g);
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

template <bool FP8, int STAGES>
size_t decode_smem_bytes(int T)
{
    return decode_layout(T, STAGES, Cfg<FP8, STAGES>::kTileBytes).total;
}

template <bool FP8, int STAGES>
cudaError_t launch_decode_t(const DecodeParams &p, const CUtensorMap &map, int ctas,
                            cudaStream_t stream, bool pdl)
{
    const size_t smem = decode_smem_bytes<FP8, STAGES>(p.T);
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_kernel<FP8, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = launch_kernel(sparse_decode_kernel<FP8, STAGES>, dim3(ctas), dim3(kDecThreads), smem,
                      stream, pdl, map, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

// The deepest ring that fits next to the token prefix (T + 1 ints).
template <bool FP8>
cudaError_t launch_decode_fit(const DecodeParams &p, const CUtensorMap &map, int ctas,
                              cudaStream_t stream, bool pdl)
{
    constexpr int kDeep = FP8 ? 12 : 6, kShallow = FP8 ? 8 : 4;
    if (decode_smem_bytes<FP8, kDeep>(p.T) <= (size_t)kMaxSmem)
        return launch_decode_t<FP8, kDeep>(p, map, ctas, stream, pdl);
    return launch_decode_t<FP8, kShallow>(p, map, ctas, stream, pdl);
}

// Query rows [T * Hq][128] bf16, boxes of 64 dims x 16 rows, 128-byte swizzle.
bool encode_q_map(CUtensorMap *map, const void *q, int T, int Hkv)
{
    EncodeFn enc = get_encode();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)T * Hkv * kGroup};
    const cuuint64_t strides[1] = {(cuuint64_t)kDim * 2};
    const cuuint32_t box[2] = {64u, (cuuint32_t)kGroup};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, int STAGES>
cudaError_t launch_umma_t(const DecodeParams &p, const CUtensorMap &kv, const CUtensorMap &qm,
                          int ctas, cudaStream_t stream, bool pdl)
{
    const size_t smem = umma_layout(p.T, STAGES, FP8).total;
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_umma_kernel<FP8, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = launch_kernel(sparse_decode_umma_kernel<FP8, STAGES>, dim3(ctas), dim3(kUThreadsT<FP8>), smem,
                      stream, pdl, kv, qm, p);
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
    CUtensorMap qmap;
    if (!encode_q_map(&qmap, p.q, p.T, p.Hkv))
        return cudaErrorInvalidValue;
    if (kv_dtype == MSA_FP8_E4M3) {
        if (umma_layout(p.T, 8, true).total <= (size_t)kMaxSmem)
            return launch_umma_t<true, 8>(p, map, qmap, ctas, stream, pdl);
        return launch_umma_t<true, 4>(p, map, qmap, ctas, stream, pdl);
    }
    if (umma_layout(p.T, 6, false).total <= (size_t)kMaxSmem)
        return launch_umma_t<false, 6>(p, map, qmap, ctas, stream, pdl);
    return launch_umma_t<false, 4>(p, map, qmap, ctas, stream, pdl);
}

} // namespace msa
