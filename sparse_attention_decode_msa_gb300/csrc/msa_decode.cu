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
//   mbarrier (tile consumed), and the 16 query rows of each unit (4 KiB) by
//   TMA.  A K stage goes back to the producer as soon as S has read it.
// * Math.  On the tensor cores (tcgen05.mma, accumulators in TMEM), per page:
//   S^T = K Q^T and O^T = V^T P^T, M = 128 (tokens, then dimensions), N = 16
//   query heads; see the section before the kernel.  E4M3 keys and values are
//   MMA operands as loaded (kind::f8f6f4, the query and P as E4M3 hi + lo
//   pairs); NVFP4 keys and values are widened to f16 in shared memory by eight
//   converter warps (exact).  The tensor scales k_scale and v_scale are folded
//   into the logit scale and the output.  Logits are kept in base 2.
// * Every wait is bounded; a timeout sets MSA_ERR_TIMEOUT, raises a CTA abort
//   flag that ends every other wait, and the producer waits (bounded) for its
//   copies in flight before the CTA exits.
#include <cmath>
#include <cstring>

#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kWin = 128;                    // task-table window (two windows resident)
constexpr int kMaxSmem = 232448;             // dynamic shared memory limit per CTA

struct Task {
    int t, g, i;
};

// qt[t] = sum_{t' < t} n_t' (the tasks of one KV head before token t); qt[T] =
// total.  Called by every thread of the CTA: each loads the counts of a
// contiguous chunk of tokens (one round of global loads, however many
// tokens), then a CTA-wide exclusive scan of the chunk sums (tmp: one int per
// warp + 1); the caller synchronises before reading qt.
__device__ void build_token_prefix(const DecodeParams &p, int *qt, int *tmp)
{
    const int T = p.T, nth = blockDim.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = nth >> 5;
    const int per = (T + nth - 1) / nth;
    const int lo = min(T, (int)threadIdx.x * per), hi = min(T, lo + per);
    int sum = 0;
    for (int t = lo; t < hi; ++t) {
        const int r = t / p.nq, j = t - r * p.nq;
        const int sl = p.seq_lens[r];
        const long long nb = ((long long)sl + p.nq - 1 + kPage - 1) / kPage;
        int n = 0;
        if (sl >= 1 && nb <= p.maxB) {
            n = ceil_div(sl + j, kPage);
            n = n < p.k ? n : p.k;
        } else if (blockIdx.x == 0) {
            set_error(p.err, kErrSeqLen); // the token gets no tasks: its outputs are not written
        }
        qt[t] = n;
        sum += n;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < nwarps ? tmp[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o)
                wi += v;
        }
        if (lane < nwarps)
            tmp[lane] = wi - w;
        if (lane == nwarps - 1)
            tmp[nwarps] = wi;
    }
    __syncthreads();
    int run = tmp[warp] + incl - sum;
    for (int t = lo; t < hi; ++t) {
        const int n = qt[t];
        qt[t] = run;
        run += n;
    }
    if (threadIdx.x == 0)
        qt[T] = tmp[nwarps];
}

__device__ __forceinline__ Task task_of(long long x, const int *qt, int T)
{
    const int PT = qt[T];
    Task tk;
    tk.g = (int)((uint32_t)x / (uint32_t)PT); // x < P < 2^32 (see owner_of)
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
// range(c) = [floor(c P / G), floor((c+1) P / G)).  The host admits only calls
// with P (G + 1) < 2^32 (it bounds P by T Hkv k), so every product here fits
// 32 bits.  These run on the unit finalize's path, whose code runs cold once
// or twice per CTA: 64-bit divisions there (long software sequences) cost
// 1-2.3 us per launch, even as a branch not taken.
__device__ __forceinline__ int owner_of(long long x, long long P, int G)
{
    return (int)((((uint32_t)x + 1u) * (uint32_t)G + ((uint32_t)P - 1u)) / (uint32_t)P) - 1;
}

__device__ __forceinline__ bool range_empty(int c, long long P, int G)
{
    return (uint32_t)c * (uint32_t)P / (uint32_t)G == (uint32_t)(c + 1) * (uint32_t)P / (uint32_t)G;
}

// Table entry of task x: {K-tile row in the KV tensor map or -1, visible
// tokens of the page (1..128: the causal limit cuts the last block), t, g}.
__device__ int4 make_entry(const DecodeParams &p, long long x, const int *qt)
{
    const Task tk = task_of(x, qt, p.T);
    const int r = tk.t / p.nq, j = tk.t - r * p.nq;
    const int n_vis = ceil_div(p.seq_lens[r] + j, kPage);
    const int b = p.selected[((size_t)tk.t * p.Hs + (p.Hs > 1 ? tk.g : 0)) * p.k + tk.i];
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
// ===========================================================================
// tcgen05 UMMA with TMEM accumulators
// ===========================================================================
//
// Per page (task) of unit (t, g):
//   S^T[128 tok][16 heads] = K[128 tok][128 dim] . Q^T          (M=128, N=16, K=128)
//   O^T[128 dim][16 heads] = V^T[128 dim][128 tok] . P^T        (M=128, N=16, K=128)
// each issued by one thread as tcgen05.mma.kind::f16 (8 instructions of K=16
// each), fp32 accumulators in TMEM (S at columns 0/16/32/48, O at 64).
// Operands: K tile and the unit's Q rows are K-major with the TMA's
// 128-byte swizzle; the V tile, as loaded, is the MN-major form of V^T; P^T is
// written by the softmax warps in the K-major 128-byte-swizzled form.
// Warps: 0 = TMA producer + task table, 1 = S^T issuer + TMEM owner,
// 2 = O^T issuer, 3 = publisher, 4..11 = softmax (thread = one TMEM lane: a
// token for S^T, a dimension for O^T; two warps per lane quarter, 8 heads
// each), 12..19 = NVFP4 converters (NVFP4 K/V only).  The two MMA issuers are
// separate threads so that S^T of the next pages (four accumulators) is
// never queued behind P^T of this one.  The softmax warps exchange per-head
// page maxima through shared memory and keep a reference maximum and a
// denominator per head; O^T accumulates in TMEM over the pages of a unit and
// is rescaled there only when a head's maximum passes the reference by more
// than rescale_slack (so P stays below 2^slack).

constexpr int kUSmxWarps = 8;              // softmax warps: two per TMEM lane quarter
constexpr int kUCvtWarps = 8;              // NVFP4 only: e2m1 x E4M3 -> f16 converter warps
// KV formats of the kernel instances
constexpr int kKvBf16 = 0, kKvFp8 = 1, kKvNvfp4 = 2;
template <int KVF>
constexpr int kUThreadsT = 32 * (4 + kUSmxWarps + (KVF == kKvNvfp4 ? kUCvtWarps : 0)); // producer, S MMA, softmax, PV MMA, publisher[, converters]
// Warp roles by warpgroup: 0 = producer, S issuer, P.V issuer, publisher;
// 1, 2 = softmax; 3, 4 = NVFP4 converters.
constexpr int kUWarpPV = 2;                // the warp that issues the P.V MMAs
constexpr int kUWarpPub = 3;               // the warp that publishes the first unit's partial
constexpr int kUWarpSmx = 4;               // the first softmax warp
constexpr int kUWarpCvt = 4 + kUSmxWarps;  // NVFP4: the first converter warp
// NVFP4: registers a thread at launch (the most 640 threads can hold, in
// steps of 8) and after the reallocation between warpgroups; the split must
// fit in the launch allocation, or a raise would wait forever.
constexpr int kURegsLaunchF4 = 65536 / (32 * (4 + kUSmxWarps + kUCvtWarps)) / 8 * 8;
constexpr int kURegsWg0 = 64, kURegsSmx = 144, kURegsCvt = 64;
static_assert(128 * kURegsWg0 + 32 * kUSmxWarps * kURegsSmx + 32 * kUCvtWarps * kURegsCvt <=
                  32 * (4 + kUSmxWarps + kUCvtWarps) * kURegsLaunchF4,
              "NVFP4 register split above the launch allocation");
constexpr int kF4Tile = kPage * kDim / 2 + kPage * kDim / 16; // NVFP4 K or V tile: codes then scales
constexpr int kUQScales = 16;              // FP8: ring of per-unit query scales (> units in flight)
constexpr float kPScale = 256.f;           // FP8: P^T is stored as 256 * P (E4M3 hi + lo)
constexpr int kUHeads = 8;                 // heads per softmax thread (half of the group)
constexpr int kUSBufs = 4;                 // S^T accumulators: the S issuer runs up to 4 pages ahead
constexpr int kUOCol = 16 * kUSBufs;       // first TMEM column of the O^T accumulator
constexpr int kUTmemCols = 128;            // S[4] + O, 16 columns each (80, allocated as 128)
constexpr int kUTile = 32768;              // bf16 K or V tile of one (page, KV head)
constexpr int kUQTile = 4096;              // 16 query rows of one unit: bf16 (two 64-dim boxes) or E4M3 hi + lo
constexpr int kUPTile = 4096;              // P^T of one page, [16 heads][128 tokens], one part: bf16 / f16, or E4M3 hi + lo

// How far (log2 units) a head's running maximum may trail the largest
// logit seen before O^T and the denominator are rescaled: P = 2^(s - m) stays
// below 2^slack.  None: with the reference at the running maximum, the
// position that sets it has P = 1 exactly, while one with P near 2^slack
// would carry a rounding of 2^-9 (bf16) into every output it dominates; the
// E4M3 form of P (256 P, largest finite 448) takes no slack either.
__host__ __device__ constexpr float rescale_slack(int)
{
    return 0.f;
}

// Bytes of one softmax pass's P^T buffer.  bf16 and E4M3 values: a pass
// covers up to two pages of one unit, one 4 KiB part each (bf16 P; E4M3 hi +
// lo pair of 256 P); a pass over the page of a unit that has only that page
// uses the second part for the low half of P as a bf16 hi + lo pair (see the
// softmax section).  NVFP4 values: one page per pass, one f16 part.
__host__ __device__ constexpr int p_tile_bytes(int kvf)
{
    return kvf == kKvNvfp4 ? kUPTile : 2 * kUPTile;
}

// Softmax passes: up to two consecutive pages of the same unit for E4M3
// values (bound by the softmax: two pages share one max exchange and one P^T
// hand-off), one page for bf16 values (bound by the copies
// in flight: a pass that waits for its second page keeps the first page's V
// tile in the ring longer) and NVFP4 values (bound by the converter warps).
__host__ __device__ constexpr int pass_pages(int kvf)
{
    return kvf == kKvFp8 ? 2 : 1;
}

// Order of the copies into the ring: K(0), V(0), K(1), V(1), ...; copy
// number z takes ring stage z % STAGES.  (Issuing V(l) after K(l + 1), so
// that it lands closer to its use, was measured slower.)
__device__ __forceinline__ int copy_of_k(int l)
{
    return 2 * l;
}

__device__ __forceinline__ int copy_of_v(int l, int)
{
    return 2 * l + 1;
}

struct USmem {
    size_t ring, stage, qbuf, pbuf, bars, table, xbuf, lbuf, qsc, misc, qt, total;
};

// Bytes of one ring tile: bf16 (32 KiB) and E4M3 (16 KiB) tiles are the MMA
// operands as loaded; NVFP4 tiles (9 KiB) are widened to f16 staging tiles.
__host__ __device__ constexpr int ring_tile_bytes(int kvf)
{
    return kvf == kKvBf16 ? kUTile : kvf == kKvFp8 ? kUTile / 2 : kF4Tile;
}

__host__ __device__ inline USmem umma_layout(int T, int stages, int kvf)
{
    USmem L{};
    size_t off = 0;
    L.ring = off;                          // 1024-aligned tiles
    off += (size_t)stages * ring_tile_bytes(kvf);
    L.stage = off = align_to(off, 1024);   // NVFP4: bf16 K[2], V[2]
    off += kvf == kKvNvfp4 ? 4 * (size_t)kUTile : 0;
    L.qbuf = off = align_to(off, 1024);    // [2] query tiles (swizzle atoms: 1024-aligned)
    off += 2 * kUQTile;
    L.pbuf = off = align_to(off, 1024);    // [2] P^T tiles
    off += 2 * (size_t)p_tile_bytes(kvf);
    // full[S], empty[S], qfull[2], qempty[2], s_full[4], s_free[4], p_full[2],
    // p_free[2], softmax sync, done, then NVFP4 only:
    // kst_full[2], kst_empty[2], vst_full[2], vst_empty[2], qconv[2]; S and
    // PV drains, PV issuer done, first unit's slot written, last unit checked
    L.bars = off = align_to(off, 8);
    off += (size_t)(2 * stages + 8 + 2 * kUSBufs + 2 + 10 + 5) * 8;
    L.table = off = align_to(off, 16);     // [2][kWin] int4
    off += (size_t)2 * kWin * 16;
    L.xbuf = off = align_to(off, 16);      // [2][4 quarters][16] page maxima
    off += 2 * 4 * 16 * 4;
    L.lbuf = off = align_to(off, 16);      // [4 quarters][16] denominators
    off += 4 * 16 * 4;
    L.qsc = off = align_to(off, 16);       // FP8: [kUQScales] 1 / query scale of a unit
    off += kUQScales * 4;
    L.misc = off = align_to(off, 16);      // tmem base, flags, the last unit's merge check
    off += 32;
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

// v into 8 consecutive 32-bit TMEM columns of this thread's lane (warp-wide);
// the store has completed on return.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                 "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                 "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 8 consecutive 32-bit TMEM columns of this thread's lane (warp-wide), without
// waiting: the registers are valid after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two floats to E4M3 (round to nearest, saturating): a -> high byte, b -> low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float a, float b)
{
    uint32_t out;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}\n"
        : "=r"(out)
        : "f"(a), "f"(b));
    return out;
}

// x0, x1 as E4M3 pairs hi + lo with x - hi exact in fp32 and lo its rounding:
// hi + lo carries 8 significant bits (bf16's) for values in E4M3's normal
// range.  Returns (hi1 << 8 | hi0) and (lo1 << 8 | lo0).
__device__ __forceinline__ void split_e4m3x2(float x0, float x1, uint32_t &hi, uint32_t &lo)
{
    hi = f32x2_to_e4m3x2(x1, x0);
    float h0, h1;
    f16x2_to_f32x2(e4m3x2_to_f16x2(hi), h0, h1);
    lo = f32x2_to_e4m3x2(x1 - h1, x0 - h0);
}

// One step of the fixed-order merge of split partials: the weights that
// rescale the running (M, L, acc) and the incoming slot to their joint
// maximum.  Every merge (softmax warps, publisher) goes through these, with
// explicit roundings, so that any CTA produces the same bits.
struct MergeW {
    float a_old, a_s, m;
};

__device__ __forceinline__ MergeW merge_weights(float M, float ms)
{
    MergeW w;
    w.m = fmaxf(M, ms);
    const float ref = (w.m == -INFINITY) ? 0.f : w.m;
    w.a_old = ex2(M - ref); // 0 for -inf
    w.a_s = ex2(ms - ref);
    return w;
}

__device__ __forceinline__ float merge_acc(float acc, float x, const MergeW &w)
{
    return __fmaf_rn(acc, w.a_old, __fmul_rn(x, w.a_s));
}

template <int KVF, int STAGES>
__global__ void __launch_bounds__(kUThreadsT<KVF>, 1)
    sparse_decode_umma_kernel(const __grid_constant__ CUtensorMap kv_map,
                              const __grid_constant__ CUtensorMap q_map, const DecodeParams p)
{
    constexpr bool FP8 = KVF == kKvFp8;
    constexpr bool F4 = KVF == kKvNvfp4;
    constexpr int kRaw = ring_tile_bytes(KVF); // bytes of one ring tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const USmem lay = umma_layout(p.T, STAGES, KVF);
    uint8_t *ring = base + lay.ring;
    uint8_t *kst = base + lay.stage;   // NVFP4: [2] bf16 K tiles
    uint8_t *vst = kst + 2 * kUTile;   // NVFP4: [2] bf16 V tiles
    uint8_t *qbuf = base + lay.qbuf;
    uint8_t *pbuf = base + lay.pbuf;
    uint64_t *full = reinterpret_cast<uint64_t *>(base + lay.bars);
    uint64_t *empty = full + STAGES;
    uint64_t *qfull = empty + STAGES;
    uint64_t *qempty = qfull + 2;
    uint64_t *s_full = qempty + 2;       // [kUSBufs]
    uint64_t *s_free = s_full + kUSBufs; // [kUSBufs]
    uint64_t *p_full = s_free + kUSBufs;
    uint64_t *p_free = p_full + 2;
    uint64_t *smx_bar = p_free + 2;    // softmax-warps barrier (kUSmxWarps arrivals)
    uint64_t *done_bar = smx_bar + 1;  // softmax warps finished with TMEM (kUSmxWarps arrivals)
    uint64_t *kst_full = done_bar + 1; // NVFP4: [2] staging K written (kUCvtWarps arrivals)
    uint64_t *kst_empty = kst_full + 2; // NVFP4: [2] staging K read by the MMA (commit)
    uint64_t *vst_full = kst_empty + 2; // NVFP4: [2] staging V written
    uint64_t *vst_empty = vst_full + 2; // NVFP4: [2] staging V read by the MMA
    uint64_t *qconv = vst_empty + 2;    // NVFP4: [2] query tile widened to f16 (kUCvtWarps)
    uint64_t *s_drain = qconv + 2;      // the S MMAs issued before a timeout have completed (commit)
    uint64_t *pv_drain = s_drain + 1;   // the same for the PV MMAs
    uint64_t *pv_done = pv_drain + 1;   // the PV issuer has finished (1 arrival)
    uint64_t *pub_full = pv_done + 1;   // the first unit's partial is in its slot (kUSmxWarps)
    uint64_t *last_bar = pub_full + 1;  // the producer has checked the last unit's other part (1)
    float *qscale = reinterpret_cast<float *>(base + lay.qsc);
    int4 *table = reinterpret_cast<int4 *>(base + lay.table);
    float *xbuf = reinterpret_cast<float *>(base + lay.xbuf);
    float *lbuf = reinterpret_cast<float *>(base + lay.lbuf);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + lay.misc);
    int *s_flag = reinterpret_cast<int *>(base + lay.misc) + 1; // [0] last arrival, [1] abort
    // [0] the last unit's other part is published, [1] the CTA that holds it
    volatile int *last_chk = reinterpret_cast<int *>(base + lay.misc) + 4;
    volatile int *smx_done = reinterpret_cast<int *>(base + lay.misc) + 6; // the softmax warps have finished
    int *qt = reinterpret_cast<int *>(base + lay.qt);
    volatile int *abort_flag = s_flag + 1;
    const long long wl = p.wait_limit; // clocks of every wait below but the final drains
    // A wait made by every lane of a warp, with one outcome for the whole
    // warp: a lane that saw the phase complete and one that gave up would
    // otherwise part ways before warp-wide instructions.
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, mbar_wait_or_abort(bar, parity, abort_flag, wl));
    };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        if (!F4)
            prefetch_tensormap(&kv_map);
        prefetch_tensormap(&q_map);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), F4 ? kUCvtWarps : 1); // NVFP4: freed by the converters
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&kst_full[b]), kUCvtWarps);
            mbar_init(smem_u32(&kst_empty[b]), 1);
            mbar_init(smem_u32(&vst_full[b]), kUCvtWarps);
            mbar_init(smem_u32(&vst_empty[b]), 1);
            mbar_init(smem_u32(&qconv[b]), kUCvtWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&qfull[b]), 1);
            mbar_init(smem_u32(&qempty[b]), 1);
            mbar_init(smem_u32(&p_full[b]), kUSmxWarps);
            mbar_init(smem_u32(&p_free[b]), 1);
        }
        for (int i = 0; i < kUSBufs; ++i) {
            mbar_init(smem_u32(&s_full[i]), 1);
            mbar_init(smem_u32(&s_free[i]), kUSmxWarps);
        }
        mbar_init(smem_u32(smx_bar), kUSmxWarps);
        mbar_init(smem_u32(done_bar), kUSmxWarps);
        mbar_init(smem_u32(s_drain), 1);
        mbar_init(smem_u32(pv_drain), 1);
        mbar_init(smem_u32(pv_done), 1);
        mbar_init(smem_u32(pub_full), kUSmxWarps);
        mbar_init(smem_u32(last_bar), 1);
        s_flag[0] = 0;
        s_flag[1] = 0;
        *smx_done = 0;
        fence_mbar_init();
    }
    if (warp == 1)
        tmem_alloc(smem_u32(tmem_slot), kUTmemCols);
    build_token_prefix(p, qt, reinterpret_cast<int *>(lbuf)); // lbuf is free until the first finalize
    tcgen05_before_sync();
    __syncthreads();
    tcgen05_after_sync();
    const uint32_t tmem = *tmem_slot;

    const long long P = (long long)p.Hkv * qt[p.T];
    const int G = gridDim.x, c = blockIdx.x;
    const long long x_begin = (uint32_t)c * (uint32_t)P / (uint32_t)G; // 32-bit: see owner_of
    const long long x_end = (uint32_t)(c + 1) * (uint32_t)P / (uint32_t)G;
    const int ntasks = (int)(x_end - x_begin);

    // Unit (t, g): its tasks [first, end) in the order all CTAs cut, and the
    // CTAs whose ranges hold them.
    struct UnitOwn {
        long long first, end;
        int u, c_first, c_last;
    };
    auto own_of = [&](int t, int g) {
        UnitOwn w;
        w.first = (long long)g * qt[p.T] + qt[t];
        w.end = w.first + (qt[t + 1] - qt[t]);
        w.c_first = owner_of(w.first, P, G);
        w.c_last = owner_of(w.end - 1, P, G);
        w.u = g * p.T + t;
        return w;
    };
    auto arrivals_of = [&](const UnitOwn &w) { // CTAs with tasks of the unit
        int a = 0;
        for (int cc = w.c_first; cc <= w.c_last; ++cc)
            a += !range_empty(cc, P, G);
        return a;
    };

    // The query rows of unit number unit_no of this CTA (16 rows from `row`)
    // into query buffer qb; called by the whole producer warp.  bf16 and
    // NVFP4 K/V: one TMA copy (two 64-dim boxes); E4M3 K/V: converted here.
    int q_issued = 0; // TMA query loads issued (for the drain after a timeout)
    auto load_q = [&](int qb, int row, int unit_no) {
        if (!FP8) {
            if (lane == 0) {
                const uint32_t qbar = smem_u32(&qfull[qb]);
                const uint32_t dst = smem_u32(qbuf + qb * kUQTile);
                mbar_arrive_expect_tx(qbar, kUQTile);
                tma_load_2d(dst, &q_map, 0, row, qbar);
                tma_load_2d(dst + kUQTile / 2, &q_map, 64, row, qbar);
                q_issued = unit_no + 1;
            }
        } else {
            // E4M3 hi + lo tiles of s * q (K-major, 128-byte swizzle),
            // s = 2^k with max |s q| in [128, 256): lane = (row, 64 dims)
            const int r = lane >> 1, hf = lane & 1;
            const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (size_t)(row + r) * kDim + hf * 64);
            uint4 v[8];
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v[i] = __ldg(src + i);
                const uint32_t w4[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[j] << 16)),
                                         fabsf(__uint_as_float(w4[j] & 0xFFFF0000u))));
            }
            mx = warp_max_f32(mx);
            int k = 0;
            if (mx > 0.f && mx < INFINITY) {
                k = 7 - ((int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127);
                k = k < -100 ? -100 : (k > 100 ? 100 : k);
            }
            const float sq = __uint_as_float((uint32_t)(127 + k) << 23);
            uint8_t *qhi = qbuf + qb * kUQTile, *qlo = qhi + kUQTile / 2;
#pragma unroll
            for (int j = 0; j < 4; ++j) { // 16 dims = one 16-byte chunk of E4M3
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int w = 0; w < 4; ++w) { // 4 dims = 2 words of the bf16 input
                    const int i = 2 * j + (w >> 1);
                    const uint32_t a = (&v[i].x)[2 * (w & 1)], b = (&v[i].x)[2 * (w & 1) + 1];
                    uint32_t h01, l01, h23, l23;
                    split_e4m3x2(__uint_as_float(a << 16) * sq, __uint_as_float(a & 0xFFFF0000u) * sq, h01, l01);
                    split_e4m3x2(__uint_as_float(b << 16) * sq, __uint_as_float(b & 0xFFFF0000u) * sq, h23, l23);
                    hw[w] = h01 | (h23 << 16);
                    lw[w] = l01 | (l23 << 16);
                }
                const int off = r * 128 + (((4 * hf + j) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(qhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                *reinterpret_cast<uint4 *>(qlo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
            if (lane == 0)
                qscale[unit_no % kUQScales] = __uint_as_float((uint32_t)(127 - k) << 23);
            fence_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(&qfull[qb]));
        }
    };
    // The queries do not depend on the previous kernel of the step: the first
    // unit's rows are staged before the grid wait.
    if (warp == 0 && ntasks > 0) {
        const Task t0 = task_of(x_begin, qt, p.T);
        load_q(0, (t0.t * p.Hkv + t0.g) * kGroup, 0);
    }

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
    // the first two table windows, filled by all threads (one round of the
    // two dependent reads for up to blockDim.x tasks) and visible to every
    // warp before anything starts
    for (int i = threadIdx.x; i < 2 * kWin && i < ntasks; i += blockDim.x)
        table[i] = make_entry(p, x_begin + i, qt);
    __syncthreads();

    // Instruction descriptors.  bf16: kind::f16, 8 steps of K = 16.  FP8:
    // kind::f8f6f4 on the E4M3 tiles as loaded, 4 steps of K = 32 for each of
    // the hi and lo parts of Q (in S^T) and of P (in O^T); operand types
    // E4M3 = 0.  NVFP4: kind::f16 with f16 operands (format 0), widened in
    // shared memory.
    constexpr uint32_t kE4M3 = (FP8 || F4) ? ~((7u << 7) | (7u << 10)) : ~0u;
    constexpr uint32_t kIdescS = umma_idesc_bf16(128, 16, 0, 0) & kE4M3; // K and Q^T both K-major
    constexpr uint32_t kIdescO = umma_idesc_bf16(128, 16, 1, 0) & kE4M3; // V^T MN-major, P^T K-major

    // Pages per softmax pass: a pass takes the next two tasks if they belong
    // to one unit (bf16 / E4M3 values), else one.  The softmax warps and the
    // P.V issuer walk the same passes.
    auto pass_len = [&](int l0) -> int {
        if (pass_pages(KVF) == 1 || l0 + 1 >= ntasks)
            return 1;
        return unit_of(entry(l0 + 1)) == unit_of(entry(l0)) ? 2 : 1;
    };

    if (warp < kUWarpSmx) {
        // ======== warpgroup 0: producer, S issuer, P.V issuer, publisher ========
        if constexpr (F4)
            setmaxnreg_dec<kURegsWg0>(); // the NVFP4 CTA's registers go to the softmax warps

        if (warp == 0) {
            // =================== producer ===================
            constexpr int kAhead = STAGES / 2;
            const uint64_t kv_policy = l2_evict_first_policy(); // pages are streamed
            int issued = 0, prod_units = 0, prod_last = -1;
            bool ok = true;
            for (int z = 0; z < 2 * ntasks && ok; ++z) {
                // copy z: K(l) or V(l) (the order of copy_of_k / copy_of_v)
                const bool is_k = (z & 1) == 0;
                const int l = z >> 1;
                if (lane == 0 && z >= STAGES)
                    ok = mbar_wait_or_abort(smem_u32(&empty[z % STAGES]), ((z / STAGES) - 1) & 1,
                                            abort_flag, wl);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                const int4 e = entry(l);
                if (is_k) {
                    // The slowest reader of the table is the P.V issuer: copy
                    // K(l) comes after V(l - 1), which took the stage of
                    // V(l - 1 - kAhead) once its P.V MMAs had freed it, so that
                    // reader trails this warp by at most kAhead tasks (+ 2 with
                    // the NVFP4 converters and their two staging tiles between
                    // them); the softmax warps, the S issuer and the converters
                    // are ahead of it.  Only kAhead + 3 (+ 2) tasks into a window
                    // has every reader left the window before it.
                    if (l % kWin == kAhead + 3 + (F4 ? 2 : 0) && l >= kWin && (l / kWin + 1) * kWin < ntasks)
                        fill_window(l / kWin + 1);
                    const int u = unit_of(e);
                    if (u != prod_last) {
                        // the unit's 16 query rows into query buffer qb (the first
                        // unit's were staged before the grid wait)
                        prod_last = u;
                        const int qb = prod_units & 1;
                        if (prod_units > 0) {
                            if (lane == 0 && prod_units >= 2)
                                ok = mbar_wait_or_abort(smem_u32(&qempty[qb]), ((prod_units >> 1) - 1) & 1, abort_flag, wl);
                            ok = __shfl_sync(0xffffffffu, ok, 0);
                            if (!ok)
                                break;
                            load_q(qb, (e.z * p.Hkv + e.w) * kGroup, prod_units);
                        }
                        ++prod_units;
                    }
                }
                if (lane == 0) {
                    const int st = z % STAGES;
                    const uint32_t bar = smem_u32(&full[st]);
                    issued = z + 1;
                    if (e.x < 0) {
                        mbar_arrive(bar); // no data: consumers skip the task
                    } else {
                        const uint32_t dst = smem_u32(ring + (size_t)st * kRaw);
                        const int krow = e.x + (is_k ? 0 : p.Hkv * kPage);
                        mbar_arrive_expect_tx(bar, kRaw);
                        if (F4) { // one contiguous tile: codes then scales
                            bulk_load_hint(dst, p.kv_raw + (size_t)(krow / kPage) * kF4Tile, kF4Tile, bar,
                                           kv_policy);
                        } else {
                            tma_load_2d_hint(dst, &kv_map, 0, krow, bar, kv_policy);
                            if (!FP8)
                                tma_load_2d_hint(dst + kUTile / 2, &kv_map, 64, krow, bar, kv_policy);
                        }
                    }
                }
            }
            // The CTA's last unit, begun here and continued by later CTAs, which
            // publish their parts at their starts: with every copy issued, one
            // acquire load tells whether the one other part is in, so that the
            // softmax warps can read it during their last pass and merge at once.
            if (ok && ntasks > 0 && lane == 0) {
                const int4 el = entry(ntasks - 1);
                const UnitOwn w = own_of(el.z, el.w);
                if (w.c_first == c && w.c_last > c) {
                    int other = -1, n_other = 0;
                    for (int cc = c + 1; cc <= w.c_last; ++cc)
                        if (!range_empty(cc, P, G)) {
                            other = cc;
                            ++n_other;
                        }
                    int in = 0;
                    if (n_other == 1 && (long long)w.c_last + w.u < p.slots)
                        in = ld_acquire_gpu(&p.counters[w.u]) == 1;
                    last_chk[0] = in;
                    last_chk[1] = other;
                    mbar_arrive(smem_u32(last_bar));
                }
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
            // =================== S issuer (lane 0) + TMEM owner ===================
            // S^T(l) into accumulator l % kUSBufs as soon as K(l) has landed and
            // the softmax warps have read S^T(l - kUSBufs): the S MMAs run ahead
            // of the softmax, independently of the P.V MMAs (their own thread).
            bool ok = true;
            if (lane == 0) {
                int s_units = 0, s_unit = -1;
                for (int l = 0; l < ntasks; ++l) {
                    const int zk = copy_of_k(l), sb = l % kUSBufs;
                    // NVFP4: K(l) widened into staging tile l & 1; else the ring tile landed
                    if (F4 ? !mbar_wait_or_abort(smem_u32(&kst_full[l & 1]), (l >> 1) & 1, abort_flag, wl)
                           : !mbar_wait_or_abort(smem_u32(&full[zk % STAGES]), (zk / STAGES) & 1, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    const int4 e = entry(l);
                    const int u = unit_of(e);
                    if (u != s_unit) {
                        // NVFP4: the converter warps widen the query tile to f16 in place
                        uint64_t *qready = F4 ? qconv : qfull;
                        if (!mbar_wait_or_abort(smem_u32(&qready[s_units & 1]), (s_units >> 1) & 1, abort_flag, wl)) {
                            ok = false;
                            break;
                        }
                        s_unit = u;
                        ++s_units;
                    }
                    const int qb = (s_units - 1) & 1;
                    if (l >= kUSBufs &&
                        !mbar_wait_or_abort(smem_u32(&s_free[sb]), ((l / kUSBufs) - 1) & 1, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    tcgen05_after_sync();
                    if (e.x >= 0) {
                        const uint32_t tileK = F4 ? smem_u32(kst + (l & 1) * kUTile)
                                                  : smem_u32(ring + (size_t)(zk % STAGES) * kRaw);
                        const uint32_t qtile = smem_u32(qbuf + qb * kUQTile);
    #pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            if (!FP8) {
                                const uint64_t a = umma_desc_sw128(tileK + (ks >> 2) * (kUTile / 2) + (ks & 3) * 32, 16, 1024);
                                const uint64_t bq = umma_desc_sw128(qtile + (ks >> 2) * (kUQTile / 2) + (ks & 3) * 32, 16, 1024);
                                umma_bf16(tmem + 16 * sb, a, bq, kIdescS, ks > 0);
                            } else { // steps 0..3: Q hi, 4..7: Q lo; 32 dims (bytes) per step
                                const uint64_t a = umma_desc_sw128(tileK + (ks & 3) * 32, 16, 1024);
                                const uint64_t bq = umma_desc_sw128(qtile + (ks >> 2) * (kUQTile / 2) + (ks & 3) * 32, 16, 1024);
                                umma_f8(tmem + 16 * sb, a, bq, kIdescS, ks > 0);
                            }
                        }
                    }
                    umma_commit(smem_u32(&s_full[sb]));
                    umma_commit(F4 ? smem_u32(&kst_empty[l & 1]) : smem_u32(&empty[zk % STAGES])); // K tile read
                    // last task of its unit: the query tile can be replaced
                    if (l + 1 == ntasks || unit_of(entry(l + 1)) != u)
                        umma_commit(smem_u32(&qempty[qb]));
                }
                if (!ok) {
                    set_error(p.err, kErrTimeout);
                    *abort_flag = 1;
                    // the MMAs issued so far finish before TMEM is freed
                    umma_commit(smem_u32(s_drain));
                    (void)mbar_wait_bounded(smem_u32(s_drain), 0);
                }
            }
            __syncwarp();
            // free TMEM once the softmax warps and the PV issuer are done with it
            // (they always arrive, also after an abort; the waits are bounded)
            if (lane == 0) {
                (void)mbar_wait_bounded(smem_u32(done_bar), 0);
                (void)mbar_wait_bounded(smem_u32(pv_done), 0);
            }
            __syncwarp();
            tcgen05_after_sync();
            tmem_dealloc(tmem, kUTmemCols);
            return;
        }

        if (warp == kUWarpPV) {
            // =================== P.V issuer (lane 0) ===================
            // O^T of a unit accumulates in one TMEM accumulator over the
            // unit's passes: pass j's MMAs once the softmax warps have written
            // its P^T (and rescaled O^T, when they moved the reference), each
            // page as soon as its V tile has landed.
            if (lane == 0) {
                bool ok = true;
                int j = 0, pv_unit = -1;
                bool acc = false; // a page of the unit has written the accumulator
                for (int l0 = 0; l0 < ntasks && ok; l0 += pass_len(l0), ++j) {
                    const int np = pass_len(l0), pb = j & 1;
                    if (!mbar_wait_or_abort(smem_u32(&p_full[pb]), (j >> 1) & 1, abort_flag, wl)) {
                        ok = false;
                        break;
                    }
                    // The softmax warps have read the previous unit's O^T (before
                    // they wrote this P^T): a new unit starts it afresh.
                    const int u0 = unit_of(entry(l0));
                    if (u0 != pv_unit) {
                        pv_unit = u0;
                        acc = false;
                    }
                    for (int i = 0; i < np; ++i) {
                        const int l = l0 + i, zv = copy_of_v(l, ntasks);
                        if (F4 ? !mbar_wait_or_abort(smem_u32(&vst_full[l & 1]), (l >> 1) & 1, abort_flag, wl)
                               : !mbar_wait_or_abort(smem_u32(&full[zv % STAGES]), (zv / STAGES) & 1, abort_flag, wl)) {
                            ok = false;
                            break;
                        }
                        tcgen05_after_sync();
                        const int4 e = entry(l);
                        if (e.x >= 0) {
                            const uint32_t tileV = F4 ? smem_u32(vst + (l & 1) * kUTile)
                                                      : smem_u32(ring + (size_t)(zv % STAGES) * kRaw);
                            const uint32_t ptile = smem_u32(pbuf + pb * p_tile_bytes(KVF) + i * kUPTile);
                            // bf16: steps 0..7 take P hi, 8..15 (single-page units) P lo,
                            // over the same V^T slices
                            const int pv_steps = (KVF == kKvBf16 && qt[e.z + 1] - qt[e.z] == 1) ? 16 : 8;
    #pragma unroll
                            for (int ks = 0; ks < 16; ++ks) {
                                if (ks >= pv_steps)
                                    break;
                                if (!FP8) {
                                    // V^T, MN-major: 16 tokens per k-step = 16 rows of 128 bytes;
                                    // the two 64-dim halves of a row are 16 KiB apart (LBO)
                                    const int kt = ks & 7;
                                    const uint64_t a = umma_desc_sw128(tileV + kt * 2048, kUTile / 2, 1024);
                                    const uint64_t bp = umma_desc_sw128(
                                        ptile + (ks >> 3) * kUPTile + (kt >> 2) * (kUPTile / 2) + (kt & 3) * 32, 16, 1024);
                                    umma_bf16(tmem + kUOCol, a, bp, kIdescO, acc || ks > 0);
                                } else {
                                    // V^T, MN-major: 32 tokens per k-step = 32 rows of 128 bytes
                                    // (all 128 dims in one swizzle atom); steps 0..3: P hi, 4..7: P lo
                                    const uint64_t a = umma_desc_sw128(tileV + (ks & 3) * 4096, kUTile / 2, 1024);
                                    const uint64_t bp = umma_desc_sw128(ptile + (ks >> 2) * (kUPTile / 2) + (ks & 3) * 32, 16, 1024);
                                    umma_f8(tmem + kUOCol, a, bp, kIdescO, acc || ks > 0);
                                }
                            }
                            acc = true;
                        }
                        umma_commit(F4 ? smem_u32(&vst_empty[l & 1]) : smem_u32(&empty[zv % STAGES])); // V tile read
                    }
                    if (!ok)
                        break;
                    // P^T buffer pb read and O^T through this pass complete
                    umma_commit(smem_u32(&p_free[pb]));
                }
                if (!ok) {
                    set_error(p.err, kErrTimeout);
                    *abort_flag = 1;
                    umma_commit(smem_u32(pv_drain));
                    (void)mbar_wait_bounded(smem_u32(pv_drain), 0);
                }
                mbar_arrive(smem_u32(pv_done));
            }
            return;
        }

        if (warp == kUWarpPub) {
            // =================== publisher ===================
            // The CTA's first unit, begun by an earlier CTA, when more units
            // follow it here: the softmax warps put its partial in this CTA's
            // slot and go on; this warp counts the arrival (an acquire-release
            // atomic, a round trip to L2 the softmax warps would otherwise wait
            // for).  The arrival that completes the unit merges it: here only
            // when the earlier CTA finished first, which a CTA that was not yet
            // resident can see.
            if (ntasks == 0)
                return;
            const int4 e0 = table[0];
            const UnitOwn w = own_of(e0.z, e0.w);
            if (w.c_first == w.c_last || w.end >= x_end || (long long)w.c_last + w.u >= p.slots)
                return; // whole, or also the last unit here (the softmax warps finish it)
            // The softmax warps hand the partial over, or finish without doing
            // so (after an abort); the wait ends on either and is bounded.
            bool handed = mbar_try_wait(smem_u32(pub_full), 0);
            if (!handed) {
                const long long start = clock64();
                while (!(handed = mbar_try_wait(smem_u32(pub_full), 0))) {
                    if (*abort_flag || clock64() - start > wl)
                        break;
                    if (*smx_done) {
                        // every softmax warp passes a barrier of all of them after
                        // its hand-off, before any of them finishes: look once more
                        __threadfence_block();
                        handed = mbar_try_wait(smem_u32(pub_full), 0);
                        break;
                    }
                }
            }
            if (!__all_sync(0xffffffffu, handed))
                return; // nothing is published
            int last = 0;
            if (lane == 0)
                last = atom_add_acq_rel_gpu(&p.counters[w.u], 1) == arrivals_of(w) - 1;
            if (!__shfl_sync(0xffffffffu, last, 0))
                return;
            // Merge every slot of the unit in slot (CTA) order, one head at a
            // time: lane = dimensions 4 lane .. 4 lane + 3, with a running maximum.
            const size_t hb = (size_t)e0.z * p.Hkv * kGroup + (size_t)e0.w * kGroup;
            for (int h = 0; h < kGroup; ++h) {
                float Mx = -INFINITY, Lx = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
                for (int cc = w.c_first; cc <= w.c_last; ++cc) {
                    if (range_empty(cc, P, G))
                        continue;
                    const float *sl = p.partial + (size_t)(cc + w.u) * kPartialFloats;
                    const float ms = __ldcg(sl + kGroup * kDim + h), ls = __ldcg(sl + kGroup * kDim + kGroup + h);
                    const float4 os = __ldcg(reinterpret_cast<const float4 *>(sl + h * kDim) + lane);
                    const MergeW mw = merge_weights(Mx, ms);
                    Lx = merge_acc(Lx, ls, mw);
                    acc[0] = merge_acc(acc[0], os.x, mw);
                    acc[1] = merge_acc(acc[1], os.y, mw);
                    acc[2] = merge_acc(acc[2], os.z, mw);
                    acc[3] = merge_acc(acc[3], os.w, mw);
                    Mx = mw.m;
                }
                const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
                uint2 ov;
                ov.x = pack_bf16(acc[0] * inv, acc[1] * inv);
                ov.y = pack_bf16(acc[2] * inv, acc[3] * inv);
                *reinterpret_cast<uint2 *>(p.out + (hb + h) * kDim + 4 * lane) = ov;
                if (lane == 0)
                    p.lse[hb + h] = (Mx == -INFINITY) ? -INFINITY : (Mx + log2f(Lx)) * 0.69314718055994531f;
            }
            if (lane == 0)
                p.counters[w.u] = 0; // ready for the next call
            return;
        }

        return;
    }

    if (F4 && warp >= kUWarpCvt) {
        setmaxnreg_dec<kURegsCvt>();
        // =================== converter warps (NVFP4) ===================
        // K and V tiles from the ring (e2m1 pairs [128 tok][64 B], then E4M3
        // scales [128 tok][8]) into the f16 staging tiles, in the
        // two-64-dim-box, 128-byte-swizzled layout the MMA descriptors read:
        // one cvt.f16x2.e2m1x2 and one f16x2 multiply by the scale per two
        // values.  e2m1 x E4M3 has at most 6 significant bits: exact in f16.
        // The query tile of each new unit is widened from bf16 to f16 in
        // place.  The tensor scales are folded into the logit scale and the
        // output.
        const int ct = threadIdx.x - 32 * kUWarpCvt; // 0 .. 32 * kUCvtWarps - 1
        bool ok = true;
        int units = 0, cur = -1;
        // Thread ct widens the 16 dimensions gch = ct % 8 of rows ct / 8 + kStep i,
        // i < kRows; all loads before the first convert.
        constexpr int kStep = 4 * kUCvtWarps, kRows = kPage / kStep;
        static_assert(kStep % 8 == 0 && kPage % kStep == 0, "converter rows");
        const int gch = ct & 7, r0 = ct >> 3, sw = r0 & 7; // r & 7 == sw for every row of the thread
        const int box = gch >> 2, c0 = 2 * (gch & 3);      // 64-dim box and its first 16-byte chunk
        auto convert = [&](const uint8_t *raw, uint8_t *dst) {
            uint2 cw[kRows];
            uint32_t sc[kRows];
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const int r = r0 + kStep * i;
                cw[i] = *reinterpret_cast<const uint2 *>(raw + r * 64 + gch * 8);
                sc[i] = raw[kPage * 64 + r * 8 + gch];
            }
            uint8_t *lo_dst = dst + box * (kUTile / 2) + ((c0 ^ sw) << 4);
            uint8_t *hi_dst = dst + box * (kUTile / 2) + (((c0 + 1) ^ sw) << 4);
#pragma unroll
            for (int i = 0; i < kRows; ++i) {
                const uint32_t s2 = e4m3x2_to_f16x2(sc[i] | (sc[i] << 8)); // (scale, scale)
                uint32_t lo[4], hi[4]; // dimensions 0..7 and 8..15 of the group
                e2m1x8_scaled_f16x2(cw[i].x, s2, lo);
                e2m1x8_scaled_f16x2(cw[i].y, s2, hi);
                const int r = r0 + kStep * i;
                *reinterpret_cast<uint4 *>(lo_dst + r * 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(hi_dst + r * 128) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
            fence_async_smem();
        };
        // K(l + 1) is widened before V(l): the MMA warp issues S(l + 1)
        // before O(l).
        auto do_kv = [&](int l, int kv) -> bool {
            const int z = kv ? copy_of_v(l, ntasks) : copy_of_k(l), b = l & 1;
            uint64_t *st_full = kv ? vst_full : kst_full, *st_empty = kv ? vst_empty : kst_empty;
            if (!wait_all(smem_u32(&full[z % STAGES]), (z / STAGES) & 1))
                return false;
            const int4 e = entry(l);
            if (kv == 0 && unit_of(e) != cur) {
                const int qb = units & 1;
                if (!wait_all(smem_u32(&qfull[qb]), (units >> 1) & 1))
                    return false;
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
                cur = unit_of(e);
                ++units;
            }
            if (l >= 2 && !wait_all(smem_u32(&st_empty[b]), ((l >> 1) - 1) & 1))
                return false;
            if (e.x >= 0)
                convert(ring + (size_t)(z % STAGES) * kRaw, (kv ? vst : kst) + b * kUTile);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&st_full[b]));
                mbar_arrive(smem_u32(&empty[z % STAGES]));
            }
            return true;
        };
        if (ntasks > 0)
            ok = do_kv(0, 0);
        for (int l = 0; l < ntasks && ok; ++l) {
            if (l + 1 < ntasks)
                ok = do_kv(l + 1, 0);
            if (ok)
                ok = do_kv(l, 1);
        }
        if (!ok) {
            set_error(p.err, kErrTimeout);
            *abort_flag = 1;
        }
        return;
    }

    // =================== softmax warps 4..11 ===================
    if constexpr (F4)
        setmaxnreg_inc<kURegsSmx>(); // waits for the other warpgroups' registers
    // Warps w and w + 4 share TMEM lanes 32*(w & 3) .. +31 and split the 16
    // heads into halves: each thread holds one token (of S^T) or one dimension
    // (of O^T) for kUHeads heads.
    const int quarter = warp & 3;
    const int half = (warp - kUWarpSmx) >> 2; // heads 8*half .. 8*half + 7
    const int h0 = kUHeads * half;
    const int idx = 32 * quarter + lane;   // token of S^T / dimension of O^T
    const int sidx = threadIdx.x - 32 * kUWarpSmx; // 0 .. 32 * kUSmxWarps - 1
    const uint32_t lane_base = tmem + ((uint32_t)(32 * quarter) << 16) + h0;
    int sync_phase = 0;
    bool ok = true;
    // barrier of the softmax warps: one arrival per warp after __syncwarp
    // (which orders the warp's shared and global writes before lane 0's
    // release arrival)
    auto ssync = [&]() {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(smx_bar));
        if (!wait_all(smem_u32(smx_bar), sync_phase & 1))
            ok = false;
        ++sync_phase;
    };

    // m_run: the reference of the unit's P (base 2), within rescale_slack of
    // the largest logit seen; lsum and O^T (in TMEM) are relative to it.
    float o[kUHeads], lsum[kUHeads], m_run[kUHeads];
    bool o_live = false; // a page of the unit has been accumulated into O^T
    int cur_unit = -1, cur_t = 0, cur_g = 0;
    bool cur_cand = false; // the unit begins in this CTA and continues in later ones

    auto reset = [&]() {
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            lsum[h] = 0.f;
            m_run[h] = -INFINITY;
        }
        o_live = false;
    };

    // Wait until the P.V MMAs of pass jp (and so every earlier one) have
    // completed: they release P^T buffer jp & 1.  Called in pass jp + 1
    // before its P^T is written; that buffer's phase of pass jp - 2 was
    // waited for in pass jp, and pass jp + 2 cannot start: the parity names
    // one phase.
    auto wait_pv = [&](int jp) {
        if (!wait_all(smem_u32(&p_free[jp & 1]), (jp >> 1) & 1))
            ok = false;
        tcgen05_after_sync();
    };

    // the unit's O^T (thread = dimension) into o[] once its last pass (jp) is in
    auto read_o = [&](int jp) {
        if (!o_live) {
#pragma unroll
            for (int h = 0; h < kUHeads; ++h)
                o[h] = 0.f;
            return;
        }
        wait_pv(jp);
        if (ok)
            tmem_ld8(lane_base + kUOCol, o);
    };

    // The other CTA's partial of the last unit, read during the last pass
    // when the producer found it published (pre).
    bool pre = false;
    float ms2[kUHeads], ls2[kUHeads], os2[kUHeads];

    // final: the CTA's last unit
    auto finalize = [&](int t, int g, bool final) {
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
        // (lbuf is next written in the next unit's finalize, after at least
        // one pass and its barrier: every thread has read it by then)
        float L[kUHeads];
#pragma unroll
        for (int h = 0; h < kUHeads; ++h)
            L[h] = lbuf[h0 + h] + lbuf[16 + h0 + h] + lbuf[32 + h0 + h] + lbuf[48 + h0 + h];
        const UnitOwn w = own_of(t, g);
        const int u = w.u;
        const bool whole = w.c_first == w.c_last;
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
            o[h] *= FP8 ? p.v_scale / kPScale : p.v_scale; // 1 for bf16 values
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
        if ((long long)w.c_last + u >= p.slots) { // the caller's scratch is short: no slot is touched
            if (sidx == 0)
                set_error(p.err, kErrScratch);
            return;
        }
        if (!final) {
            // The CTA's first unit, begun by an earlier CTA, with more units
            // here: its partial goes to this CTA's slot, and the publisher
            // warp counts the arrival (and merges if it completes the unit).
#pragma unroll
            for (int h = 0; h < kUHeads; ++h)
                slot[(h0 + h) * kDim + idx] = o[h];
            if (idx < kUHeads) {
                slot[kGroup * kDim + h0 + idx] = Mi;
                slot[kGroup * kDim + kGroup + h0 + idx] = Li;
            }
            // __syncwarp orders the warp's slot writes before lane 0's
            // release arrival; the publisher's acquire wait and its
            // acquire-release atomic carry them to the CTA that merges.
            __syncwarp();
            if (lane == 0)
                mbar_arrive(smem_u32(pub_full));
            return;
        }
        bool last = pre; // pre: the one other part is in and already read
        if (!pre) {
            // The CTA's last unit otherwise: when every other CTA of the unit
            // is already in, merge at once from registers and their slots,
            // else publish and count the arrival; the arrival that completes
            // the unit merges it.
            const int arrivals = arrivals_of(w);
            if (sidx == 0)
                s_flag[0] = ld_acquire_gpu(&p.counters[u]) == arrivals - 1;
            ssync();
            last = s_flag[0] != 0;
            ssync(); // s_flag is read by every thread before it is rewritten
            if (!last) {
#pragma unroll
                for (int h = 0; h < kUHeads; ++h)
                    slot[(h0 + h) * kDim + idx] = o[h];
                if (idx < kUHeads) {
                    slot[kGroup * kDim + h0 + idx] = Mi;
                    slot[kGroup * kDim + kGroup + h0 + idx] = Li;
                }
                // The CTA barrier orders every thread's slot writes before
                // thread 0's release; its acquire makes the other CTAs' slots
                // visible to the CTA that arrives last, and the barrier after
                // it to all its threads.
                ssync();
                if (sidx == 0)
                    s_flag[0] = atom_add_acq_rel_gpu(&p.counters[u], 1) == arrivals - 1;
                ssync();
                last = s_flag[0] != 0;
            }
        }
        if (last) {
            // Combine the unit's slots in slot (CTA) order, this CTA's own
            // part from registers (thread = dimension idx for 8 heads), the
            // pre-read one from registers, the others from L2; all loads of a
            // slot are issued before its arithmetic.
            float Mx[kUHeads], Lx[kUHeads], acc[kUHeads];
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                Mx[h] = -INFINITY;
                Lx[h] = 0.f;
                acc[h] = 0.f;
            }
            for (int cc = w.c_first; cc <= w.c_last; ++cc) {
                if (range_empty(cc, P, G))
                    continue;
                float ms[kUHeads], ls[kUHeads], os[kUHeads];
                if (cc == c) {
#pragma unroll
                    for (int h = 0; h < kUHeads; ++h) {
                        ms[h] = m_run[h];
                        ls[h] = L[h];
                        os[h] = o[h];
                    }
                } else if (pre) {
#pragma unroll
                    for (int h = 0; h < kUHeads; ++h) {
                        ms[h] = ms2[h];
                        ls[h] = ls2[h];
                        os[h] = os2[h];
                    }
                } else {
                    const float *sl = p.partial + (size_t)(cc + u) * kPartialFloats;
#pragma unroll
                    for (int h = 0; h < kUHeads; ++h) {
                        ms[h] = __ldcg(sl + kGroup * kDim + h0 + h);
                        ls[h] = __ldcg(sl + kGroup * kDim + kGroup + h0 + h);
                        os[h] = __ldcg(sl + (h0 + h) * kDim + idx);
                    }
                }
#pragma unroll
                for (int h = 0; h < kUHeads; ++h) {
                    const MergeW mw = merge_weights(Mx[h], ms[h]);
                    Lx[h] = merge_acc(Lx[h], ls[h], mw);
                    acc[h] = merge_acc(acc[h], os[h], mw);
                    Mx[h] = mw.m;
                }
            }
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                const float inv = Lx[h] > 0.f ? 1.f / Lx[h] : 0.f;
                p.out[(hbase + h) * kDim + idx] = (uint16_t)(pack_bf16(acc[h] * inv, 0.f) & 0xFFFFu);
                if (idx == h)
                    p.lse[hbase + h] = (Mx[h] == -INFINITY) ? -INFINITY
                                                             : (Mx[h] + log2f(Lx[h])) * 0.69314718055994531f;
            }
            if (sidx == 0)
                p.counters[u] = 0; // ready for the next call
        }
    };

    // P^T[h][token idx] of page i of pass buffer pb, in the K-major,
    // 128-byte-swizzled B-operand form.
    auto store_p = [&](const float (&pv)[kUHeads], int pb, int i, bool hilo) {
        if (!FP8) {
            // bf16: hi = bf16(p); with hilo (the page of a single-page unit)
            // also lo = bf16(p - hi) (exact in fp32) in the second part.  There
            // a handful of positions can carry the whole softmax, and P rounded
            // to bf16 alone would put an error of up to 2^-9 |V| into O; a unit
            // with two or more pages sees at least 129 positions (every
            // selected block but the last visible one is full), where those
            // roundings average out.  NVFP4: f16(p).
            uint8_t *pt = pbuf + pb * p_tile_bytes(KVF) + i * kUPTile + (idx >> 6) * (kUPTile / 2);
            const int col = idx & 63;
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                const int hh = h0 + h;
                const uint32_t off = hh * 128 + ((((col >> 3) ^ (hh & 7))) << 4) + (col & 7) * 2;
                if (F4) {
                    *reinterpret_cast<uint16_t *>(pt + off) = (uint16_t)(pack_f16(pv[h], 0.f) & 0xFFFFu);
                } else {
                    const uint32_t hi = pack_bf16(pv[h], 0.f) & 0xFFFFu;
                    *reinterpret_cast<uint16_t *>(pt + off) = (uint16_t)hi;
                    if (hilo) {
                        const uint32_t lo = pack_bf16(pv[h] - __uint_as_float(hi << 16), 0.f) & 0xFFFFu;
                        *reinterpret_cast<uint16_t *>(pt + kUPTile + off) = (uint16_t)lo;
                    }
                }
            }
        } else {
            // FP8: 256 P as E4M3 hi + lo, one byte per (head row, token) in
            // each of two K-major tiles of 16 rows x 128 bytes
            uint8_t *phi = pbuf + pb * p_tile_bytes(KVF) + i * kUPTile, *plo = phi + kUPTile / 2;
#pragma unroll
            for (int h = 0; h < kUHeads; h += 2) {
                uint32_t hi, lo;
                split_e4m3x2(pv[h] * kPScale, pv[h + 1] * kPScale, hi, lo);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int hh = h0 + h + k;
                    const uint32_t off = hh * 128 + ((((idx >> 4) ^ (hh & 7))) << 4) + (idx & 15);
                    phi[off] = (uint8_t)(hi >> (8 * k));
                    plo[off] = (uint8_t)(lo >> (8 * k));
                }
            }
        }
    };

    int j = 0, sm_units = 0;
    float unit_scale = p.scale_log2; // logits to base 2 (FP8: / the unit's query scale)
    // Passes of one or two pages of a unit: one max exchange and one P^T
    // hand-off per pass.  One pass past the last task (l0 == ntasks)
    // finishes the last unit, so that finalize has one call site: its code,
    // run once per unit, is fetched once per CTA instead of once per copy.
    for (int l0 = 0; l0 <= ntasks && ok; ++j) {
        const bool end = l0 == ntasks;
        const int np = end ? 0 : pass_len(l0), pb = j & 1;
        int4 e0 = make_int4(-1, 0, 0, 0), e1 = make_int4(-1, 0, 0, 0);
        int u = -2; // no unit: ends the last one
        float sv0[kUHeads], sv1[kUHeads];
        if (!end) {
            for (int i = 0; i < np && ok; ++i) {
                const int l = l0 + i;
                ok = wait_all(smem_u32(&s_full[l % kUSBufs]), (l / kUSBufs) & 1);
            }
            if (!ok)
                break;
            tcgen05_after_sync();
            e0 = entry(l0);
            u = unit_of(e0);
            uint32_t r0[kUHeads], r1[kUHeads];
            if (e0.x >= 0)
                tmem_ld8_nowait(lane_base + 16 * (l0 % kUSBufs), r0);
            if (np == 2) {
                e1 = entry(l0 + 1);
                if (e1.x >= 0)
                    tmem_ld8_nowait(lane_base + 16 * ((l0 + 1) % kUSBufs), r1);
            }
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                sv0[h] = __uint_as_float(r0[h]);
                sv1[h] = __uint_as_float(r1[h]);
            }
            tcgen05_before_sync();
            __syncwarp();
            if (lane == 0)
                for (int i = 0; i < np; ++i)
                    mbar_arrive(smem_u32(&s_free[(l0 + i) % kUSBufs]));
        }
        const bool live0 = e0.x >= 0, live1 = np == 2 && e1.x >= 0;

        if (u != cur_unit) {
            if (cur_unit >= 0) {
                read_o(j - 1); // the unit's passes end with pass j - 1
                if (!ok)
                    break;
                finalize(cur_t, cur_g, end);
                if (!ok)
                    break;
            }
            if (end)
                break;
            cur_unit = u;
            cur_t = e0.z;
            cur_g = e0.w;
            reset();
            {
                const UnitOwn w = own_of(cur_t, cur_g);
                cur_cand = w.c_first == c && w.c_last > c;
            }
            // the producer wrote the unit's query scale before the Q tile it
            // made, which S^T of this page waited for
            if (FP8)
                unit_scale = p.scale_log2 * qscale[sm_units % kUQScales];
            ++sm_units;
        }

        // The last pass of the last unit, begun here and continued later: read
        // the other part now if the producer found it published, so that
        // finalize merges without a round trip.
        if (l0 + np == ntasks && cur_cand) {
            if (!wait_all(smem_u32(last_bar), 0)) {
                ok = false;
                break;
            }
            if (last_chk[0]) {
                const float *sl = p.partial + (size_t)(last_chk[1] + cur_unit) * kPartialFloats;
#pragma unroll
                for (int h = 0; h < kUHeads; ++h) {
                    ms2[h] = __ldcg(sl + kGroup * kDim + h0 + h);
                    ls2[h] = __ldcg(sl + kGroup * kDim + kGroup + h0 + h);
                    os2[h] = __ldcg(sl + (h0 + h) * kDim + idx);
                }
                pre = true;
            }
        }

        // pass maxima per head (log2 domain) across the pages' tokens
        const bool vis0 = live0 && idx < e0.y, vis1 = live1 && idx < e1.y;
        float wmax[kUHeads];
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            sv0[h] = vis0 ? sv0[h] * unit_scale : -INFINITY;
            sv1[h] = vis1 ? sv1[h] * unit_scale : -INFINITY;
            wmax[h] = warp_max_f32(fmaxf(sv0[h], sv1[h]));
        }
        if (lane == 0) {
            float4 *xw = reinterpret_cast<float4 *>(xbuf + (pb * 4 + quarter) * 16 + h0);
            xw[0] = make_float4(wmax[0], wmax[1], wmax[2], wmax[3]);
            xw[1] = make_float4(wmax[4], wmax[5], wmax[6], wmax[7]);
        }
        ssync();
        // The reference of a head moves only when the pass maximum exceeds it
        // by more than the slack; then the denominator and O^T (through the
        // previous pass, in TMEM) are rescaled.  The maxima come from shared
        // memory, so the decision is the same in every thread of a head half.
        constexpr float kSlack = rescale_slack(KVF);
        float m_new[kUHeads];
        bool resc = false;
#pragma unroll
        for (int h4 = 0; h4 < kUHeads / 4; ++h4) {
            float4 a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                a[q] = reinterpret_cast<const float4 *>(xbuf + (pb * 4 + q) * 16 + h0)[h4];
            const float pm[4] = {fmaxf(fmaxf(a[0].x, a[1].x), fmaxf(a[2].x, a[3].x)),
                                 fmaxf(fmaxf(a[0].y, a[1].y), fmaxf(a[2].y, a[3].y)),
                                 fmaxf(fmaxf(a[0].z, a[1].z), fmaxf(a[2].z, a[3].z)),
                                 fmaxf(fmaxf(a[0].w, a[1].w), fmaxf(a[2].w, a[3].w))};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int h = 4 * h4 + k;
                m_new[h] = fmaxf(m_run[h], pm[k]);
                resc = resc || m_new[h] > m_run[h] + kSlack;
            }
        }
        if (resc) {
            float alpha[kUHeads];
#pragma unroll
            for (int h = 0; h < kUHeads; ++h) {
                alpha[h] = 1.f;
                if (m_new[h] > m_run[h] + kSlack) {
                    alpha[h] = ex2(m_run[h] - m_new[h]); // 0 when m_run is -inf
                    m_run[h] = m_new[h];
                }
                lsum[h] *= alpha[h];
            }
            if (o_live) {
                wait_pv(j - 1); // O^T through the previous pass of the unit
                if (!ok)
                    break;
                float v[kUHeads];
                tmem_ld8(lane_base + kUOCol, v);
#pragma unroll
                for (int h = 0; h < kUHeads; ++h)
                    v[h] *= alpha[h];
                tmem_st8(lane_base + kUOCol, v);
            }
        }
        // bf16 P of a single-page unit goes to the MMAs as a hi + lo pair
        const bool hilo0 = KVF == kKvBf16 && np == 1 && qt[e0.z + 1] - qt[e0.z] == 1;
#pragma unroll
        for (int h = 0; h < kUHeads; ++h) {
            const float ref = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
            sv0[h] = ex2(sv0[h] - ref); // P of page 0 (0 where not visible)
            float p1 = 0.f;
            if (pass_pages(KVF) == 2 && np == 2) {
                sv1[h] = ex2(sv1[h] - ref); // P of page 1
                p1 = sv1[h];
            }
            lsum[h] += sv0[h] + p1;
        }
        // P^T of the pass into buffer pb, once the P.V MMAs of pass j - 2 read it
        if (j >= 2 && !wait_all(smem_u32(&p_free[pb]), ((j >> 1) - 1) & 1)) {
            ok = false;
            break;
        }
        if (live0)
            store_p(sv0, pb, 0, hilo0);
        if (live1)
            store_p(sv1, pb, 1, false);
        if (live0 || live1)
            fence_async_smem();
        tcgen05_before_sync(); // a rescaled O^T before the P.V MMAs of this pass
        __syncwarp();
        if (lane == 0)
            mbar_arrive(smem_u32(&p_full[pb]));
        o_live = o_live || live0 || live1;
        l0 += np;
    }
    if (!ok) {
        set_error(p.err, kErrTimeout);
        *abort_flag = 1;
    }
    tcgen05_before_sync();
    __syncwarp();
    if (lane == 0) {
        *smx_done = 1;
        mbar_arrive(smem_u32(done_bar));
    }
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

template <int KVF, int STAGES>
cudaError_t launch_umma_t(const DecodeParams &p, const CUtensorMap &kv, const CUtensorMap &qm,
                          int ctas, cudaStream_t stream, bool pdl)
{
    const size_t smem = umma_layout(p.T, STAGES, KVF).total;
    cudaError_t e = cudaFuncSetAttribute(sparse_decode_umma_kernel<KVF, STAGES>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    if (KVF == kKvNvfp4) {
        // The NVFP4 instance moves registers between its warpgroups
        // (setmaxnreg); a raise waits until the lowerings have freed enough
        // of the launch allocation, so the split must fit in it: never
        // launch an instance built with fewer registers a thread.
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, sparse_decode_umma_kernel<KVF, STAGES>)) != cudaSuccess)
            return e;
        if ((long long)fa.numRegs * kUThreadsT<KVF> <
            128ll * kURegsWg0 + 32ll * kUSmxWarps * kURegsSmx + 32ll * kUCvtWarps * kURegsCvt)
            return cudaErrorInvalidConfiguration;
    }
    e = launch_kernel(sparse_decode_umma_kernel<KVF, STAGES>, dim3(ctas), dim3(kUThreadsT<KVF>), smem,
                      stream, pdl, kv, qm, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace

bool encode_2d_sw128(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows)
{
    EncodeFn enc = get_encode();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_sparse_decode(const DecodeParams &p, const void *kv_pool, int kv_dtype, int ctas,
                                 cudaStream_t stream, bool pdl)
{
    CUtensorMap map;
    std::memset(&map, 0, sizeof(map)); // NVFP4 tiles move by bulk copies: no KV tensor map
    if (kv_dtype != MSA_NVFP4 && !encode_kv_map(&map, kv_pool, kv_dtype, p.num_pages, p.Hkv))
        return cudaErrorInvalidValue;
    CUtensorMap qmap;
    if (!encode_q_map(&qmap, p.q, p.T, p.Hkv))
        return cudaErrorInvalidValue;
    DecodeParams q = p;
    q.kv_raw = static_cast<const uint8_t *>(kv_pool);
    if (kv_dtype == MSA_NVFP4) {
        if (umma_layout(p.T, 8, kKvNvfp4).total <= (size_t)kMaxSmem)
            return launch_umma_t<kKvNvfp4, 8>(q, map, qmap, ctas, stream, pdl);
        return launch_umma_t<kKvNvfp4, 4>(q, map, qmap, ctas, stream, pdl);
    }
    if (kv_dtype == MSA_FP8_E4M3) {
        if (umma_layout(p.T, 12, kKvFp8).total <= (size_t)kMaxSmem)
            return launch_umma_t<kKvFp8, 12>(q, map, qmap, ctas, stream, pdl);
        return launch_umma_t<kKvFp8, 6>(q, map, qmap, ctas, stream, pdl);
    }
    if (umma_layout(p.T, 6, kKvBf16).total <= (size_t)kMaxSmem)
        return launch_umma_t<kKvBf16, 6>(q, map, qmap, ctas, stream, pdl);
    return launch_umma_t<kKvBf16, 4>(q, map, qmap, ctas, stream, pdl);
}

} // namespace msa
