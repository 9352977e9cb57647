// msa_internal.cuh -- shared definitions of the kernels and the C-ABI layer.
//
// Device helpers are thin inline-PTX wrappers around sm_90+/sm_100 family
// instructions (mbarrier, cp.async.bulk.tensor, ldmatrix, mma.sync,
// packed fp8/fp4 converts).  Nothing here is a math-library routine.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "msa.h"

namespace msa {

constexpr int kPage = 128;       // tokens per page (P128)
constexpr int kDim = 128;        // head_dim and index_dim
constexpr int kGroup = 16;       // query heads per KV head
constexpr int kMaxTokens = 8192; // T = R * q_per_req
constexpr int kMaxBlocks = 16384;
constexpr int kMaxTopk = 256;
constexpr int kMaxQPerReq = 64;
constexpr int kMaxRequests = 8192;
constexpr int kMaxIndexHeads = 64;
constexpr int kMaxRows = 1 << 22;      // rows of one msa_select_rows call
constexpr int kDefaultCtaBound = 1024; // workspace bound on default persistent decode CTAs

// Bits of the workspace error word.
enum : uint32_t {
    kErrPage = 1u,      // block table entry outside [0, num_pages)
    kErrSeqLen = 2u,    // seq_len < 1, or cached blocks > max_blocks_per_seq
    kErrSelection = 4u, // selected block id not a visible block of the token
    kErrTimeout = 8u,   // a bounded wait ran out
    kErrScratch = 16u,  // a decode partial slot or arrival counter outside the scratch given
};

// SM clocks after which a bounded wait gives up (about a second).
constexpr long long kWaitLimit = 1ll << 31;

// Bytes of one decode partial: o[16][128] then m[16], l[16] (fp32).
constexpr size_t kPartialFloats = size_t(kGroup) * kDim + 2 * kGroup;
constexpr size_t kPartialBytes = kPartialFloats * sizeof(float);

struct WorkspaceLayout {
    size_t counters_off; // int32 [T * Hkv]: split-arrival counters of the decode (kept at 0)
    size_t scores_off;   // fp32 [T][maxB] (decode_step when block_scores == NULL)
    size_t selected_off; // int32 [T][k]   (decode_step when selected == NULL)
    size_t partial_off;  // decode partial slots
    int64_t slots;
    size_t total;
};

// One index head `head` of `heads`: its query row of token t is
// q_idx + (t * heads + head) * Di, the keys of page pg sit at page row
// pg * heads + head of the pool, its block scores at row t * heads + head.
struct ScoreParams {
    const uint16_t *q_idx;  // bf16 bits [T][heads][Di]
    const uint8_t *idxk;    // bf16 [pages][heads][P][Di] or nvfp4 bytes [pages][heads][P][Di/2]
    const uint8_t *scales;  // E4M3 [pages][heads][P][Di/16] (nvfp4)
    const int32_t *block_table;
    const int32_t *seq_lens;
    float *block_scores;    // [T][heads][maxB]
    uint32_t *err;
    int R, nq, maxB, num_pages;
    int heads, head;
};

// Rows x = t * Hs + gs: selection head gs of token t reads the block scores
// of index heads gs * (Hi / Hs) .. (gs + 1) * (Hi / Hs) - 1 (their maximum)
// and keeps the first `init` and the last `local` visible blocks.
struct SelectParams {
    const float *block_scores; // [T][Hi][maxB]
    const int32_t *seq_lens;
    int32_t *selected;         // [T][Hs][k]
    uint32_t *err;
    int R, nq, maxB, k;
    int Hi, Hs, init, local;
    int r; // index heads per selection head: Hi / Hs
};

struct DecodeParams {
    const uint16_t *q; // bf16 bits [T][Hq][D]
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *selected; // [T][Hs][k]: one table per token (Hs = 1) or per KV head (Hs = Hkv)
    const uint8_t *kv_raw;   // the KV pool (read by bulk copies for NVFP4 tiles)
    uint16_t *out;           // bf16 bits [T][Hq][D]
    float *lse;              // [T][Hq]
    float *partial;          // slots of kPartialFloats
    int *counters;           // [T * Hkv], zero between calls
    uint32_t *err;
    int R, nq, T, Hkv, maxB, k, num_pages, Hs;
    float scale_log2; // softmax_scale * log2(e) (* k_scale for FP8 keys)
    float v_scale;    // 1 for bf16 values
    long long slots;  // partial slots in `partial` (slot c + u of CTA c and unit u is checked)
    long long wait_limit; // SM clocks of the decode's bounded waits (kWaitLimit unless testing)
};

// The decode's wait limit for the calls that follow (msa_set_decode_wait_limit).
long long decode_wait_limit();

// Shape checks of every entry point (MSA_OK, MSA_ERR_INVALID_ARGUMENT or
// MSA_ERR_UNSUPPORTED); many_rows: the row select, whose rows per request are
// not limited by the decode's and scorer's tiles.
msa_status check_shape(const msa_shape *s, bool many_rows = false);

// This step's new tokens written into their pages (the KV / index-key update).
struct UpdateParams {
    const uint16_t *k_new;    // bf16 bits [T][Hkv][D]
    const uint16_t *v_new;    // bf16 bits [T][Hkv][D]
    const uint16_t *idxk_new; // bf16 bits [T][Hi][Di]
    const int32_t *block_table;
    const int32_t *seq_lens;
    uint8_t *kv_pool;         // [pages][2][Hkv][P][D] bf16 or E4M3, or NVFP4 tiles [pages][2][Hkv][9216]
    uint8_t *idxk_pool;       // [pages][Hi][P][Di] bf16, or [pages][Hi][P][Di/2] e2m1 pairs
    uint8_t *idxk_scales;     // NVFP4: E4M3 [pages][Hi][P][Di/16]
    uint32_t *err;
    int R, nq, Hkv, Hi, maxB, num_pages;
    bool kv_fp8, kv_nvfp4, idx_nvfp4;
    float k_scale, v_scale;
};

// Host launchers (return the first CUDA error of the launch sequence).  With
// `pdl` the kernel is launched as a programmatic dependent of the previous
// kernel in the stream (it runs its prologue early and waits on the grid
// dependency before reading that kernel's outputs); only kernels of the same
// call are chained this way.
cudaError_t launch_index_score(const ScoreParams &p, int index_dtype, int num_sms,
                               cudaStream_t stream);
cudaError_t launch_select(const SelectParams &p, cudaStream_t stream, bool pdl);
cudaError_t launch_sparse_decode(const DecodeParams &p, const void *kv_pool, int kv_dtype,
                                 int ctas, cudaStream_t stream, bool pdl);
cudaError_t launch_kv_update(const UpdateParams &p, cudaStream_t stream);
// Tables of many rows from a head-major score buffer [Hs][maxB][T] (maxB <= 2048).
constexpr int kMaxRowSelectBlocks = 2048;
cudaError_t launch_select_rows(const SelectParams &p, cudaStream_t stream);

__host__ __device__ constexpr size_t align_to(size_t v, size_t a)
{
    return (v + a - 1) / a * a;
}

// Tensor map of a row-major 2-D array [rows][inner] (row pitch `row_bytes`)
// loaded in boxes of box_inner x box_rows with the 128-byte swizzle; false if
// the driver's encoder is unavailable or rejects the map.
bool encode_2d_sw128(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t inner,
                     uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);

// cudaLaunchKernelEx with an optional programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args &&...args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// device helpers

#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_error(uint32_t *err, uint32_t bits)
{
    atomicOr(err, bits);
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Test for the completion of phase `parity`, suspending the thread for the
// hardware's own time limit while it is incomplete (a longer suspend hint,
// 1 ms, measured 1-2.5% slower on every workload: the wake-up of a thread
// whose phase completed lags).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier; false if it did not complete
// within kWaitLimit SM clocks (about a second).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - start > kWaitLimit)
            return false;
    }
    return true;
}

// Like mbar_wait_bounded, but also gives up as soon as *abort_flag is set
// (another thread of the CTA already timed out), and after `limit` clocks.
__device__ __forceinline__ bool mbar_wait_or_abort(uint32_t bar, uint32_t parity,
                                                   const volatile int *abort_flag,
                                                   long long limit = kWaitLimit)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long start = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag || clock64() - start > limit)
            return false;
    }
    return true;
}

// atomicAdd with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int *addr, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// Load with acquire semantics at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int *addr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

// ---- register reallocation between warpgroups ------------------------------

// Raise / lower the registers a thread of this warpgroup holds to N (all
// four warps of the warpgroup execute it).  A raise waits until other
// warpgroups' lowerings have freed enough of the CTA's launch allocation.
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---- programmatic dependent launch ----------------------------------------

// Block until the kernels this grid depends on have completed and their
// writes are visible (a no-op without a programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next kernel in the stream to be scheduled now.
__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- TMA ------------------------------------------------------------------

// 1-D bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes,
                                               uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// L2 policy for data read once: evicted before any line without the hint, so
// a stream of pages does not push the kernel's code, tables and reused lines
// out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y,
                                                 uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- ldmatrix / mma -------------------------------------------------------

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, f16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ---- tcgen05: tensor memory and the 5th-generation MMA ------------------------

// Allocate `ncols` (power of two >= 32) TMEM columns; the base address is
// written to shared memory at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tcgen05_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tcgen05_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA, tcgen05.mma operands).
__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a tcgen05.mma operand: start address,
// leading and stride byte offsets (in 16-byte units), descriptor version 1,
// 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t smem_addr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46; // descriptor version
    d |= (uint64_t)2 << 61; // SWIZZLE_128B
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: bf16 A and B, fp32 D,
// M x N tile, A / B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, int a_mn, int b_mn)
{
    return (1u << 4)                       // D: F32
           | (1u << 7)                     // A: BF16
           | (1u << 10)                    // B: BF16
           | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16)
           | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem] * B[smem], 8-bit operands (kind::f8f6f4), issued by one thread.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread
// issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (warp-wide).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Maximum of a float over the warp (every lane gets it).
__device__ __forceinline__ float warp_max_f32(float x)
{
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

// ---- conversions ------------------------------------------------------------

// Two E4M3 codes (low byte -> low half) to f16x2.  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes)
{
    uint32_t out;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(out)
        : "r"(two_codes));
    return out;
}

// Four E4M3 codes (bytes 0..3 of w) to two f16x2 words: lo = bytes 0, 1 and
// hi = bytes 2, 3 (lower byte in the lower half).  Exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.rn.f16x2.e4m3x2 %0, a;\n"
        " cvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// f16x2 to two floats (lo = lower half).  Exact.
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t v, float &lo, float &hi)
{
    asm("{\n .reg .b16 a, b;\n mov.b32 {a, b}, %2;\n cvt.f32.f16 %0, a;\n cvt.f32.f16 %1, b;\n}\n"
        : "=f"(lo), "=f"(hi)
        : "r"(v));
}

// Two E2M1 codes in one byte (low nibble -> low half) to f16x2.  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte)
{
    uint32_t out;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
        : "=r"(out)
        : "r"(byte));
    return out;
}

// Eight e2m1 codes (one 32-bit word, byte k = codes 2k (low nibble) and
// 2k + 1) times an f16x2 scale pair: out[k] = f16x2 of the two codes of byte
// k, each multiplied by s2.  Exact when the products fit f16.
__device__ __forceinline__ void e2m1x8_scaled_f16x2(uint32_t word, uint32_t s2, uint32_t (&out)[4])
{
    asm("{\n .reg .b8 b0, b1, b2, b3;\n .reg .b32 h0, h1, h2, h3;\n"
        " mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 h0, b0;\n cvt.rn.f16x2.e2m1x2 h1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 h2, b2;\n cvt.rn.f16x2.e2m1x2 h3, b3;\n"
        " mul.rn.f16x2 %0, h0, %5;\n mul.rn.f16x2 %1, h1, %5;\n"
        " mul.rn.f16x2 %2, h2, %5;\n mul.rn.f16x2 %3, h3, %5;\n}\n"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(word), "r"(s2));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// f32 pair -> bf16x2 (lo from `lo`), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// f32 pair -> f16x2 (lo from `lo`), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// bf16x2 -> f16x2 via f32 (exact for values representable in both).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v)
{
    float lo = __uint_as_float(v << 16);
    float hi = __uint_as_float(v & 0xFFFF0000u);
    return pack_f16(lo, hi);
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Monotone map of a float's bits to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) // -0 equals +0: one key, so the tie goes by block index
        u = 0u;
    return u ^ ((u >> 31) ? 0xFFFFFFFFu : 0x80000000u);
}

__device__ __forceinline__ int ceil_div(int a, int b)
{
    return (a + b - 1) / b;
}

#endif // __CUDACC__

} // namespace msa
