// msa_update.cu -- the KV / index-key update: this step's new keys, values
// and index keys written into their pages through the block table, before
// the step scores and attends.
//
// "MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2 for
// Blackwell", section "The TP4 decode target": the attention megakernels
// carry "the KV update"; "Add Rubin (sm_107) MiniMax-M3.1 low-latency decode
// targets", q8kv4 indexer commit: the NVFP4 index-K copy is "refreshed from
// this step's slots".  The library's definitions where the pages are silent:
//   - new token j of request r sits at position seq_lens[r] - 1 + j (the last
//     position it sees): row pos % 128 of page block_table[r][pos / 128];
//   - FP8 K / V: E4M3 of x / k_scale (x / v_scale), round to nearest even,
//     saturating at 448, the quotient in binary32;
//   - NVFP4 index keys, per 16 consecutive dimensions: scale code E4M3 of
//     amax / 6, element codes e2m1 of x / scale (0 when the scale is 0), both
//     round to nearest even and saturating, quotients in binary32, no
//     second-level scale;
//   - a code that rounds to zero is stored as +0.
//
// The work is 256 bytes per (token, row) -- rows are K and V of each KV head
// and the index key of each index head -- and bound by launch latency: one
// warp per row, 4 elements (8 input bytes) per lane, the NVFP4 group of 16
// across 4 lanes.
#include "msa_internal.cuh"

namespace msa {
namespace {

constexpr int kUpdWarps = 8;

// Two floats to E4M3 codes (round to nearest even, saturating): a -> high
// byte, b -> low byte; a zero result is +0.
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float a, float b)
{
    uint32_t out;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}\n"
        : "=r"(out)
        : "f"(a), "f"(b));
    if ((out & 0x7Fu) == 0)
        out &= ~0x80u;
    if ((out & 0x7F00u) == 0)
        out &= ~0x8000u;
    return out;
}

// Four floats to e2m1 codes (round to nearest even, saturating) packed in 16
// bits, x0 in the lowest nibble; a zero result is +0.
__device__ __forceinline__ uint32_t e2m1x4_rn_sat(float x0, float x1, float x2, float x3)
{
    uint32_t out;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, 0f00000000, 0f00000000;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, 0f00000000, 0f00000000;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}\n"
        : "=r"(out)
        : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (((out >> (4 * i)) & 7u) == 0)
            out &= ~(8u << (4 * i));
    return out;
}

constexpr int kF4KvTile = kPage * kDim / 2 + kPage * kDim / 16; // NVFP4 K or V tile

// One row of 128 bf16 values as NVFP4, warp-wide: lane holds elements
// 4 lane .. + 3 (v), divides them by `scale`, and writes its 4 codes (2
// bytes at codes + 2 lane); the group of 16 = lanes 4 q .. 4 q + 3 shares
// one E4M3 scale, written by lane 4 q at scales[q].
__device__ __forceinline__ void nvfp4_quad(uint2 v, float scale, uint8_t *codes, uint8_t *scales)
{
    const int lane = threadIdx.x & 31;
    const float x0 = __fdiv_rn(__uint_as_float(v.x << 16), scale);
    const float x1 = __fdiv_rn(__uint_as_float(v.x & 0xFFFF0000u), scale);
    const float x2 = __fdiv_rn(__uint_as_float(v.y << 16), scale);
    const float x3 = __fdiv_rn(__uint_as_float(v.y & 0xFFFF0000u), scale);
    float amax = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint32_t sc = e4m3x2_rn_sat(0.f, __fdiv_rn(amax, 6.f)) & 0xFFu;
    float S, unused;
    f16x2_to_f32x2(e4m3x2_to_f16x2(sc), S, unused);
    uint32_t c = 0;
    if (S > 0.f)
        c = e2m1x4_rn_sat(__fdiv_rn(x0, S), __fdiv_rn(x1, S), __fdiv_rn(x2, S), __fdiv_rn(x3, S));
    *reinterpret_cast<uint16_t *>(codes + 2 * lane) = (uint16_t)c;
    if ((lane & 3) == 0)
        scales[lane >> 2] = (uint8_t)sc;
}

__global__ void __launch_bounds__(32 * kUpdWarps) kv_update_kernel(const UpdateParams p)
{
    const int lane = threadIdx.x & 31;
    const int rows = 2 * p.Hkv + p.Hi; // K of each KV head, V of each, index key of each index head
    const long long x = (long long)blockIdx.x * kUpdWarps + (threadIdx.x >> 5);
    const int T = p.R * p.nq;
    if (x >= (long long)T * rows)
        return;
    const int t = (int)(x / rows), kind = (int)(x - (long long)t * rows);
    const int r = t / p.nq, j = t - r * p.nq;
    const int seq_len = p.seq_lens[r];
    const long long nb = ((long long)seq_len + p.nq - 1 + kPage - 1) / kPage;
    if (seq_len < 1 || nb > p.maxB) {
        if (lane == 0)
            set_error(p.err, kErrSeqLen);
        return;
    }
    const int pos = seq_len - 1 + j;
    const long long page = p.block_table[(size_t)r * p.maxB + pos / kPage];
    if (page < 0 || page >= p.num_pages) {
        if (lane == 0)
            set_error(p.err, kErrPage);
        return;
    }
    const int row = pos % kPage;

    if (kind < 2 * p.Hkv) {
        const int kv = kind / p.Hkv, g = kind - kv * p.Hkv;
        const uint16_t *src = (kv ? p.v_new : p.k_new) + ((size_t)t * p.Hkv + g) * kDim;
        const uint2 v = reinterpret_cast<const uint2 *>(src)[lane]; // elements 4 lane .. + 3
        if (p.kv_nvfp4) { // the tile of (page, K/V, head g): codes [P][64], then scales [P][8]
            uint8_t *tile = p.kv_pool + (((size_t)page * 2 + kv) * p.Hkv + g) * kF4KvTile;
            const float s = kv ? p.v_scale : p.k_scale;
            nvfp4_quad(v, s, tile + (size_t)row * (kDim / 2), tile + (size_t)kPage * (kDim / 2) +
                                                                  (size_t)row * (kDim / 16));
            return;
        }
        const size_t elem = (((size_t)page * 2 + kv) * p.Hkv + g) * (size_t)kPage * kDim +
                            (size_t)row * kDim + 4 * lane;
        if (!p.kv_fp8) {
            *reinterpret_cast<uint2 *>(p.kv_pool + elem * 2) = v;
        } else {
            const float s = kv ? p.v_scale : p.k_scale;
            const float x0 = __fdiv_rn(__uint_as_float(v.x << 16), s);
            const float x1 = __fdiv_rn(__uint_as_float(v.x & 0xFFFF0000u), s);
            const float x2 = __fdiv_rn(__uint_as_float(v.y << 16), s);
            const float x3 = __fdiv_rn(__uint_as_float(v.y & 0xFFFF0000u), s);
            const uint32_t c = e4m3x2_rn_sat(x1, x0) | (e4m3x2_rn_sat(x3, x2) << 16);
            *reinterpret_cast<uint32_t *>(p.kv_pool + elem) = c;
        }
        return;
    }
    const int i = kind - 2 * p.Hkv;
    const uint16_t *src = p.idxk_new + ((size_t)t * p.Hi + i) * kDim;
    const uint2 v = reinterpret_cast<const uint2 *>(src)[lane];
    const size_t prow = ((size_t)page * p.Hi + i) * kPage + row;
    if (!p.idx_nvfp4) {
        *reinterpret_cast<uint2 *>(p.idxk_pool + prow * (kDim * 2) + 8 * lane) = v;
        return;
    }
    nvfp4_quad(v, 1.f, p.idxk_pool + prow * (kDim / 2), p.idxk_scales + prow * (kDim / 16));
}

} // namespace

cudaError_t launch_kv_update(const UpdateParams &p, cudaStream_t stream)
{
    const long long rows = (long long)p.R * p.nq * (2 * p.Hkv + p.Hi);
    if (rows == 0)
        return cudaSuccess;
    const dim3 grid((unsigned)((rows + kUpdWarps - 1) / kUpdWarps)), block(32 * kUpdWarps);
    const cudaError_t e = launch_kernel(kv_update_kernel, grid, block, 0, stream, false, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

} // namespace msa
