// msa_noalloc.cu -- msa_sparse_decode_noalloc: the sparse decode for callers
// that cannot allocate device memory.
//
// Some hosts of this library have no way to hand it a workspace: a plugin
// that is given only its input and output tensors by the runtime that owns
// all device memory, code whose allocator may not be called on the path
// that issues the decode, or a deployment that forbids run-time cudaMalloc
// altogether.  For them this entry point keeps the decode's scratch (the
// split partials, their arrival counters and the device error word) in a fixed array compiled into
// the library.  The array lives in every GPU's memory from the moment the
// library is loaded on it until the process exits.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
//
// The kernels are exactly those of msa_sparse_decode; only where their
// scratch lives differs.
#include "msa_internal.cuh"

namespace msa {
namespace {

// Device scratch: [0, 256) error word, then one arrival counter per
// (token, KV head) unit, then the decode's partial slots.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MSA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the current device's context.  In
// host code the array's name only stands in for the symbol; the address the
// kernels need comes from cudaGetSymbolAddress, asked on every call (a cheap
// lookup once the module is loaded) so that it is always the address in the
// context that is current now, also after a cudaDeviceReset.
void *scratch_address()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess)
        return nullptr;
    return p;
}

int sm_count(int dev)
{
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    return n;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

} // namespace
} // namespace msa

using namespace msa;

extern "C" msa_status msa_sparse_decode_noalloc(const msa_shape *shape, const void *q,
                                                const void *kv_pool, const int32_t *block_table,
                                                const int32_t *seq_lens, const int32_t *selected,
                                                void *out, float *lse, cudaStream_t stream)
{
    // the shape rules of every other entry point, with their status
    const msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if (!q || !kv_pool || !block_table || !seq_lens || !selected || !out || !lse)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(block_table) || !aligned16(seq_lens) ||
        !aligned16(selected) || !aligned16(out) || !aligned16(lse))
        return MSA_ERR_INVALID_ARGUMENT;
    const int T = shape->num_requests * shape->q_per_req;
    if (T == 0)
        return MSA_OK;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MSA_ERR_CUDA;
    int ctas = shape->decode_ctas;
    if (ctas == 0) {
        ctas = sm_count(dev);
        if (ctas < 1)
            return MSA_ERR_CUDA;
        const long long max_tasks = (long long)T * shape->num_kv_heads * shape->topk;
        if (ctas > max_tasks)
            ctas = (int)max_tasks;
    }
    // scratch needed: error word, one arrival counter per unit (rounded up to
    // 256 bytes), one partial slot per (CTA + unit)
    const long long units = (long long)T * shape->num_kv_heads;
    const long long head = 256 + (units * 4 + 255) / 256 * 256;
    const long long slots = (long long)ctas + units;
    if (head + slots * (long long)kPartialBytes > (long long)MSA_NOALLOC_SCRATCH_BYTES)
        return MSA_ERR_UNSUPPORTED; // too big for the fixed scratch: use msa_sparse_decode
    // The decode cuts its P <= units * topk tasks into ctas ranges in 32-bit
    // arithmetic (P (ctas + 1) < 2^32); the fixed scratch bounds ctas + units
    // far below what could break that.
    static_assert((unsigned long long)(MSA_NOALLOC_SCRATCH_BYTES / kPartialBytes) * kMaxTopk *
                          (MSA_NOALLOC_SCRATCH_BYTES / kPartialBytes + 1) <
                      (1ull << 32),
                  "fixed scratch admits task ranges beyond 32 bits");

    unsigned char *scratch = static_cast<unsigned char *>(scratch_address());
    if (!scratch)
        return MSA_ERR_CUDA;
    // the error word and the arrival counters must start at zero; the partial
    // slots are written before they are read
    if (cudaMemsetAsync(scratch, 0, (size_t)head, stream) != cudaSuccess)
        return MSA_ERR_CUDA;

    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.selected = selected;
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.partial = reinterpret_cast<float *>(scratch + head);
    p.counters = reinterpret_cast<int *>(scratch + 256);
    p.err = reinterpret_cast<uint32_t *>(scratch);
    p.R = shape->num_requests;
    p.nq = shape->q_per_req;
    p.T = T;
    p.Hkv = shape->num_kv_heads;
    p.maxB = shape->max_blocks_per_seq;
    p.k = shape->topk;
    p.num_pages = shape->num_pages;
    p.Hs = shape->num_index_heads == 1 ? 1 : shape->num_kv_heads; // tables per token
    const bool scaled = shape->kv_dtype != MSA_BF16; // E4M3 and NVFP4 carry tensor scales
    p.scale_log2 = shape->softmax_scale * 1.4426950408889634f * (scaled ? shape->k_scale : 1.f);
    p.v_scale = scaled ? shape->v_scale : 1.f;
    // slots the array holds after the head (the kernel checks every slot it
    // touches against it, so no problem can write past the array)
    p.slots = ((long long)MSA_NOALLOC_SCRATCH_BYTES - head) / (long long)kPartialBytes;
    p.wait_limit = decode_wait_limit();
    return launch_sparse_decode(p, kv_pool, shape->kv_dtype, ctas, stream, false) == cudaSuccess
               ? MSA_OK
               : MSA_ERR_CUDA;
}
