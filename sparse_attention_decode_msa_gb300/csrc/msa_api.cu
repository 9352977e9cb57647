// msa_api.cu -- the C ABI of include/msa.h: host-side validation, workspace
// layout and the launch sequence.  No allocation, no global state beyond the
// per-device SM count and the driver entry point used to encode tensor maps.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "msa_internal.cuh"

namespace msa {

// Clock limit of the decode's bounded waits (changed only by the test hook
// msa_set_decode_wait_limit).
std::atomic<long long> g_decode_wait_limit{kWaitLimit};

long long decode_wait_limit()
{
    return g_decode_wait_limit.load(std::memory_order_relaxed);
}

// Shape checks shared by every entry point.  many_rows: the row select, whose
// rows per request are not limited by the decode's and scorer's tiles.
msa_status check_shape(const msa_shape *s, bool many_rows)
{
    if (!s)
        return MSA_ERR_INVALID_ARGUMENT;
    if (s->num_requests < 0 || s->q_per_req < 1 || s->num_kv_heads < 1 || s->num_pages < 1 ||
        s->max_blocks_per_seq < 1 || s->topk < 1 || s->decode_ctas < 0)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(s->softmax_scale) || !std::isfinite(s->k_scale) ||
        !std::isfinite(s->v_scale))
        return MSA_ERR_INVALID_ARGUMENT;
    if (s->num_index_heads < 1 || s->init_blocks < 0 || s->local_blocks < 0 ||
        (long long)s->init_blocks + s->local_blocks > s->topk)
        return MSA_ERR_INVALID_ARGUMENT;
    if (s->head_dim != kDim || s->index_dim != kDim || s->page_size != kPage ||
        s->num_q_heads != kGroup * s->num_kv_heads)
        return MSA_ERR_UNSUPPORTED;
    // one index head (one table per token) or a whole number per KV head
    if (s->num_index_heads > kMaxIndexHeads ||
        (s->num_index_heads > 1 && s->num_index_heads % s->num_kv_heads != 0))
        return MSA_ERR_UNSUPPORTED;
    if (!many_rows && (s->q_per_req > kMaxQPerReq ||
                       (long long)s->num_requests * s->q_per_req > kMaxTokens))
        return MSA_ERR_UNSUPPORTED;
    if (many_rows && (long long)s->num_requests * s->q_per_req > kMaxRows)
        return MSA_ERR_UNSUPPORTED;
    if (s->topk > kMaxTopk || s->max_blocks_per_seq > kMaxBlocks || s->num_requests > kMaxRequests)
        return MSA_ERR_UNSUPPORTED;
    if (s->kv_dtype != MSA_BF16 && s->kv_dtype != MSA_FP8_E4M3 && s->kv_dtype != MSA_NVFP4)
        return MSA_ERR_UNSUPPORTED;
    if (s->index_dtype != MSA_BF16 && s->index_dtype != MSA_NVFP4)
        return MSA_ERR_UNSUPPORTED;
    // page row indices of the KV and index-key tensor maps must fit in int32
    if ((long long)s->num_pages * 2 * s->num_kv_heads * kPage > 0x7FFFFFFFll ||
        (long long)s->num_pages * s->num_index_heads * kPage > 0x7FFFFFFFll)
        return MSA_ERR_UNSUPPORTED;
    return MSA_OK;
}

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v)
{
    return (v + kAlign - 1) / kAlign * kAlign;
}

bool aligned16(const void *p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int tokens_of(const msa_shape *s)
{
    return s->num_requests * s->q_per_req;
}

// Selection tables per token: one shared by every KV head with one index
// head, else one per KV head.
int selection_heads(const msa_shape *s)
{
    return s->num_index_heads == 1 ? 1 : s->num_kv_heads;
}

int cta_bound(const msa_shape *s)
{
    return s->decode_ctas > 0 ? s->decode_ctas : kDefaultCtaBound;
}

WorkspaceLayout layout_of(const msa_shape *s)
{
    const size_t T = (size_t)tokens_of(s);
    WorkspaceLayout w;
    size_t off = kAlign; // error word
    w.counters_off = off;
    off = align_up(off + T * s->num_kv_heads * sizeof(int32_t));
    w.scores_off = off;
    off = align_up(off + T * s->num_index_heads * s->max_blocks_per_seq * sizeof(float));
    w.selected_off = off;
    off = align_up(off + T * selection_heads(s) * s->topk * sizeof(int32_t));
    w.partial_off = off;
    w.slots = (int64_t)cta_bound(s) + (int64_t)T * s->num_kv_heads;
    off = align_up(off + (size_t)w.slots * kPartialBytes);
    w.total = off;
    return w;
}

int num_sms_current()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cached[dev] > 0)
        return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -1;
    if (dev >= 0 && dev < 64)
        cached[dev] = n;
    return n;
}

msa_status check_workspace(const msa_shape *s, const void *ws, size_t bytes)
{
    if (!ws || !aligned16(ws))
        return MSA_ERR_INVALID_ARGUMENT;
    if (bytes < layout_of(s).total)
        return MSA_ERR_INVALID_ARGUMENT;
    return MSA_OK;
}

msa_status cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status score_impl(const msa_shape *s, const void *q_idx, const void *idxk_pool,
                      const void *idxk_scales, const int32_t *block_table,
                      const int32_t *seq_lens, float *block_scores, void *ws, cudaStream_t stream)
{
    ScoreParams p;
    p.q_idx = static_cast<const uint16_t *>(q_idx);
    p.idxk = static_cast<const uint8_t *>(idxk_pool);
    p.scales = static_cast<const uint8_t *>(idxk_scales);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.block_scores = block_scores;
    p.err = static_cast<uint32_t *>(ws);
    p.R = s->num_requests;
    p.nq = s->q_per_req;
    p.maxB = s->max_blocks_per_seq;
    p.num_pages = s->num_pages;
    p.heads = s->num_index_heads;
    const int sms = num_sms_current();
    if (sms < 1)
        return MSA_ERR_CUDA;
    // one pass of the scorer per index head
    for (int h = 0; h < p.heads; ++h) {
        p.head = h;
        const cudaError_t e = launch_index_score(p, s->index_dtype, sms, stream);
        if (e != cudaSuccess)
            return MSA_ERR_CUDA;
    }
    return MSA_OK;
}

msa_status select_impl(const msa_shape *s, const float *block_scores, const int32_t *seq_lens,
                       int32_t *selected, void *ws, cudaStream_t stream, bool pdl)
{
    SelectParams p;
    p.block_scores = block_scores;
    p.seq_lens = seq_lens;
    p.selected = selected;
    p.err = static_cast<uint32_t *>(ws);
    p.R = s->num_requests;
    p.nq = s->q_per_req;
    p.maxB = s->max_blocks_per_seq;
    p.k = s->topk;
    p.Hi = s->num_index_heads;
    p.Hs = selection_heads(s);
    p.r = p.Hi / p.Hs;
    p.init = s->init_blocks;
    p.local = s->local_blocks;
    return cuda_status(launch_select(p, stream, pdl));
}

// Persistent CTAs of the decode: the shape's, else one per SM (at most the
// workspace bound and the number of tasks); -1 if the device cannot be read.
int decode_ctas(const msa_shape *s)
{
    int ctas = s->decode_ctas;
    if (ctas == 0) {
        const int sms = num_sms_current();
        if (sms < 1)
            return -1;
        ctas = sms < kDefaultCtaBound ? sms : kDefaultCtaBound;
        const long long max_tasks = (long long)tokens_of(s) * s->num_kv_heads * s->topk;
        if (ctas > max_tasks)
            ctas = (int)max_tasks;
    }
    return ctas;
}

msa_status decode_impl(const msa_shape *s, const void *q, const void *kv_pool,
                       const int32_t *block_table, const int32_t *seq_lens,
                       const int32_t *selected, void *out, float *lse, void *ws,
                       cudaStream_t stream, bool pdl)
{
    const WorkspaceLayout w = layout_of(s);
    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.selected = selected;
    p.out = static_cast<uint16_t *>(out);
    p.lse = lse;
    p.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + w.partial_off);
    p.counters = reinterpret_cast<int *>(static_cast<uint8_t *>(ws) + w.counters_off);
    p.err = static_cast<uint32_t *>(ws);
    p.R = s->num_requests;
    p.nq = s->q_per_req;
    p.T = tokens_of(s);
    p.Hkv = s->num_kv_heads;
    p.maxB = s->max_blocks_per_seq;
    p.k = s->topk;
    p.num_pages = s->num_pages;
    p.Hs = selection_heads(s);
    const bool scaled = s->kv_dtype != MSA_BF16; // E4M3 and NVFP4 carry tensor scales
    p.scale_log2 = s->softmax_scale * 1.4426950408889634f * (scaled ? s->k_scale : 1.f);
    p.v_scale = scaled ? s->v_scale : 1.f;
    p.slots = w.slots;
    p.wait_limit = decode_wait_limit();
    const int ctas = decode_ctas(s);
    if (ctas < 1)
        return MSA_ERR_CUDA;
    return cuda_status(launch_sparse_decode(p, kv_pool, s->kv_dtype, ctas, stream, pdl));
}

// The decode cuts its P <= T * Hkv * k tasks into G ranges in 32-bit
// arithmetic: calls with P (G + 1) >= 2^32 are not taken.
msa_status check_decode_size(const msa_shape *s)
{
    const int ctas = decode_ctas(s);
    if (ctas < 1)
        return MSA_ERR_CUDA;
    const long long bound = (long long)tokens_of(s) * s->num_kv_heads * s->topk;
    return bound * (ctas + 1) < (1ll << 32) ? MSA_OK : MSA_ERR_UNSUPPORTED;
}

} // namespace
} // namespace msa

using namespace msa;

extern "C" {

size_t msa_workspace_bytes(const msa_shape *shape)
{
    if (check_shape(shape) != MSA_OK)
        return 0;
    return layout_of(shape).total;
}

msa_status msa_workspace_init(void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (!workspace || !aligned16(workspace) || workspace_bytes < kAlign)
        return MSA_ERR_INVALID_ARGUMENT;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, stream));
}

msa_status msa_index_score(const msa_shape *shape, const void *q_idx, const void *idxk_pool,
                           const void *idxk_scales, const int32_t *block_table,
                           const int32_t *seq_lens, float *block_scores, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream)
{
    msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != MSA_OK)
        return st;
    const bool nvfp4 = shape->index_dtype == MSA_NVFP4;
    if (!q_idx || !idxk_pool || !block_table || !seq_lens || !block_scores ||
        (nvfp4 && !idxk_scales))
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || !aligned16(idxk_pool) || !aligned16(block_table) ||
        !aligned16(seq_lens) || !aligned16(block_scores) || (nvfp4 && !aligned16(idxk_scales)))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    return score_impl(shape, q_idx, idxk_pool, idxk_scales, block_table, seq_lens, block_scores,
                      workspace, stream);
}

msa_status msa_select_topk(const msa_shape *shape, const float *block_scores,
                           const int32_t *seq_lens, int32_t *selected, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream)
{
    msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != MSA_OK)
        return st;
    if (!block_scores || !seq_lens || !selected)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(block_scores) || !aligned16(seq_lens) || !aligned16(selected))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    return select_impl(shape, block_scores, seq_lens, selected, workspace, stream, false);
}

msa_status msa_sparse_decode(const msa_shape *shape, const void *q, const void *kv_pool,
                             const int32_t *block_table, const int32_t *seq_lens,
                             const int32_t *selected, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream)
{
    msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != MSA_OK)
        return st;
    if (!q || !kv_pool || !block_table || !seq_lens || !selected || !out || !lse)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(kv_pool) || !aligned16(block_table) || !aligned16(seq_lens) ||
        !aligned16(selected) || !aligned16(out) || !aligned16(lse))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    if ((st = check_decode_size(shape)) != MSA_OK)
        return st;
    return decode_impl(shape, q, kv_pool, block_table, seq_lens, selected, out, lse, workspace,
                       stream, false);
}

msa_status msa_decode_step(const msa_shape *shape, const void *q_idx, const void *idxk_pool,
                           const void *idxk_scales, const void *q, const void *kv_pool,
                           const int32_t *block_table, const int32_t *seq_lens,
                           float *block_scores, int32_t *selected, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != MSA_OK)
        return st;
    const bool nvfp4 = shape->index_dtype == MSA_NVFP4;
    if (!q_idx || !idxk_pool || !q || !kv_pool || !block_table || !seq_lens || !out || !lse ||
        (nvfp4 && !idxk_scales))
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q_idx) || !aligned16(idxk_pool) || !aligned16(q) || !aligned16(kv_pool) ||
        !aligned16(block_table) || !aligned16(seq_lens) || !aligned16(out) || !aligned16(lse) ||
        (nvfp4 && !aligned16(idxk_scales)) || (block_scores && !aligned16(block_scores)) ||
        (selected && !aligned16(selected)))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    if ((st = check_decode_size(shape)) != MSA_OK)
        return st;
    const WorkspaceLayout w = layout_of(shape);
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    if (!block_scores)
        block_scores = reinterpret_cast<float *>(wsb + w.scores_off);
    if (!selected)
        selected = reinterpret_cast<int32_t *>(wsb + w.selected_off);
    if ((st = score_impl(shape, q_idx, idxk_pool, idxk_scales, block_table, seq_lens,
                         block_scores, workspace, stream)) != MSA_OK)
        return st;
    // the select and the decode are programmatic dependents of the kernel before them
    if ((st = select_impl(shape, block_scores, seq_lens, selected, workspace, stream, true)) != MSA_OK)
        return st;
    return decode_impl(shape, q, kv_pool, block_table, seq_lens, selected, out, lse, workspace,
                       stream, true);
}

msa_status msa_kv_update(const msa_shape *shape, const void *k_new, const void *v_new,
                         const void *idxk_new, const int32_t *block_table,
                         const int32_t *seq_lens, void *kv_pool, void *idxk_pool,
                         void *idxk_scales, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream)
{
    msa_status st = check_shape(shape);
    if (st != MSA_OK)
        return st;
    if ((st = check_workspace(shape, workspace, workspace_bytes)) != MSA_OK)
        return st;
    const bool nvfp4 = shape->index_dtype == MSA_NVFP4;
    if (!k_new || !v_new || !idxk_new || !block_table || !seq_lens || !kv_pool || !idxk_pool ||
        (nvfp4 && !idxk_scales))
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(idxk_new) ||
        !aligned16(block_table) || !aligned16(seq_lens) || !aligned16(kv_pool) ||
        !aligned16(idxk_pool) || (nvfp4 && !aligned16(idxk_scales)))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    UpdateParams p;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.idxk_new = static_cast<const uint16_t *>(idxk_new);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.kv_pool = static_cast<uint8_t *>(kv_pool);
    p.idxk_pool = static_cast<uint8_t *>(idxk_pool);
    p.idxk_scales = static_cast<uint8_t *>(idxk_scales);
    p.err = static_cast<uint32_t *>(workspace);
    p.R = shape->num_requests;
    p.nq = shape->q_per_req;
    p.Hkv = shape->num_kv_heads;
    p.Hi = shape->num_index_heads;
    p.maxB = shape->max_blocks_per_seq;
    p.num_pages = shape->num_pages;
    p.kv_fp8 = shape->kv_dtype == MSA_FP8_E4M3;
    p.kv_nvfp4 = shape->kv_dtype == MSA_NVFP4;
    p.idx_nvfp4 = nvfp4;
    p.k_scale = shape->k_scale;
    p.v_scale = shape->v_scale;
    if ((p.kv_fp8 || p.kv_nvfp4) && !(shape->k_scale > 0.f && shape->v_scale > 0.f))
        return MSA_ERR_INVALID_ARGUMENT;
    return cuda_status(launch_kv_update(p, stream));
}

msa_status msa_select_rows(const msa_shape *shape, const float *scores_hbt,
                           const int32_t *seq_lens, int32_t *selected, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream)
{
    msa_status st = check_shape(shape, true);
    if (st != MSA_OK)
        return st;
    if (shape->max_blocks_per_seq > kMaxRowSelectBlocks)
        return MSA_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace) || workspace_bytes < kAlign)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!scores_hbt || !seq_lens || !selected)
        return MSA_ERR_INVALID_ARGUMENT;
    if (!aligned16(scores_hbt) || !aligned16(seq_lens) || !aligned16(selected))
        return MSA_ERR_INVALID_ARGUMENT;
    if (tokens_of(shape) == 0)
        return MSA_OK;
    SelectParams p;
    p.block_scores = scores_hbt;
    p.seq_lens = seq_lens;
    p.selected = selected;
    p.err = static_cast<uint32_t *>(workspace);
    p.R = shape->num_requests;
    p.nq = shape->q_per_req;
    p.maxB = shape->max_blocks_per_seq;
    p.k = shape->topk;
    p.Hs = selection_heads(shape);
    p.Hi = p.Hs; // the buffer holds the selection heads' scores already
    p.r = 1;
    p.init = shape->init_blocks;
    p.local = shape->local_blocks;
    return cuda_status(launch_select_rows(p, stream));
}

msa_status msa_set_decode_wait_limit(int64_t clocks)
{
    g_decode_wait_limit.store(clocks > 0 ? (long long)clocks : kWaitLimit,
                              std::memory_order_relaxed);
    return MSA_OK;
}

msa_status msa_check_device_status(void *workspace, cudaStream_t stream)
{
    if (!workspace || !aligned16(workspace))
        return MSA_ERR_INVALID_ARGUMENT;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (word == 0)
        return MSA_OK;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MSA_ERR_CUDA;
    return (word & kErrTimeout) ? MSA_ERR_TIMEOUT : MSA_ERR_DEVICE_CHECK;
}

const char *msa_status_string(msa_status status)
{
    switch (status) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARGUMENT: return "MSA_ERR_INVALID_ARGUMENT";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_DEVICE_CHECK: return "MSA_ERR_DEVICE_CHECK";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
    }
    return "MSA_ERR_UNKNOWN";
}

} // extern "C"
