/*
 * msa.h -- block-sparse paged decode attention for one NVIDIA GB300 (sm_103a).
 *
 * One decode step of the MiniMax-M3 sparse-attention ("MSA") path, as the
 * TensorRT-LLM pages describe it, for every query token t of the step:
 *   (a) score every cached token's index key against the token's index
 *       query and keep the maximum per 128-token block;
 *   (b) select the top-k blocks, ties going to the smaller block index,
 *       as an ascending, -1-padded table;
 *   (c) grouped-query attention (16 query heads per KV head) over only the
 *       selected 128-token pages, reached through the block table, giving
 *       the bf16 output and the log-sum-exp.
 *
 * Sources (prose only; none prints a formula or a layout):
 *   "MiniMax-M3 NVFP4 low-latency decode megakernel for modeling_v2 for
 *    Blackwell" -- sections "The TP4 decode target" (index scorer over
 *    index-K pages, long-context block selector and its smaller-block tie
 *    contract, long-context sparse decode) and "The TP8 decode target"
 *    (index scoring fused with block selection, 8-head sparse decode);
 *   "Add Rubin (sm_107) MiniMax-M3.1 low-latency decode targets" -- section
 *    "Items and numerics" (split-K merge of the long-context sparse decode:
 *    fixed order, no atomics, one divide per output), section "Disclosures
 *    and known gaps" (int32 KV offsets overflow at 1M context), and the
 *    commit messages on the selector / sparse-decode hooks (identical
 *    arguments), the long-context select (top-16 over up to 9216 blocks),
 *    the prefill select tile (per-block max-score buffer) and the q8kv4
 *    indexer (the ascending, -1-padded table contract);
 *   "MiniMax-M3: native P128 draft KV view for the NVFP4 hybrid cache" --
 *    section "Description" (128-token pages filled through one block table).
 * Where the pages are silent the library follows these definitions:
 *   - token t = r * q_per_req + j (request r, query j) sees positions
 *     0 .. seq_lens[r] + j - 1 (the causal limit);
 *   - index score = plain dot product; block score = max over the block's
 *     visible positions, -inf for a block with none;
 *   - only blocks with a visible position can be selected;
 *   - query head h uses KV head h / 16;
 *   - with one index head every KV head of a token uses one table; with
 *     Hi = num_index_heads > 1 (a multiple of Hkv), index head i belongs to
 *     KV head i / (Hi / Hkv) and each KV head g gets its own table, selected
 *     on the maximum over its index heads of their block scores
 *     ("KV-head-reduced scores", selector-hook commit of "Add Rubin (sm_107)
 *     ..."; the select op's table is [tokens, heads, topk]);
 *   - init / local forcing (prefill-select commit of "Add Rubin (sm_107)
 *     ..."): the first init_blocks and the last local_blocks blocks a token
 *     sees are always selected (init_blocks + local_blocks <= topk); the
 *     other places go to the best block scores as above;
 *   - logits are softmax_scale * q . k (FP8 keys times k_scale), the output
 *     is the softmax-weighted mean of V (FP8 values times v_scale), and
 *     lse = ln(sum exp(logit)) (natural log); NVFP4 keys and values are
 *     e2m1 x E4M3 scale x the tensor scale (k_scale, v_scale);
 *   - NVFP4 index keys: dimension 2i is the low nibble of byte i, one E4M3
 *     scale per 16 consecutive dimensions, no global scale.
 *
 * Conventions for every entry point:
 *   - Pointers are caller-owned device memory unless stated; the library
 *     allocates nothing and keeps no per-call state.
 *   - Calls are asynchronous on `stream`; only msa_check_device_status
 *     synchronises.
 *   - Arguments are validated on the host before anything is launched.  A
 *     shape the kernels do not cover returns MSA_ERR_UNSUPPORTED (never a
 *     silent fallback); bad pointers, sizes or alignment return
 *     MSA_ERR_INVALID_ARGUMENT.  Nothing is launched in either case.
 *   - Values that can only be checked on the device (page ids in the block
 *     table, seq_lens, selected block ids) are bounds-checked by the
 *     kernels before use (each of msa_index_score, msa_select_topk and
 *     msa_sparse_decode checks the ones it reads); a bad one sets a bit in
 *     the workspace's error word, the offending access is skipped, and the
 *     outputs of that call are unspecified.  msa_check_device_status
 *     reports and clears it.
 *   - Every device pointer must be 16-byte aligned.
 *
 * Layouts (row-major, element type as stored; T = num_requests * q_per_req,
 * Hi = num_index_heads, Hs = 1 if Hi == 1 else num_kv_heads (tables per
 * token), P = page_size = 128, D = head_dim = 128, Di = index_dim = 128):
 *   q_idx        bf16 [T][Hi][Di]
 *   idxk_pool    MSA_BF16:  bf16 [num_pages][Hi][P][Di]
 *                MSA_NVFP4: uint8 [num_pages][Hi][P][Di/2]  (e2m1 pairs)
 *   idxk_scales  MSA_NVFP4 only: E4M3 [num_pages][Hi][P][Di/16], else NULL
 *   q            bf16 [T][Hq][D]
 *   kv_pool      MSA_BF16 or MSA_FP8_E4M3 [num_pages][2][Hkv][P][D]: the K
 *                page of KV head g of page p, then the V pages after all K;
 *                MSA_NVFP4 [num_pages][2][Hkv] tiles of 9216 bytes: e2m1
 *                pairs [P][D/2] (dimension 2i in the low nibble) then E4M3
 *                scales [P][D/16], one per 16 dimensions; k_scale and
 *                v_scale are the tensor (second-level) scales
 *   block_table  int32 [num_requests][max_blocks_per_seq]; entry b of row r
 *                is the page of logical block b of request r.  Only blocks
 *                b < ceil((seq_lens[r] + q_per_req - 1) / P) are read.
 *   seq_lens     int32 [num_requests], each >= 1
 *   block_scores fp32 [T][Hi][max_blocks_per_seq]; entries b < the
 *                request's cached block count are written (-inf where the
 *                token sees no position of block b); the rest are untouched
 *   selected     int32 [T][Hs][topk], ascending, -1 padded
 *   out          bf16 [T][Hq][D] (round to nearest even from fp32)
 *   lse          fp32 [T][Hq]
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum msa_status {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARGUMENT = 1, /* null / misaligned pointer, bad size, small workspace */
    MSA_ERR_UNSUPPORTED = 2,      /* a shape or dtype the kernels do not cover */
    MSA_ERR_CUDA = 3,             /* a CUDA runtime call failed */
    MSA_ERR_DEVICE_CHECK = 4,     /* a kernel found a bad page id, seq_len or block id */
    MSA_ERR_TIMEOUT = 5           /* a kernel's bounded wait ran out */
} msa_status;

typedef enum msa_dtype {
    MSA_BF16 = 0,
    MSA_FP8_E4M3 = 1,
    MSA_NVFP4 = 2
} msa_dtype;

/* Shape and scalars of one call.  Covered today: head_dim = index_dim =
 * page_size = 128, num_q_heads = 16 * num_kv_heads, num_index_heads = 1 or
 * a multiple of num_kv_heads up to 64, 1 <= q_per_req <= 64,
 * 1 <= topk <= 256, max_blocks_per_seq <= 16384,
 * num_requests * q_per_req <= 8192, kv_dtype in {BF16, FP8_E4M3, NVFP4},
 * index_dtype in {BF16, NVFP4}. */
typedef struct msa_shape {
    int32_t num_requests;       /* R */
    int32_t q_per_req;          /* query tokens per request (1 + draft length) */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv */
    int32_t head_dim;           /* D */
    int32_t num_index_heads;    /* Hi */
    int32_t index_dim;          /* Di */
    int32_t page_size;          /* P, tokens per page */
    int32_t num_pages;          /* pages in kv_pool and idxk_pool */
    int32_t max_blocks_per_seq; /* block_table row width */
    int32_t topk;               /* blocks selected per token */
    int32_t kv_dtype;           /* msa_dtype of kv_pool */
    int32_t index_dtype;        /* msa_dtype of idxk_pool */
    int32_t decode_ctas;        /* persistent CTAs of the sparse decode; 0 = library default */
    float softmax_scale;        /* multiplies q . k (1/sqrt(128) in the workloads) */
    float k_scale;              /* FP8 K dequantisation scale (ignored for bf16) */
    float v_scale;              /* FP8 V dequantisation scale (ignored for bf16) */
    int32_t init_blocks;        /* first blocks every token keeps (0: none) */
    int32_t local_blocks;       /* most recent blocks every token keeps (0: none) */
} msa_shape;

/* Bytes of device workspace the calls below need for `shape` (0 if the
 * shape is invalid or unsupported).  Pure host function. */
size_t msa_workspace_bytes(const msa_shape *shape);

/* Zero the workspace (error word and the decode's split-arrival counters).
 * Call once after allocating it, and again after a call reported
 * MSA_ERR_TIMEOUT; every other call leaves the counters at zero. */
msa_status msa_workspace_init(void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Stage (a): block_scores[t][i][b] = max over the visible positions of
 * block b of dot(q_idx[t][i], index key of head i).  One pass per index
 * head.  Exact in fp32 for integer-valued
 * bf16 inputs with |score| < 2^24 and for NVFP4 keys with power-of-two
 * scales.  ("MiniMax-M3 NVFP4 low-latency decode megakernel ...", "The TP4
 * decode target": the index scorer; prefill-select commit of "Add Rubin
 * (sm_107) ...": the per-block max-score buffer.) */
msa_status msa_index_score(const msa_shape *shape, const void *q_idx, const void *idxk_pool,
                           const void *idxk_scales, const int32_t *block_table,
                           const int32_t *seq_lens, float *block_scores, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* Stage (b): for each token (and KV head, when Hs > 1), the topk blocks
 * with the largest block score (the maximum over the KV head's index heads)
 * among blocks 0 .. ceil((seq_lens[r] + j) / 128) - 1, ties to the smaller
 * block index, after the init_blocks first and local_blocks last of them,
 * which are always kept; written ascending and -1 padded.  Bit-exact.
 * init_blocks + local_blocks > topk, or either negative, returns
 * MSA_ERR_INVALID_ARGUMENT.
 * ("MiniMax-M3 NVFP4 low-latency decode megakernel ...", "The TP4 decode
 * target": tie contract; q8kv4 indexer commit of "Add Rubin (sm_107) ...":
 * the ascending, -1-padded table.) */
msa_status msa_select_topk(const msa_shape *shape, const float *block_scores,
                           const int32_t *seq_lens, int32_t *selected, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* Stage (c): attention of each token over the visible positions of its
 * selected blocks, split over persistent CTAs and merged in a fixed order
 * with one reciprocal per output row (no atomics).  out: bf16, lse: fp32.
 * The CTAs' task ranges are cut in 32-bit arithmetic: a call with
 * T * num_kv_heads * topk * (decode CTAs + 1) >= 2^32 returns
 * MSA_ERR_UNSUPPORTED (so does msa_decode_step).
 * ("MiniMax-M3 NVFP4 low-latency decode megakernel ...", "The TP4 decode
 * target": long-context sparse decode; "Add Rubin (sm_107) ...", "Items and
 * numerics": the split-K merge.) */
msa_status msa_sparse_decode(const msa_shape *shape, const void *q, const void *kv_pool,
                             const int32_t *block_table, const int32_t *seq_lens,
                             const int32_t *selected, void *out, float *lse, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* Stages (a) + (b) + (c) in one call (the fused decode step).  block_scores
 * and selected may be NULL, in which case the workspace holds them. */
msa_status msa_decode_step(const msa_shape *shape, const void *q_idx, const void *idxk_pool,
                           const void *idxk_scales, const void *q, const void *kv_pool,
                           const int32_t *block_table, const int32_t *seq_lens,
                           float *block_scores, int32_t *selected, void *out, float *lse,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* The KV / index-key update: writes this step's new tokens into their pages
 * through the block table, to run before msa_index_score / msa_decode_step
 * on the same stream.  ("MiniMax-M3 NVFP4 low-latency decode megakernel
 * ...", "The TP4 decode target": the attention megakernels carry "the KV
 * update"; q8kv4 indexer commit of "Add Rubin (sm_107) ...": the NVFP4
 * index-K copy is "refreshed from this step's slots".)
 *   k_new, v_new  bf16 [T][Hkv][D]   this step's keys and values
 *   idxk_new      bf16 [T][Hi][Di]   this step's index keys
 *   kv_pool, idxk_pool, idxk_scales  the pools of the layouts above (written)
 * New token j of request r goes to position seq_lens[r] - 1 + j (the last
 * position it sees): row (pos % 128) of page block_table[r][pos / 128].
 * Only those rows are written.  Encodings: bf16 pools take the inputs as
 * they are; MSA_FP8_E4M3 pools store E4M3(x / k_scale) for K and
 * E4M3(x / v_scale) for V; MSA_NVFP4 K / V pools store y = x / k_scale
 * (x / v_scale) by the index keys' recipe; MSA_NVFP4 index keys store, per 16 consecutive
 * dimensions, the E4M3 scale c = E4M3(max |x| / 6) and the e2m1 codes of
 * x / value(c) (0 when c is 0), dimension 2i in the low nibble.  Every
 * rounding is to nearest even and saturating, quotients in fp32, and a code
 * that rounds to zero is stored as +0.  A bad seq_len or page id is
 * reported through the workspace error word (that row is skipped). */
msa_status msa_kv_update(const msa_shape *shape, const void *k_new, const void *v_new,
                         const void *idxk_new, const int32_t *block_table,
                         const int32_t *seq_lens, void *kv_pool, void *idxk_pool,
                         void *idxk_scales, void *workspace, size_t workspace_bytes,
                         cudaStream_t stream);

/* Block tables of many query rows (a prefill's context rows) from a
 * head-major max-score buffer, one table per row and selection head, the
 * same table bit for bit as msa_select_topk gives each row (ties to the
 * smaller block, init / local forcing).  ("Add Rubin (sm_107) ...",
 * prefill-select commit: context rows take a tile select, one CTA per KV
 * head and 8 queries over a [heads, max_k_tiles, tokens] max-score block,
 * each score sector read once.)
 *   scores_hbt  fp32 [Hs][max_blocks_per_seq][T], the row index innermost:
 *               the selection heads' block scores (already reduced over
 *               index heads); entry b of row t is read for
 *               b < ceil((seq_lens[r] + j) / 128), t = r * q_per_req + j
 *   selected    int32 [T][Hs][topk], ascending, -1 padded
 * q_per_req may exceed the decode's 64 here (a prefill of C tokens is one
 * request with q_per_req = C and seq_lens = 1).  max_blocks_per_seq above
 * 2048 returns MSA_ERR_UNSUPPORTED (msa_select_topk covers longer rows in
 * the token-major layout).  Only the workspace's error word is used: a
 * workspace of 256 bytes suffices. */
msa_status msa_select_rows(const msa_shape *shape, const float *scores_hbt,
                           const int32_t *seq_lens, int32_t *selected, void *workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/* Size of the fixed device scratch used by msa_sparse_decode_noalloc. */
#define MSA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* The paper has no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory: a plugin handed only its input and
 * output tensors by a runtime that owns every device allocation, or code on
 * a path where the allocator may not be called.  It computes exactly what
 * msa_sparse_decode computes, with the same kernels, but keeps the scratch
 * (split partials, their arrival counters and the error word) in a fixed
 * array of MSA_NOALLOC_SCRATCH_BYTES compiled into the library, which every
 * GPU that loads the library holds until the process exits.  It allocates
 * nothing.
 *   - Every call asks the CUDA runtime for the address of the array in the
 *     current device's context (cudaGetSymbolAddress).  The first call on a
 *     device loads the library's device code there; make that first call
 *     before any stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, or different host threads) race and give wrong
 *     results.  Each call clears the error word and the arrival counters it
 *     needs; the partial slots are always written before they are read.
 *   - Device-side failures are not reported (there is no workspace to read
 *     them from): neither a bounds failure (bad page id, seq_len or block id)
 *     nor a bounded wait that ran out (MSA_ERR_TIMEOUT elsewhere).  After one
 *     the call still returns MSA_OK and its outputs are unspecified; callers
 *     that need to detect them use msa_sparse_decode.
 *   - Shapes are checked as by every other entry point, with the same
 *     statuses (MSA_ERR_INVALID_ARGUMENT, MSA_ERR_UNSUPPORTED).
 *   - Returns MSA_ERR_UNSUPPORTED when the scratch it needs exceeds
 *     MSA_NOALLOC_SCRATCH_BYTES: 256 bytes of error word, a 4-byte counter per
 *     (token, KV head) pair rounded up to 256 bytes, and (decode CTAs + pairs)
 *     partial slots of 8320 bytes (with 152 decode CTAs, the default on a
 *     152-SM GPU: at most 855 (token, KV head) pairs). */
msa_status msa_sparse_decode_noalloc(const msa_shape *shape, const void *q, const void *kv_pool,
                                     const int32_t *block_table, const int32_t *seq_lens,
                                     const int32_t *selected, void *out, float *lse,
                                     cudaStream_t stream);

/* Test hook, not for production use: the SM-clock limit of the sparse
 * decode's bounded waits in the calls that follow, for the whole process
 * (clocks <= 0 restores the default, 2^31).  With a limit of a few clocks a
 * normal decode gives up at its first wait that is not already complete: its
 * CTAs stop, wait (with the default limit) for their copies and tensor-core
 * work in flight, free their tensor memory and exit, and the call reports
 * MSA_ERR_TIMEOUT through msa_check_device_status.  That is how the timeout
 * path is tested without a hang or a fault.  Always returns MSA_OK. */
msa_status msa_set_decode_wait_limit(int64_t clocks);

/* Synchronise `stream`, read the workspace's error word and clear it.
 * Returns MSA_OK, MSA_ERR_DEVICE_CHECK, MSA_ERR_TIMEOUT or MSA_ERR_CUDA. */
msa_status msa_check_device_status(void *workspace, cudaStream_t stream);

/* Static, human-readable name of a status. */
const char *msa_status_string(msa_status status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
