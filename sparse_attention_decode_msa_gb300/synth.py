"""Seeded synthetic inputs for block-sparse paged decode attention.

This module only draws random numbers and lays them out in the byte formats
the library reads.  It holds none of the method's arithmetic: no scoring, no
selection, no softmax.  The CUDA path (tests, bench) and the CPU oracle both
consume exactly the arrays built here, so they see the same bytes.

Layouts (all C-contiguous, element types as stored):

    q_idx        uint16 (bf16 bits)  [T, Hi, 128]   (Hi index heads; 1 in the workloads)
    idxk_pool    bf16:  uint16       [num_pages, Hi, 128 tokens, 128 dims]
                 nvfp4: uint8        [num_pages, Hi, 128 tokens, 64]   two e2m1 codes
                                     per byte, dimension 2i in the low nibble
    idxk_scales  nvfp4 only: uint8   [num_pages, Hi, 128 tokens, 8]    one E4M3
                                     scale per 16 consecutive dimensions
    q            uint16 (bf16 bits)  [T, Hq, 128]
    kv_pool      bf16: uint16 / fp8: uint8 (E4M3)
                                     [num_pages, 2 (K then V), Hkv, 128 tokens, 128 dims]
                 nvfp4: uint8        [num_pages, 2, Hkv, 9216]: per (page, K/V, KV head) a
                                     tile of e2m1 pairs [128 tokens][64] (dimension 2i in
                                     the low nibble) then E4M3 scales [128 tokens][8], one
                                     per 16 dimensions; k_scale / v_scale are the tensor scales
    block_table  int32               [R, max_blocks]; entries past a request's last
                                     cached block are -1 and are never read
    seq_lens     int32               [R]; query token j of request r sees positions
                                     0 .. seq_lens[r] + j - 1, so the cache holds
                                     seq_lens[r] + q_per_req - 1 tokens

Token t of the step is request r = t // q_per_req, query j = t % q_per_req.

The five workloads follow the decode shapes of the MiniMax-M3 pages (P128 pages,
16 query heads per KV head, top-16 blocks, speculative steps of several query
tokens, contexts up to 128k); the pages measure on an agentic serving workload
and a math benchmark that are not used here: these seeded inputs stand in for them.
"""

from __future__ import annotations

import dataclasses
import math
import statistics
from typing import Optional

import numpy as np

PAGE = 128          # tokens per KV page (P128)
HEAD_DIM = 128      # attention head dimension
INDEX_DIM = 128     # index-key dimension
GROUP = 16          # query heads per KV head

BF16 = "bf16"
FP8 = "fp8"
NVFP4 = "nvfp4"


@dataclasses.dataclass
class Problem:
    name: str
    num_requests: int
    q_per_req: int
    num_kv_heads: int
    num_q_heads: int
    num_pages: int
    max_blocks: int
    topk: int
    kv_dtype: str
    index_dtype: str
    softmax_scale: float
    k_scale: float
    v_scale: float
    q_idx: np.ndarray
    idxk_pool: np.ndarray
    idxk_scales: Optional[np.ndarray]
    q: np.ndarray
    kv_pool: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    seed: int = 0
    recipe: str = ""
    num_index_heads: int = 1   # Hi: 1, or a multiple of num_kv_heads
    init_blocks: int = 0       # first blocks every token keeps
    local_blocks: int = 0      # most recent blocks every token keeps

    @property
    def num_tokens(self) -> int:
        return self.num_requests * self.q_per_req

    @property
    def contexts(self) -> np.ndarray:
        """Cached tokens per request (what the workload calls the context)."""
        return self.seq_lens.astype(np.int64) + self.q_per_req - 1

    def blocks_per_request(self) -> np.ndarray:
        return (self.contexts + PAGE - 1) // PAGE

    def visible(self, t: int) -> int:
        """Positions visible to token t (the causal limit)."""
        r, j = divmod(t, self.q_per_req)
        return int(self.seq_lens[r]) + j


# ---------------------------------------------------------------------------
# value tables

_NORMAL_TABLE: Optional[np.ndarray] = None


def _normal_quantiles() -> np.ndarray:
    """float32 N(0,1) quantiles at (i + 0.5) / 65536, i = 0..65535.

    A uniform 16-bit draw indexes this table: inverse-transform sampling of a
    standard normal on a 65536-point grid, far finer than bf16 resolves.
    """
    global _NORMAL_TABLE
    if _NORMAL_TABLE is None:
        nd = statistics.NormalDist()
        vals = [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)]
        _NORMAL_TABLE = np.asarray(vals, dtype=np.float32)
    return _NORMAL_TABLE


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest even), returned as uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


_BF16_NORMAL: Optional[np.ndarray] = None


def _bf16_normal_table() -> np.ndarray:
    global _BF16_NORMAL
    if _BF16_NORMAL is None:
        _BF16_NORMAL = f32_to_bf16_bits(_normal_quantiles())
    return _BF16_NORMAL


_FP8_NORMAL = None


def fp8_normal_table():
    """(uint8 E4M3 codes of N(0,1)/scale on the quantile grid, scale).

    scale = max|x| / 448 over the grid, so the largest draw maps to the
    largest finite E4M3 value.  The encoding uses torch's float8_e4m3fn cast
    (round to nearest even).
    """
    global _FP8_NORMAL
    if _FP8_NORMAL is None:
        import torch

        x = _normal_quantiles().astype(np.float64)
        scale = float(np.float32(np.max(np.abs(x)) / 448.0))
        codes = torch.from_numpy((x / scale).astype(np.float32)).to(torch.float8_e4m3fn)
        _FP8_NORMAL = (codes.view(torch.uint8).numpy().copy(), scale)
    return _FP8_NORMAL


def _u16(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.integers(0, 65536, size=n, dtype=np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return _bf16_normal_table()[_u16(rng, n)].reshape(shape)


def ints_bf16(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi], stored as bf16 bits (exact)."""
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


def _fill_chunked(out: np.ndarray, fn, rows_per_chunk: int):
    """Fill out[i0:i1] = fn(i1 - i0) chunk by chunk (bounded host memory)."""
    n = out.shape[0]
    for i0 in range(0, n, rows_per_chunk):
        i1 = min(n, i0 + rows_per_chunk)
        out[i0:i1] = fn(i1 - i0)


# ---------------------------------------------------------------------------
# generic builder

def make_problem(
    *,
    name: str,
    contexts,
    q_per_req: int,
    num_kv_heads: int,
    topk: int,
    kv_dtype: str = BF16,
    index_dtype: str = BF16,
    index_range=(-8, 8),
    num_pages: Optional[int] = None,
    guard_page: bool = False,
    max_blocks: Optional[int] = None,
    seed: int = 0,
    softmax_scale: Optional[float] = None,
    recipe: str = "",
    num_index_heads: int = 1,
    init_blocks: int = 0,
    local_blocks: int = 0,
) -> Problem:
    """Build a seeded problem.

    contexts[r] is the number of cached tokens of request r; its query token
    j sees contexts[r] - q_per_req + 1 + j positions.  Each request gets a
    disjoint set of pages drawn from one shuffled pool.  With guard_page,
    page 0 is a guard page that no block table references.
    """
    rng = np.random.default_rng(seed)
    contexts = np.asarray(contexts, dtype=np.int64).reshape(-1)
    R = int(contexts.shape[0])
    nq = int(q_per_req)
    if np.any(contexts < nq):
        raise ValueError("every context must hold at least q_per_req tokens")
    nblocks = (contexts + PAGE - 1) // PAGE
    need = int(nblocks.sum())
    first = 1 if guard_page else 0
    if num_pages is None:
        num_pages = need + first
    if need + first > num_pages:
        raise ValueError("pool too small for the contexts")
    if max_blocks is None:
        max_blocks = int(nblocks.max()) if R else 1
    Hkv = int(num_kv_heads)
    Hq = GROUP * Hkv
    T = R * nq

    perm = rng.permutation(np.arange(first, num_pages, dtype=np.int32))
    block_table = np.full((R, max_blocks), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        nb = int(nblocks[r])
        block_table[r, :nb] = perm[off:off + nb]
        off += nb
    seq_lens = (contexts - nq + 1).astype(np.int32)

    # index query and index-K pool
    lo, hi = index_range
    Hi = int(num_index_heads)
    q_idx = ints_bf16(rng, (T, Hi, INDEX_DIM), lo, hi)
    if index_dtype == BF16:
        idxk = np.empty((num_pages, Hi, PAGE, INDEX_DIM), dtype=np.uint16)
        _fill_chunked(idxk, lambda n: ints_bf16(rng, (n, Hi, PAGE, INDEX_DIM), lo, hi),
                      max(1, 1024 // Hi))
        scales = None
    elif index_dtype == NVFP4:
        idxk = np.empty((num_pages, Hi, PAGE, INDEX_DIM // 2), dtype=np.uint8)
        _fill_chunked(idxk, lambda n: rng.integers(0, 256, size=(n, Hi, PAGE, INDEX_DIM // 2),
                                                   dtype=np.uint8), max(1, 4096 // Hi))
        # E4M3 scale codes of 2^e, e uniform in [-4, 4]: code = (e + 7) << 3
        e = rng.integers(-4, 5, size=(num_pages, Hi, PAGE, INDEX_DIM // 16))
        scales = ((e + 7) << 3).astype(np.uint8)
    else:
        raise ValueError(index_dtype)

    q = normal_bf16(rng, (T, Hq, HEAD_DIM))

    kv_shape = (num_pages, 2, Hkv, PAGE, HEAD_DIM)
    per_page = 2 * Hkv * PAGE * HEAD_DIM
    k_scale = v_scale = 1.0
    if kv_dtype == BF16:
        kv = np.empty(kv_shape, dtype=np.uint16)
        table = _bf16_normal_table()
        _fill_chunked(kv, lambda n: table[_u16(rng, n * per_page)].reshape((n,) + kv_shape[1:]),
                      256)
    elif kv_dtype == FP8:
        kv = np.empty(kv_shape, dtype=np.uint8)
        codes, s = fp8_normal_table()
        k_scale = v_scale = s
        _fill_chunked(kv, lambda n: codes[_u16(rng, n * per_page)].reshape((n,) + kv_shape[1:]),
                      256)
    elif kv_dtype == NVFP4:
        tile = PAGE * HEAD_DIM // 2 + PAGE * HEAD_DIM // 16
        kv = np.empty((num_pages, 2, Hkv, tile), dtype=np.uint8)

        def nvfp4_tiles(n):
            # e2m1 codes uniform over the 16 codes; scales 2^e, e uniform in [-4, 0]
            t = np.empty((n, 2, Hkv, tile), dtype=np.uint8)
            t[..., : PAGE * HEAD_DIM // 2] = rng.integers(0, 256, size=(n, 2, Hkv, PAGE * HEAD_DIM // 2),
                                                          dtype=np.uint8)
            e = rng.integers(-4, 1, size=(n, 2, Hkv, PAGE * HEAD_DIM // 16))
            t[..., PAGE * HEAD_DIM // 2:] = ((e + 7) << 3).astype(np.uint8)
            return t

        _fill_chunked(kv, nvfp4_tiles, 256)
    else:
        raise ValueError(kv_dtype)

    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(HEAD_DIM)
    return Problem(
        name=name, num_requests=R, q_per_req=nq, num_kv_heads=Hkv, num_q_heads=Hq,
        num_pages=int(num_pages), max_blocks=int(max_blocks), topk=int(topk),
        kv_dtype=kv_dtype, index_dtype=index_dtype,
        softmax_scale=float(softmax_scale), k_scale=float(k_scale), v_scale=float(v_scale),
        q_idx=q_idx, idxk_pool=idxk, idxk_scales=scales, q=q, kv_pool=kv,
        block_table=block_table, seq_lens=seq_lens, seed=seed, recipe=recipe,
        num_index_heads=Hi, init_blocks=int(init_blocks), local_blocks=int(local_blocks),
    )


# ---------------------------------------------------------------------------
# the five workloads

WORKLOADS = {
    0: "tiny",
    1: "spec-verify",
    2: "long-context-ties",
    3: "high-concurrency-fp8",
    4: "nvfp4-index",
}


def workload_contexts(idx: int, rng: np.random.Generator) -> np.ndarray:
    if idx == 0:
        return np.array([4096])
    if idx == 1:
        return rng.integers(8192, 32768 + 1, size=8)
    if idx == 2:
        return np.array([131072, 131072])
    if idx == 3:
        c = np.exp(math.log(16384.0) + rng.standard_normal(48))
        return np.clip(np.round(c), 2048, 65536).astype(np.int64)
    if idx == 4:
        return np.full(32, 65536)
    raise ValueError(idx)


RECIPES = {
    0: "R=1 nq=1 C=4096 pool=64 Hkv=1 k=8 index ints[-8,8] bf16, Q/K/V bf16 N(0,1)",
    1: "R=8 nq=4 C~U[8192,32768] pool=4096 Hkv=4 k=16 index ints[-8,8], KV bf16 N(0,1)",
    2: "R=2 nq=48 C=131072 pool=2048+guard Hkv=4 k=16 index {-1,0,1}, KV bf16 N(0,1)",
    3: ("R=48 nq=1 C=clip(round(exp(ln 16384 + N(0,1))),2048,65536) pool=sum+guard Hkv=4 k=16 "
        "index ints[-8,8], KV e4m3 with per-tensor scale max|x|/448"),
    4: ("R=32 nq=2 C=65536 pool=16384+guard Hkv=4 k=32 index NVFP4 (e2m1 codes uniform, "
        "E4M3 scales 2^U{-4..4} per 16 dims), q_idx ints[-4,4], KV bf16 N(0,1)"),
}


def make_workload(idx: int, seed: Optional[int] = None, kv_dtype: Optional[str] = None) -> Problem:
    """The full-size workload number idx (0..4), seeded with seed (default idx).
    kv_dtype replaces the workload's KV dtype (same shapes; e.g. NVFP4 KV)."""
    seed = idx if seed is None else seed
    ctx = workload_contexts(idx, np.random.default_rng(10_000 + seed))
    name = WORKLOADS[idx]
    rec = RECIPES[idx]
    if kv_dtype is not None:
        name += f"-{kv_dtype}-kv"
        rec += f"; KV replaced by {kv_dtype}"
    kv = kv_dtype or BF16
    if idx == 0:
        return make_problem(name=name, contexts=ctx, q_per_req=1, num_kv_heads=1, topk=8,
                            num_pages=64, max_blocks=32, seed=seed, recipe=rec, kv_dtype=kv)
    if idx == 1:
        return make_problem(name=name, contexts=ctx, q_per_req=4, num_kv_heads=4, topk=16,
                            num_pages=4096, max_blocks=256, seed=seed, recipe=rec, kv_dtype=kv)
    if idx == 2:
        return make_problem(name=name, contexts=ctx, q_per_req=48, num_kv_heads=4, topk=16,
                            index_range=(-1, 1), num_pages=2049, guard_page=True, max_blocks=1024,
                            seed=seed, recipe=rec, kv_dtype=kv)
    if idx == 3:
        return make_problem(name=name, contexts=ctx, q_per_req=1, num_kv_heads=4, topk=16,
                            kv_dtype=kv_dtype or FP8, guard_page=True, max_blocks=512, seed=seed,
                            recipe=rec)
    if idx == 4:
        return make_problem(name=name, contexts=ctx, q_per_req=2, num_kv_heads=4, topk=32,
                            index_dtype=NVFP4, index_range=(-4, 4), num_pages=16385,
                            guard_page=True, max_blocks=512, seed=seed, recipe=rec, kv_dtype=kv)
    raise ValueError(idx)


def make_small_workload(idx: int, seed: Optional[int] = None) -> Problem:
    """A reduced copy of workload idx that the oracle finishes in about a
    second: same dtypes, head counts, q_per_req and top-k, shorter and ragged
    contexts (not multiples of 128) so every path meets a partial last block."""
    seed = 100 + idx if seed is None else seed
    rng = np.random.default_rng(20_000 + seed)
    if idx == 0:
        return make_problem(name="tiny-small", contexts=[1000], q_per_req=1, num_kv_heads=1,
                            topk=4, num_pages=16, seed=seed)
    if idx == 1:
        ctx = rng.integers(1500, 4000, size=3)
        return make_problem(name="spec-verify-small", contexts=ctx, q_per_req=4, num_kv_heads=4,
                            topk=16, num_pages=128, seed=seed)
    if idx == 2:
        return make_problem(name="long-ties-small", contexts=[3001, 2500], q_per_req=48,
                            num_kv_heads=4, topk=16, index_range=(-1, 1), guard_page=True,
                            seed=seed)
    if idx == 3:
        ctx = rng.integers(300, 5000, size=6)
        return make_problem(name="high-conc-fp8-small", contexts=ctx, q_per_req=1, num_kv_heads=4,
                            topk=16, kv_dtype=FP8, guard_page=True, seed=seed)
    if idx == 4:
        return make_problem(name="nvfp4-small", contexts=[4200, 5000, 3333], q_per_req=2,
                            num_kv_heads=4, topk=32, index_dtype=NVFP4, index_range=(-4, 4),
                            guard_page=True, seed=seed)
    raise ValueError(idx)


# ---------------------------------------------------------------------------
# this step's new tokens (the KV / index-key update)

# magnitudes of the sixteen e2m1 codes (sign in bit 3)
_E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def make_update(pb: Problem, seed: Optional[int] = None, exact_nvfp4: bool = False,
                index_range=(-8, 8)) -> dict:
    """Seeded new-token inputs of one step for problem pb (bf16 bits):

        k_new, v_new  [T, Hkv, 128]  N(0, 1)
        idxk_new      [T, Hi, 128]   bf16 index keys: integers in index_range, as the
                                     workloads' pools hold; NVFP4 index keys: N(0, 1) times 2^e with e
                                     uniform in [-4, 4] per group of 16 dimensions, or with
                                     exact_nvfp4 e2m1 magnitudes times 2^e with a +-6 in
                                     every group (values the NVFP4 format holds exactly)
    """
    rng = np.random.default_rng(pb.seed + 1000 if seed is None else seed)
    T, Hkv, Hi = pb.num_tokens, pb.num_kv_heads, pb.num_index_heads
    k_new = normal_bf16(rng, (T, Hkv, HEAD_DIM))
    v_new = normal_bf16(rng, (T, Hkv, HEAD_DIM))
    groups = (T, Hi, INDEX_DIM // 16, 16)
    if pb.index_dtype == BF16:
        idxk_new = ints_bf16(rng, (T, Hi, INDEX_DIM), *index_range)
    elif not exact_nvfp4:
        x = bf16_bits_to_f32(normal_bf16(rng, groups)).astype(np.float64)
        e = rng.integers(-4, 5, size=groups[:3] + (1,))
        idxk_new = f32_to_bf16_bits((x * np.exp2(e)).astype(np.float32)).reshape(T, Hi, INDEX_DIM)
    else:
        mag = _E2M1_MAGNITUDES[rng.integers(0, 8, size=groups)]
        mag[..., 0] = 6.0                      # the group's largest magnitude
        sign = np.where(rng.integers(0, 2, size=groups) == 1, -1.0, 1.0)
        e = rng.integers(-4, 5, size=groups[:3] + (1,))
        x = (sign * mag * np.exp2(e)).astype(np.float32)
        perm = np.argsort(rng.random(groups), axis=-1)   # the 6 at a random place
        x = np.take_along_axis(x, perm, axis=-1)
        idxk_new = f32_to_bf16_bits(x).reshape(T, Hi, INDEX_DIM)
    return {"k_new": k_new, "v_new": v_new, "idxk_new": idxk_new}
