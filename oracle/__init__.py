"""CPU oracle of block-sparse paged decode attention (TEST INFRASTRUCTURE).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library never calls it and shares
no code with it.  The arithmetic lives in ``msa_oracle.c`` (plain C, double
precision); this module compiles it with gcc on first use and marshals numpy
arrays through ctypes.  See ``msa_oracle.c`` for the definition each function
follows and the readings taken where the source pages are silent.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleShape(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("q_per_req", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("index_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("kv_fp8", ctypes.c_int32),
        ("index_nvfp4", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("k_scale", ctypes.c_double),
        ("v_scale", ctypes.c_double),
        ("num_index_heads", ctypes.c_int32),
        ("init_blocks", ctypes.c_int32),
        ("local_blocks", ctypes.c_int32),
    ]


ERRORS = {1: "page id out of range", 2: "bad seq_len", 3: "bad selection", 4: "out of memory",
          5: "bad shape"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile msa_oracle.c into a shared library (gcc, -O2, OpenMP)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            os.makedirs(_BUILD, exist_ok=True)
            tmp = _LIB_PATH + f".{os.getpid()}.tmp"
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC,
                   "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        p = ctypes.c_void_p
        L.oracle_bf16.restype = ctypes.c_double
        L.oracle_bf16.argtypes = [ctypes.c_uint16]
        L.oracle_e4m3.restype = ctypes.c_double
        L.oracle_e4m3.argtypes = [ctypes.c_uint8]
        L.oracle_e2m1.restype = ctypes.c_double
        L.oracle_e2m1.argtypes = [ctypes.c_uint8]
        L.oracle_block_scores.restype = ctypes.c_int
        L.oracle_block_scores.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, p, ctypes.c_int,
                                          ctypes.c_int, p]
        L.oracle_select.restype = ctypes.c_int
        L.oracle_select.argtypes = [p, ctypes.c_int, ctypes.c_int, p]
        L.oracle_select_forced.restype = ctypes.c_int
        L.oracle_select_forced.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, p]
        L.oracle_reduce_heads.restype = None
        L.oracle_reduce_heads.argtypes = [ctypes.POINTER(OracleShape), p, ctypes.c_int, p]
        L.oracle_attend.restype = ctypes.c_int
        L.oracle_attend.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, ctypes.c_int, p, p, p]
        L.oracle_decode_step.restype = ctypes.c_int
        L.oracle_decode_step.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, p, p, p, p,
                                         ctypes.c_int, ctypes.c_int, p, p, p, p]
        L.oracle_encode_e4m3.restype = ctypes.c_uint8
        L.oracle_encode_e4m3.argtypes = [ctypes.c_double]
        L.oracle_encode_e2m1.restype = ctypes.c_uint8
        L.oracle_encode_e2m1.argtypes = [ctypes.c_double]
        L.oracle_kv_update.restype = ctypes.c_int
        L.oracle_kv_update.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, p, p, p, p]
        L.oracle_select_rows.restype = ctypes.c_int
        L.oracle_select_rows.argtypes = [p, ctypes.c_int, ctypes.c_int, ctypes.c_int, p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, p]
        L.oracle_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def shape_of(pb) -> OracleShape:
    """OracleShape of a synthetic problem (any object with the Problem fields)."""
    return OracleShape(
        num_requests=pb.num_requests, q_per_req=pb.q_per_req, num_q_heads=pb.num_q_heads,
        num_kv_heads=pb.num_kv_heads, head_dim=pb.q.shape[-1], index_dim=pb.q_idx.shape[-1],
        page_size=128, num_pages=pb.num_pages, max_blocks=pb.max_blocks,
        topk=pb.topk, kv_fp8={"bf16": 0, "fp8": 1, "nvfp4": 2}[pb.kv_dtype],
        index_nvfp4=int(pb.index_dtype == "nvfp4"),
        softmax_scale=pb.softmax_scale, k_scale=pb.k_scale, v_scale=pb.v_scale,
        num_index_heads=pb.num_index_heads, init_blocks=pb.init_blocks,
        local_blocks=pb.local_blocks,
    )


def selection_heads(pb) -> int:
    """Tables per token: 1 with one index head, else one per KV head."""
    return 1 if pb.num_index_heads == 1 else pb.num_kv_heads


def _check(rc):
    if rc != 0:
        raise OracleError(ERRORS.get(rc, f"oracle error {rc}"))


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


def bf16(bits) -> float:
    return lib().oracle_bf16(int(bits))


def e4m3(code) -> float:
    return lib().oracle_e4m3(int(code))


def e2m1(nibble) -> float:
    return lib().oracle_e2m1(int(nibble))


def block_scores(pb, t: int, head: int = 0) -> np.ndarray:
    """float64 [max_blocks] per-block max index scores of token t, index head `head`."""
    s = shape_of(pb)
    out = np.empty(pb.max_blocks, dtype=np.float64)
    arrs = [_c(pb.q_idx), _c(pb.idxk_pool), _c(pb.idxk_scales), _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_block_scores(ctypes.byref(s), *[_ptr(a) for a in arrs], int(t), int(head),
                                     _ptr(out)))
    return out


def select(scores, n_valid: int, k: int, init: int = 0, local: int = 0) -> np.ndarray:
    """int32 [k] top-k block table (ascending, -1 padded) of a score row,
    keeping the first `init` and the last `local` of the n_valid blocks."""
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    sel = np.empty(k, dtype=np.int32)
    if init == 0 and local == 0:
        _check(lib().oracle_select(_ptr(sc), int(n_valid), int(k), _ptr(sel)))
    else:
        _check(lib().oracle_select_forced(_ptr(sc), int(n_valid), int(k), int(init), int(local),
                                          _ptr(sel)))
    return sel


def reduce_heads(pb, scores_by_head, gs: int) -> np.ndarray:
    """float64 [max_blocks]: the scores of selection head gs from [Hi, max_blocks]."""
    s = shape_of(pb)
    sc = np.ascontiguousarray(scores_by_head, dtype=np.float64)
    if sc.shape != (pb.num_index_heads, pb.max_blocks):
        raise ValueError("scores must be [num_index_heads, max_blocks]")
    out = np.empty(pb.max_blocks, dtype=np.float64)
    lib().oracle_reduce_heads(ctypes.byref(s), _ptr(sc), int(gs), _ptr(out))
    return out


def attend(pb, t: int, sel) -> tuple[np.ndarray, np.ndarray]:
    """(out float64 [Hq, D], lse float64 [Hq]) of token t over its tables
    sel ([topk] with one table, else [Hs, topk])."""
    s = shape_of(pb)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    if sel.size != selection_heads(pb) * pb.topk:
        raise ValueError("selection must have Hs x topk entries")
    out = np.empty((pb.num_q_heads, pb.q.shape[-1]), dtype=np.float64)
    lse = np.empty(pb.num_q_heads, dtype=np.float64)
    arrs = [_c(pb.q), _c(pb.kv_pool), _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_attend(ctypes.byref(s), *[_ptr(a) for a in arrs], int(t), _ptr(sel),
                               _ptr(out), _ptr(lse)))
    return out, lse


def decode_step(pb, tokens=None, threads: int = 1) -> dict:
    """Run the whole step for the given tokens (default: all).

    Returns block_scores float32 [n, max_blocks] ([n, Hi, max_blocks] with
    several index heads), selected int32 [n, topk] ([n, Hs, topk] with
    several index heads), out float64 [n, Hq, D], lse float64 [n, Hq],
    tokens int32 [n].
    """
    if tokens is None:
        tokens = np.arange(pb.num_tokens, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = int(tokens.shape[0])
    s = shape_of(pb)
    Hi, Hs = pb.num_index_heads, selection_heads(pb)
    bs = np.empty((n, Hi, pb.max_blocks), dtype=np.float32)
    sel = np.empty((n, Hs, pb.topk), dtype=np.int32)
    out = np.empty((n, pb.num_q_heads, pb.q.shape[-1]), dtype=np.float64)
    lse = np.empty((n, pb.num_q_heads), dtype=np.float64)
    arrs = [_c(pb.q_idx), _c(pb.idxk_pool), _c(pb.idxk_scales), _c(pb.q), _c(pb.kv_pool),
            _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_decode_step(ctypes.byref(s), *[_ptr(a) for a in arrs], _ptr(tokens), n,
                                    int(threads), _ptr(bs), _ptr(sel), _ptr(out), _ptr(lse)))
    if Hi == 1:
        bs, sel = bs[:, 0], sel[:, 0]
    return {"block_scores": bs, "selected": sel, "out": out, "lse": lse, "tokens": tokens}


def encode_e4m3(x) -> int:
    return int(lib().oracle_encode_e4m3(float(x)))


def encode_e2m1(x) -> int:
    return int(lib().oracle_encode_e2m1(float(x)))


def kv_update(pb, k_new, v_new, idxk_new) -> dict:
    """The pools after writing this step's new tokens (copies; pb is unchanged).

    k_new, v_new: bf16 bits [T, Hkv, D]; idxk_new: bf16 bits [T, Hi, Di].
    Returns kv_pool, idxk_pool, idxk_scales (None for bf16 index keys).
    """
    s = shape_of(pb)
    kv = np.array(pb.kv_pool, copy=True, order="C")
    ik = np.array(pb.idxk_pool, copy=True, order="C")
    sc = None if pb.idxk_scales is None else np.array(pb.idxk_scales, copy=True, order="C")
    arrs = [_c(np.asarray(k_new, dtype=np.uint16)), _c(np.asarray(v_new, dtype=np.uint16)),
            _c(np.asarray(idxk_new, dtype=np.uint16)), _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_kv_update(ctypes.byref(s), *[_ptr(a) for a in arrs], _ptr(kv), _ptr(ik),
                                  _ptr(sc)))
    return {"kv_pool": kv, "idxk_pool": ik, "idxk_scales": sc}


def select_rows(scores_hbt, n_visible, k: int, init: int = 0, local: int = 0) -> np.ndarray:
    """int32 [n_rows, Hs, k] tables of the rows of a [Hs, max_blocks, n_rows] score buffer."""
    sc = np.ascontiguousarray(scores_hbt, dtype=np.float64)
    hs, maxb, n = sc.shape
    nv = np.ascontiguousarray(n_visible, dtype=np.int32)
    sel = np.empty((n, hs, k), dtype=np.int32)
    _check(lib().oracle_select_rows(_ptr(sc), hs, maxb, n, _ptr(nv), int(k), int(init), int(local),
                                    _ptr(sel)))
    return sel


def max_threads() -> int:
    return int(lib().oracle_max_threads())
