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
    ]


ERRORS = {1: "page id out of range", 2: "bad seq_len", 3: "bad selection", 4: "out of memory"}


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
        L.oracle_block_scores.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, p, ctypes.c_int, p]
        L.oracle_select.restype = ctypes.c_int
        L.oracle_select.argtypes = [p, ctypes.c_int, ctypes.c_int, p]
        L.oracle_attend.restype = ctypes.c_int
        L.oracle_attend.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, ctypes.c_int, p, p, p]
        L.oracle_decode_step.restype = ctypes.c_int
        L.oracle_decode_step.argtypes = [ctypes.POINTER(OracleShape), p, p, p, p, p, p, p, p,
                                         ctypes.c_int, ctypes.c_int, p, p, p, p]
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
        page_size=pb.kv_pool.shape[3], num_pages=pb.num_pages, max_blocks=pb.max_blocks,
        topk=pb.topk, kv_fp8=int(pb.kv_dtype == "fp8"), index_nvfp4=int(pb.index_dtype == "nvfp4"),
        softmax_scale=pb.softmax_scale, k_scale=pb.k_scale, v_scale=pb.v_scale,
    )


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


def block_scores(pb, t: int) -> np.ndarray:
    """float64 [max_blocks] per-block max index scores of token t."""
    s = shape_of(pb)
    out = np.empty(pb.max_blocks, dtype=np.float64)
    arrs = [_c(pb.q_idx), _c(pb.idxk_pool), _c(pb.idxk_scales), _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_block_scores(ctypes.byref(s), *[_ptr(a) for a in arrs], int(t), _ptr(out)))
    return out


def select(scores, n_valid: int, k: int) -> np.ndarray:
    """int32 [k] top-k block table (ascending, -1 padded) of a score row."""
    sc = np.ascontiguousarray(scores, dtype=np.float64)
    sel = np.empty(k, dtype=np.int32)
    _check(lib().oracle_select(_ptr(sc), int(n_valid), int(k), _ptr(sel)))
    return sel


def attend(pb, t: int, sel) -> tuple[np.ndarray, np.ndarray]:
    """(out float64 [Hq, D], lse float64 [Hq]) of token t over selection sel."""
    s = shape_of(pb)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    if sel.shape[0] != pb.topk:
        raise ValueError("selection must have topk entries")
    out = np.empty((pb.num_q_heads, pb.q.shape[-1]), dtype=np.float64)
    lse = np.empty(pb.num_q_heads, dtype=np.float64)
    arrs = [_c(pb.q), _c(pb.kv_pool), _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_attend(ctypes.byref(s), *[_ptr(a) for a in arrs], int(t), _ptr(sel),
                               _ptr(out), _ptr(lse)))
    return out, lse


def decode_step(pb, tokens=None, threads: int = 1) -> dict:
    """Run the whole step for the given tokens (default: all).

    Returns block_scores float32 [n, max_blocks], selected int32 [n, topk],
    out float64 [n, Hq, D], lse float64 [n, Hq], tokens int32 [n].
    """
    if tokens is None:
        tokens = np.arange(pb.num_tokens, dtype=np.int32)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    n = int(tokens.shape[0])
    s = shape_of(pb)
    bs = np.empty((n, pb.max_blocks), dtype=np.float32)
    sel = np.empty((n, pb.topk), dtype=np.int32)
    out = np.empty((n, pb.num_q_heads, pb.q.shape[-1]), dtype=np.float64)
    lse = np.empty((n, pb.num_q_heads), dtype=np.float64)
    arrs = [_c(pb.q_idx), _c(pb.idxk_pool), _c(pb.idxk_scales), _c(pb.q), _c(pb.kv_pool),
            _c(pb.block_table), _c(pb.seq_lens)]
    _check(lib().oracle_decode_step(ctypes.byref(s), *[_ptr(a) for a in arrs], _ptr(tokens), n,
                                    int(threads), _ptr(bs), _ptr(sel), _ptr(out), _ptr(lse)))
    return {"block_scores": bs, "selected": sel, "out": out, "lse": lse, "tokens": tokens}


def max_threads() -> int:
    return int(lib().oracle_max_threads())
