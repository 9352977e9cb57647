"""Python binding of the block-sparse paged decode attention library.

Argument marshalling only: every function forwards to the C ABI of
``include/msa.h`` in ``libmsa_gb300.so`` (built in-tree by ``build.py``),
passing device pointers (``torch.Tensor.data_ptr()`` or plain ints) and the
CUDA stream handle.  Every step of the computation runs in the library's
CUDA kernels; there is no fallback.  If the library is missing, loading
raises.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

MSA_OK = 0
MSA_ERR_INVALID_ARGUMENT = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_CUDA = 3
MSA_ERR_DEVICE_CHECK = 4
MSA_ERR_TIMEOUT = 5

MSA_BF16 = 0
MSA_FP8_E4M3 = 1
MSA_NVFP4 = 2

DTYPE_CODES = {"bf16": MSA_BF16, "fp8": MSA_FP8_E4M3, "nvfp4": MSA_NVFP4}

# C entry points and their argument / return types (see include/msa.h).
_p = ctypes.c_void_p


class MsaShape(ctypes.Structure):
    _fields_ = [
        ("num_requests", ctypes.c_int32),
        ("q_per_req", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("num_index_heads", ctypes.c_int32),
        ("index_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("index_dtype", ctypes.c_int32),
        ("decode_ctas", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
        ("init_blocks", ctypes.c_int32),
        ("local_blocks", ctypes.c_int32),
    ]


_SIGNATURES = {
    "msa_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(MsaShape)]),
    "msa_workspace_init": (ctypes.c_int, [_p, ctypes.c_size_t, _p]),
    "msa_index_score": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, _p, _p, _p,
                                       ctypes.c_size_t, _p]),
    "msa_select_topk": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, ctypes.c_size_t,
                                       _p]),
    "msa_sparse_decode": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, _p, _p, _p, _p,
                                         ctypes.c_size_t, _p]),
    "msa_decode_step": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                       _p, _p, _p, ctypes.c_size_t, _p]),
    "msa_kv_update": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                     ctypes.c_size_t, _p]),
    "msa_select_rows": (ctypes.c_int, [ctypes.POINTER(MsaShape), _p, _p, _p, _p, ctypes.c_size_t,
                                       _p]),
    "msa_set_decode_wait_limit": (ctypes.c_int, [ctypes.c_int64]),
    "msa_check_device_status": (ctypes.c_int, [_p, _p]),
    "msa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load (once) the in-tree library; raises OSError if it has not been built."""
    global _lib
    if _lib is None:
        path = path or _build.LIB_PATH
        if not os.path.exists(path):
            raise OSError(f"{path} is missing: run __graft_entry__.build() (nvcc, sm_103a) first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != MSA_OK:
        raise MsaError(status, where)


def make_shape(*, num_requests, q_per_req, num_kv_heads, num_pages, max_blocks_per_seq, topk,
               kv_dtype="bf16", index_dtype="bf16", softmax_scale=128 ** -0.5, k_scale=1.0,
               v_scale=1.0, decode_ctas=0, head_dim=128, index_dim=128, page_size=128,
               num_index_heads=1, num_q_heads=None, init_blocks=0, local_blocks=0) -> MsaShape:
    if isinstance(kv_dtype, str):
        kv_dtype = DTYPE_CODES[kv_dtype]
    if isinstance(index_dtype, str):
        index_dtype = DTYPE_CODES[index_dtype]
    return MsaShape(
        num_requests=num_requests, q_per_req=q_per_req,
        num_q_heads=16 * num_kv_heads if num_q_heads is None else num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, num_index_heads=num_index_heads,
        index_dim=index_dim, page_size=page_size, num_pages=num_pages,
        max_blocks_per_seq=max_blocks_per_seq, topk=topk, kv_dtype=kv_dtype,
        index_dtype=index_dtype, decode_ctas=decode_ctas, softmax_scale=softmax_scale,
        k_scale=k_scale, v_scale=v_scale, init_blocks=init_blocks, local_blocks=local_blocks)


def msa_workspace_bytes(shape: MsaShape) -> int:
    return int(load().msa_workspace_bytes(ctypes.byref(shape)))


def msa_workspace_init(workspace, nbytes: int, stream=None):
    _check(load().msa_workspace_init(_ptr(workspace), int(nbytes), _stream(stream)),
           "msa_workspace_init")


def msa_index_score(shape, q_idx, idxk_pool, idxk_scales, block_table, seq_lens, block_scores,
                    workspace, workspace_bytes, stream=None):
    _check(load().msa_index_score(ctypes.byref(shape), _ptr(q_idx), _ptr(idxk_pool),
                                  _ptr(idxk_scales), _ptr(block_table), _ptr(seq_lens),
                                  _ptr(block_scores), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)), "msa_index_score")


def msa_select_topk(shape, block_scores, seq_lens, selected, workspace, workspace_bytes,
                    stream=None):
    _check(load().msa_select_topk(ctypes.byref(shape), _ptr(block_scores), _ptr(seq_lens),
                                  _ptr(selected), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)), "msa_select_topk")


def msa_sparse_decode(shape, q, kv_pool, block_table, seq_lens, selected, out, lse, workspace,
                      workspace_bytes, stream=None):
    _check(load().msa_sparse_decode(ctypes.byref(shape), _ptr(q), _ptr(kv_pool),
                                    _ptr(block_table), _ptr(seq_lens), _ptr(selected), _ptr(out),
                                    _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                    _stream(stream)), "msa_sparse_decode")


def msa_decode_step(shape, q_idx, idxk_pool, idxk_scales, q, kv_pool, block_table, seq_lens,
                    block_scores, selected, out, lse, workspace, workspace_bytes, stream=None):
    _check(load().msa_decode_step(ctypes.byref(shape), _ptr(q_idx), _ptr(idxk_pool),
                                  _ptr(idxk_scales), _ptr(q), _ptr(kv_pool), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(block_scores), _ptr(selected), _ptr(out),
                                  _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)), "msa_decode_step")


def msa_kv_update(shape, k_new, v_new, idxk_new, block_table, seq_lens, kv_pool, idxk_pool,
                  idxk_scales, workspace, workspace_bytes, stream=None):
    _check(load().msa_kv_update(ctypes.byref(shape), _ptr(k_new), _ptr(v_new), _ptr(idxk_new),
                                _ptr(block_table), _ptr(seq_lens), _ptr(kv_pool), _ptr(idxk_pool),
                                _ptr(idxk_scales), _ptr(workspace), int(workspace_bytes),
                                _stream(stream)), "msa_kv_update")


def msa_select_rows(shape, scores_hbt, seq_lens, selected, workspace, workspace_bytes,
                    stream=None):
    _check(load().msa_select_rows(ctypes.byref(shape), _ptr(scores_hbt), _ptr(seq_lens),
                                  _ptr(selected), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream)), "msa_select_rows")


def msa_check_device_status(workspace, stream=None) -> int:
    """Synchronise, read and clear the workspace error word; returns the status code."""
    return int(load().msa_check_device_status(_ptr(workspace), _stream(stream)))


def msa_set_decode_wait_limit(clocks: int):
    """Test hook: the clock limit of the decode's bounded waits (<= 0: the default)."""
    _check(load().msa_set_decode_wait_limit(int(clocks)), "msa_set_decode_wait_limit")
