"""msa_sparse_decode_noalloc: the sparse decode for callers that cannot
allocate device memory (a plugin given only its inputs and outputs by a
runtime that owns all device allocations, or code where the allocator may not
be called).  It keeps its scratch in a fixed array inside the library; these
tests check, through the C ABI, that two calls in a row give what the
workspace-based msa_sparse_decode gives, and that it refuses problems bigger
than that array.

This file is collected last, so a run that stops at the first failure has run
every other test before it.
"""

import ctypes

import numpy as np
import pytest

from sparse_attention_decode_msa_gb300 import synth

pytestmark = pytest.mark.gpu

OUT_ATOL = 4e-3
LSE_RTOL = 1e-4


@pytest.fixture(scope="module")
def lib():
    import torch

    import sparse_attention_decode_msa_gb300 as msa
    from sparse_attention_decode_msa_gb300 import build

    build.build()
    L = msa.load()
    p = ctypes.c_void_p
    L.msa_sparse_decode_noalloc.restype = ctypes.c_int
    L.msa_sparse_decode_noalloc.argtypes = [ctypes.POINTER(msa.MsaShape), p, p, p, p, p, p, p, p]
    torch.cuda.init()
    return L


def noalloc(L, dp, out, lse):
    import torch

    return L.msa_sparse_decode_noalloc(
        ctypes.byref(dp.shape), dp.q.data_ptr(), dp.kv.data_ptr(), dp.block_table.data_ptr(),
        dp.seq_lens.data_ptr(), dp.selected.data_ptr(), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def test_two_calls_in_a_row_match_the_workspace_entry_point(lib):
    import torch

    from sparse_attention_decode_msa_gb300.runner import DeviceProblem

    # two different problems back to back: the second call must not see the
    # first call's leftovers in the shared scratch
    for idx in (1, 3):
        pb = synth.make_small_workload(idx)
        dp = DeviceProblem(pb)
        dp.index_score()
        dp.select()
        dp.sparse_decode()                     # existing entry point, caller workspace
        want_out = dp.out.float().cpu().numpy()
        want_lse = dp.lse.cpu().numpy()
        out = torch.full_like(dp.out, float("nan"))
        lse = torch.full_like(dp.lse, float("nan"))
        assert noalloc(lib, dp, out, lse) == 0
        torch.cuda.synchronize()
        got_out = out.float().cpu().numpy()
        got_lse = lse.cpu().numpy()
        assert np.all(np.isfinite(got_out)) and np.all(np.isfinite(got_lse))
        assert np.abs(got_out - want_out).max() <= OUT_ATOL
        assert (np.abs(got_lse - want_lse) / np.maximum(np.abs(want_lse), 1)).max() <= LSE_RTOL


def test_problems_beyond_the_scratch_are_refused(lib):
    import sparse_attention_decode_msa_gb300 as msa

    # 8192 tokens x 4 KV heads needs far more partial slots than the array holds
    s = msa.make_shape(num_requests=2048, q_per_req=4, num_kv_heads=4, num_pages=64,
                       max_blocks_per_seq=8, topk=4)
    fake = 0x10000  # never dereferenced: the size check comes first
    st = lib.msa_sparse_decode_noalloc(ctypes.byref(s), *([fake] * 7), None)
    assert st == msa.MSA_ERR_UNSUPPORTED
