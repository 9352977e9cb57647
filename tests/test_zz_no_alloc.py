"""msa_sparse_decode_noalloc: the sparse decode for callers that cannot
allocate device memory (a plugin given only its inputs and outputs by a
runtime that owns all device allocations, or code where the allocator may not
be called).  It keeps its scratch in a fixed array inside the library; these
tests call it through the C ABI and check that two calls in a row give what
the workspace-based msa_sparse_decode gives and what the CPU oracle gives,
that a problem at the documented size limit runs and one (token, KV head)
pair more is refused, and that shapes get the statuses of the other entry
points.  Every call gets real device buffers sized for its shape.

This file is collected last, so a run that stops at the first failure has run
every other test before it.
"""

import ctypes

import numpy as np
import pytest

import oracle
from sparse_attention_decode_msa_gb300 import synth
from test_parity_gpu import THREADS, assert_attention_close, visible_positions

pytestmark = pytest.mark.gpu

OUT_ATOL = 4e-3
LSE_RTOL = 1e-4
SCRATCH_BYTES = 8 << 20          # MSA_NOALLOC_SCRATCH_BYTES
PARTIAL_BYTES = (16 * 128 + 32) * 4


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


def noalloc(L, dp, out, lse, selected=None):
    import torch

    sel = dp.selected if selected is None else selected
    return L.msa_sparse_decode_noalloc(
        ctypes.byref(dp.shape), dp.q.data_ptr(), dp.kv.data_ptr(), dp.block_table.data_ptr(),
        dp.seq_lens.data_ptr(), sel.data_ptr(), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


def scratch_fits(pairs, ctas):
    head = 256 + (pairs * 4 + 255) // 256 * 256
    return head + (ctas + pairs) * PARTIAL_BYTES <= SCRATCH_BYTES


def test_two_calls_in_a_row_match_the_workspace_entry_point_and_the_oracle(lib):
    import torch

    from sparse_attention_decode_msa_gb300.runner import DeviceProblem

    # two different problems back to back: the second call must not see the
    # first call's leftovers in the shared scratch
    for idx in (1, 3):
        pb = synth.make_small_workload(idx)
        ref = oracle.decode_step(pb, threads=THREADS)
        dp = DeviceProblem(pb)
        dp.index_score()
        dp.select()
        dp.sparse_decode()                     # existing entry point, caller workspace
        want_out = dp.out.float().cpu().numpy()
        want_lse = dp.lse.cpu().numpy()
        assert np.array_equal(dp.selected[:, 0].cpu().numpy(), ref["selected"])
        out = torch.full_like(dp.out, float("nan"))
        lse = torch.full_like(dp.lse, float("nan"))
        assert noalloc(lib, dp, out, lse) == 0
        torch.cuda.synchronize()
        got_out = out.float().cpu().numpy()
        got_lse = lse.cpu().numpy()
        assert np.all(np.isfinite(got_out)) and np.all(np.isfinite(got_lse))
        assert np.abs(got_out - want_out).max() <= OUT_ATOL
        assert (np.abs(got_lse - want_lse) / np.maximum(np.abs(want_lse), 1)).max() <= LSE_RTOL
        assert_attention_close(got_out.astype(np.float64), got_lse.astype(np.float64), ref["out"],
                               ref["lse"], range(pb.num_tokens))


def test_the_documented_limit_runs_and_one_pair_more_is_refused(lib):
    import torch

    import sparse_attention_decode_msa_gb300 as msa
    from sparse_attention_decode_msa_gb300.runner import DeviceProblem

    # with 152 decode CTAs the array holds 855 (token, KV head) pairs
    ctas = 152
    assert scratch_fits(855, ctas) and not scratch_fits(856, ctas)
    rng = np.random.default_rng(90)
    ctx = rng.integers(1, 400, size=856)
    for pairs in (855, 856):
        pb = synth.make_problem(name="noalloc-limit", contexts=ctx[:pairs], q_per_req=1,
                                num_kv_heads=1, topk=2, seed=91)
        ref = oracle.decode_step(pb, threads=THREADS)
        dp = DeviceProblem(pb, decode_ctas=ctas)
        sel = torch.from_numpy(ref["selected"][:, None, :].copy()).cuda()
        out = torch.full_like(dp.out, float("nan"))
        lse = torch.full_like(dp.lse, float("nan"))
        st = noalloc(lib, dp, out, lse, selected=sel)
        torch.cuda.synchronize()
        if pairs == 856:
            assert st == msa.MSA_ERR_UNSUPPORTED
            continue
        assert st == msa.MSA_OK
        tokens = range(pb.num_tokens)
        assert_attention_close(out.float().cpu().numpy().astype(np.float64),
                               lse.cpu().numpy().astype(np.float64), ref["out"], ref["lse"],
                               tokens, visible=visible_positions(pb, ref["selected"], tokens))


@pytest.mark.parametrize("field,value,status", [
    ("topk", 0, 1), ("init_blocks", 3, 1), ("softmax_scale", float("nan"), 1),
    ("head_dim", 64, 2), ("kv_dtype", 3, 2),
])
def test_shapes_get_the_statuses_of_the_other_entry_points(lib, field, value, status):
    import torch

    from sparse_attention_decode_msa_gb300.runner import DeviceProblem

    pb = synth.make_small_workload(1)
    dp = DeviceProblem(pb)
    if field == "init_blocks":
        dp.shape.init_blocks, dp.shape.local_blocks = value, pb.topk   # init + local > topk
    else:
        setattr(dp.shape, field, value)
    out = torch.empty_like(dp.out)
    lse = torch.empty_like(dp.lse)
    assert noalloc(lib, dp, out, lse) == status
