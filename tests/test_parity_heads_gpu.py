"""Parity of the CUDA path with the CPU oracle for the selection variants:
several index heads (one table per KV head, selected on the maximum over the
KV head's index heads) and init / local block forcing.

Block scores and tables are bit-exact; out within 4e-3 and LSE within
1e-4 * max(|lse|, 1) of the float64 oracle (the workload contract).
"""

import numpy as np
import pytest

import oracle
from sparse_attention_decode_msa_gb300 import synth
from test_parity_gpu import THREADS, assert_attention_close, check_device_ok, device_problem

pytestmark = pytest.mark.gpu

P = synth.PAGE


def heads_problem(hkv, hi, nq, index_dtype=synth.BF16, kv_dtype=synth.BF16, init=0, local=0,
                  contexts=(900, 2500, 1700), topk=4, seed=31, **kw):
    return synth.make_problem(
        name=f"heads{hi}", contexts=list(contexts), q_per_req=nq, num_kv_heads=hkv, topk=topk,
        kv_dtype=kv_dtype, index_dtype=index_dtype, num_index_heads=hi, seed=seed,
        index_range=(-2, 2) if index_dtype == synth.BF16 else (-4, 4), init_blocks=init,
        local_blocks=local, **kw)


def assert_tables_equal(pb, got, want):
    """Per-head block scores: every entry the token can see; tables: all."""
    for t in range(pb.num_tokens):
        n = (pb.visible(t) + P - 1) // P
        assert np.array_equal(got["block_scores"][t, :, :n], want["block_scores"][t, :, :n]), t
    assert np.array_equal(got["selected"], want["selected"])


# bf16 keys: nq 1 and 4 take the mma.sync scorer, 12 the tcgen05 scorer;
# NVFP4 keys: nq 1 the bulk-copy scorer, 17 the mma.sync NVFP4 scorer.
@pytest.mark.parametrize("hkv,hi", [(1, 2), (2, 2), (2, 4), (4, 4)])
@pytest.mark.parametrize("nq,index_dtype", [(1, synth.BF16), (4, synth.BF16), (12, synth.BF16),
                                            (1, synth.NVFP4), (17, synth.NVFP4)])
def test_index_heads_fused_step(torch_cuda, hkv, hi, nq, index_dtype):
    pb = heads_problem(hkv, hi, nq, index_dtype)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert res["selected"].shape == (pb.num_tokens, hkv, pb.topk)
    assert_tables_equal(pb, res, ref)
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


def test_index_heads_stage_by_stage(torch_cuda):
    torch = torch_cuda
    pb = heads_problem(2, 4, 3, contexts=(1300, 600), init=1, local=1)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.index_score()
    res = dp.results()
    for t in range(pb.num_tokens):
        n = (pb.visible(t) + P - 1) // P
        assert np.array_equal(res["block_scores"][t, :, :n], ref["block_scores"][t, :, :n]), t
    # select on the oracle's scores, decode on the oracle's tables
    dp.block_scores.copy_(torch.from_numpy(ref["block_scores"]))
    dp.select()
    assert np.array_equal(dp.results()["selected"], ref["selected"])
    dp.selected.copy_(torch.from_numpy(ref["selected"]))
    dp.sparse_decode()
    res = dp.results()
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("init,local", [(1, 0), (0, 1), (1, 1), (2, 2), (4, 0), (0, 4)])
@pytest.mark.parametrize("hi", [1, 2])
def test_forcing_fused_step(torch_cuda, init, local, hi):
    pb = heads_problem(2, hi, 2, init=init, local=local, contexts=(1100, 300, 2000, 129))
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    if hi == 1:
        for t in range(pb.num_tokens):
            n = (pb.visible(t) + P - 1) // P
            assert np.array_equal(res["block_scores"][t, :n], ref["block_scores"][t, :n]), t
        assert np.array_equal(res["selected"], ref["selected"])
    else:
        assert_tables_equal(pb, res, ref)
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("hi,max_blocks", [(2, 600), (4, 300), (1, 2048)])
def test_index_heads_and_forcing_on_the_four_warp_select(torch_cuda, hi, max_blocks):
    # tables wider than 256 blocks take the select by four warps of a CTA:
    # its group maxima over index heads, forced blocks and tie order must be
    # those of the oracle too
    pb = heads_problem(2, hi, 3, init=2, local=3, contexts=(9000, 30000, 4100), topk=12,
                       max_blocks=max_blocks)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    if hi == 1:
        for t in range(pb.num_tokens):
            n = (pb.visible(t) + P - 1) // P
            assert np.array_equal(res["block_scores"][t, :n], ref["block_scores"][t, :n]), t
        assert np.array_equal(res["selected"], ref["selected"])
    else:
        assert_tables_equal(pb, res, ref)
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


def test_forcing_on_the_long_row_select(torch_cuda):
    # more than 2048 blocks in the table row: the one-CTA-per-row select
    pb = synth.make_problem(name="wide-forced", contexts=[40000], q_per_req=2, num_kv_heads=1,
                            topk=32, max_blocks=4000, seed=26, init_blocks=3, local_blocks=5)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))


def test_forcing_all_places(torch_cuda):
    # init + local = topk: the table is exactly the forced blocks
    pb = heads_problem(1, 1, 1, init=2, local=2, contexts=(3000,), topk=4)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    n = (pb.visible(0) + P - 1) // P
    assert res["selected"][0].tolist() == [0, 1, n - 2, n - 1]


def test_index_heads_fp8_kv_and_split_independence(torch_cuda):
    pb = heads_problem(2, 2, 4, kv_dtype=synth.FP8, contexts=(5000, 2200))
    ref = oracle.decode_step(pb, threads=THREADS)
    for ctas in (1, 7, 152):
        dp = device_problem(pb, decode_ctas=ctas)
        dp.decode_step()
        res = dp.results()
        assert np.array_equal(res["selected"], ref["selected"])
        assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"],
                               range(pb.num_tokens))
        check_device_ok(dp)
