"""Parity of the CUDA KV / index-key update with the CPU oracle: the pools
after the update are compared byte for byte (FP8 and NVFP4 codes included),
and a step run on the updated pools matches the oracle's step on its own
updated pools."""

import numpy as np
import pytest

import oracle
import sparse_attention_decode_msa_gb300 as msa
from sparse_attention_decode_msa_gb300 import synth
from test_parity_gpu import THREADS, assert_attention_close, check_device_ok, device_problem

pytestmark = pytest.mark.gpu

P = synth.PAGE


@pytest.mark.parametrize("kv_dtype", [synth.BF16, synth.FP8])
@pytest.mark.parametrize("index_dtype", [synth.BF16, synth.NVFP4])
@pytest.mark.parametrize("hkv,hi,nq", [(1, 1, 1), (2, 2, 3), (4, 1, 2), (2, 4, 1)])
def test_update_writes_the_oracles_bytes(torch_cuda, kv_dtype, index_dtype, hkv, hi, nq):
    pb = synth.make_problem(name="upd", contexts=[300, 1000, 129, 2047], q_per_req=nq,
                            num_kv_heads=hkv, topk=4, kv_dtype=kv_dtype, index_dtype=index_dtype,
                            num_index_heads=hi, seed=40 + hkv + hi + nq)
    if kv_dtype == synth.FP8:
        pb.v_scale = pb.k_scale * 0.75
    upd = synth.make_update(pb)
    want = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    dp = device_problem(pb)
    dp.kv_update(upd)
    got = dp.pools()
    assert np.array_equal(got["kv_pool"], want["kv_pool"])
    assert np.array_equal(got["idxk_pool"], want["idxk_pool"])
    if index_dtype == synth.NVFP4:
        assert np.array_equal(got["idxk_scales"], want["idxk_scales"])
    check_device_ok(dp)


@pytest.mark.parametrize("kv_dtype,index_dtype", [(synth.BF16, synth.BF16), (synth.FP8, synth.NVFP4)])
def test_step_after_update(torch_cuda, kv_dtype, index_dtype):
    # NVFP4 keys written from values the format holds exactly, so the index
    # scores stay exact in fp32 and the tables compare bit for bit
    pb = synth.make_problem(name="upd-step", contexts=[1500, 700, 3000], q_per_req=2,
                            num_kv_heads=2, topk=4, kv_dtype=kv_dtype, index_dtype=index_dtype,
                            index_range=(-4, 4), seed=47)
    upd = synth.make_update(pb, exact_nvfp4=True, index_range=(-4, 4))
    new = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    ref_pb = synth.Problem(**{**pb.__dict__, **new})
    ref = oracle.decode_step(ref_pb, threads=THREADS)
    dp = device_problem(pb)
    dp.kv_update(upd)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


def test_update_reports_a_missing_page(torch_cuda):
    pb = synth.make_problem(name="upd-bad", contexts=[300], q_per_req=1, num_kv_heads=1, topk=2,
                            seed=48)
    r, pos = 0, int(pb.seq_lens[0]) - 1
    before = pb.kv_pool.copy()
    pb.block_table[r, pos // P] = pb.num_pages + 5         # out of the pool
    dp = device_problem(pb)
    dp.kv_update(synth.make_update(pb))
    assert msa.msa_check_device_status(dp.ws) == msa.MSA_ERR_DEVICE_CHECK
    assert np.array_equal(dp.pools()["kv_pool"], before)
