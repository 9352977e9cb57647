"""Parity of the NVFP4 K/V decode (tiles widened to bf16 in shared memory
by converter warps) and of the NVFP4 K/V update with the CPU oracle.

Tables bit-exact; out within 4e-3 plus half a bf16 ulp of the reference
(NVFP4 values reach 6, so |O| can exceed 2 where bf16 storage alone rounds by
more than 4e-3), LSE within 1e-4 * max(|lse|, 1)."""

import numpy as np
import pytest

import oracle
from sparse_attention_decode_msa_gb300 import synth
from test_parity_gpu import THREADS, assert_attention_close, check_device_ok, device_problem

pytestmark = pytest.mark.gpu


def f4_problem(hkv, nq, contexts=(1500, 700, 3000, 200), k=6, seed=61, **kw):
    pb = synth.make_problem(name="f4kv", contexts=list(contexts), q_per_req=nq, num_kv_heads=hkv,
                            topk=k, kv_dtype=synth.NVFP4, seed=seed, **kw)
    pb.k_scale, pb.v_scale = 0.75, 0.5
    return pb


@pytest.mark.parametrize("hkv,nq", [(1, 1), (4, 4), (2, 12)])
def test_nvfp4_kv_fused_step(torch_cuda, hkv, nq):
    pb = f4_problem(hkv, nq)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens),
                           nvfp4_kv=True)
    check_device_ok(dp)


@pytest.mark.parametrize("ctas", [1, 5, 152])
def test_nvfp4_kv_split_independence_on_oracle_tables(torch_cuda, ctas):
    torch = torch_cuda
    pb = f4_problem(2, 3, contexts=(9000, 4000), k=16, seed=62)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb, decode_ctas=ctas)
    dp.selected.copy_(torch.from_numpy(ref["selected"])[:, None])
    dp.sparse_decode()
    res = dp.results()
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens),
                           nvfp4_kv=True)
    check_device_ok(dp)


def test_nvfp4_kv_with_index_heads_and_forcing(torch_cuda):
    pb = f4_problem(2, 2, num_index_heads=2, init_blocks=1, local_blocks=1)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens),
                           nvfp4_kv=True)


def test_nvfp4_kv_update_bytes_and_step(torch_cuda):
    pb = f4_problem(2, 3, seed=63)
    upd = synth.make_update(pb)
    want = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    dp = device_problem(pb)
    dp.kv_update(upd)
    got = dp.pools()
    assert np.array_equal(got["kv_pool"], want["kv_pool"])
    ref = oracle.decode_step(synth.Problem(**{**pb.__dict__, **want}), threads=THREADS)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens),
                           nvfp4_kv=True)
    check_device_ok(dp)
