"""Parity of msa_select_rows (many query rows from a head-major score buffer,
the prefill select tile) with the CPU oracle, and its same-table property
against the per-token select.  Tables are compared bit for bit."""

import numpy as np
import pytest

import oracle
import sparse_attention_decode_msa_gb300 as msa
from sparse_attention_decode_msa_gb300 import synth
from test_parity_gpu import THREADS, check_device_ok, device_problem

pytestmark = pytest.mark.gpu

P = synth.PAGE


def visible_blocks(seq_lens, nq):
    R = len(seq_lens)
    t = np.arange(R * nq)
    return ((np.asarray(seq_lens)[t // nq] + t % nq + P - 1) // P).astype(np.int32)


def run_rows(torch, scores_hbt, seq_lens, nq, k, init=0, local=0, hkv=1, hi=1):
    hs, maxb, T = scores_hbt.shape
    shape = msa.make_shape(num_requests=len(seq_lens), q_per_req=nq, num_kv_heads=hkv,
                           num_pages=1, max_blocks_per_seq=maxb, topk=k, num_index_heads=hi,
                           init_blocks=init, local_blocks=local)
    sc = torch.from_numpy(np.ascontiguousarray(scores_hbt, dtype=np.float32)).cuda()
    sl = torch.from_numpy(np.asarray(seq_lens, dtype=np.int32)).cuda()
    sel = torch.full((T, hs, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    msa.msa_select_rows(shape, sc, sl, sel, ws, 256)
    status = msa.msa_check_device_status(ws)
    return sel.cpu().numpy(), status


@pytest.mark.parametrize("maxb", [16, 200, 600, 2048])
@pytest.mark.parametrize("init,local", [(0, 0), (1, 2)])
def test_prefill_rows_of_one_request(torch_cuda, maxb, init, local):
    # a prefill of C tokens: one request, q_per_req = C, seq_len = 1, so row
    # j sees ceil((j + 1) / 128) blocks
    C = min(maxb * P, 3000)
    rng = np.random.default_rng(maxb + init)
    scores = rng.integers(-3, 4, size=(1, maxb, C)).astype(np.float32)
    nvis = visible_blocks([1], C)
    want = oracle.select_rows(scores, nvis, 4, init, local)
    got, status = run_rows(torch_cuda, scores, [1], C, 4, init, local)
    assert status == msa.MSA_OK
    assert np.array_equal(got, want)


@pytest.mark.parametrize("maxb,k", [(40, 3), (300, 16), (1100, 32)])
def test_ragged_rows_several_requests_and_heads(torch_cuda, maxb, k):
    rng = np.random.default_rng(maxb)
    nq = 37                                       # 3 * 37 = 111 rows: ragged tiles, T % 4 != 0
    seq_lens = rng.integers(1, maxb * P - nq + 2, size=3).astype(np.int32)
    T = 3 * nq
    scores = rng.integers(-2, 3, size=(2, maxb, T)).astype(np.float32)
    want = oracle.select_rows(scores, visible_blocks(seq_lens, nq), k, 1, 1)
    got, status = run_rows(torch_cuda, scores, seq_lens, nq, k, 1, 1, hkv=2, hi=2)
    assert status == msa.MSA_OK
    assert np.array_equal(got, want)


def test_same_table_as_the_per_token_select(torch_cuda):
    torch = torch_cuda
    pb = synth.make_small_workload(2)             # heavy ties at the k-th place
    dp = device_problem(pb)
    dp.index_score()
    dp.select()
    res = dp.results()
    scores_hbt = np.ascontiguousarray(res["block_scores"].T[None])     # [1, maxB, T]
    T = pb.num_tokens
    nvis = visible_blocks(pb.seq_lens, pb.q_per_req)
    # entries a row cannot see were never written by the scorer: any value
    for t in range(T):
        scores_hbt[0, nvis[t]:, t] = 0.0
    got, status = run_rows(torch, scores_hbt, pb.seq_lens, pb.q_per_req, pb.topk,
                           hkv=pb.num_kv_heads)
    assert status == msa.MSA_OK
    assert np.array_equal(got[:, 0], res["selected"])
    check_device_ok(dp)


def test_bad_seq_len_is_reported(torch_cuda):
    scores = np.zeros((1, 8, 4), dtype=np.float32)
    got, status = run_rows(torch_cuda, scores, [0, 5], 2, 2)
    assert status == msa.MSA_ERR_DEVICE_CHECK
    assert np.all(got[:2] == -1)
