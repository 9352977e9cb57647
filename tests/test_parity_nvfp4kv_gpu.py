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


def test_nvfp4_kv_late_large_logit_rescales_the_accumulated_output(torch_cuda):
    """One key row per (token, KV head) on the token's third selected page set
    to e2m1 magnitude 6 with the signs of one query head and scales 2^-1, so
    that this head's logit is about 29 in base 2, far above the first pages'
    maxima: the output accumulated in tensor memory over the first two pages
    is rescaled, and the position carries the head's softmax."""
    pb = f4_problem(4, 4, contexts=(3000, 2500), k=8, seed=63)
    sel = oracle.decode_step(pb, threads=THREADS)["selected"]
    kv = np.array(pb.kv_pool, copy=True)
    q = synth.bf16_bits_to_f32(pb.q)
    rng = np.random.default_rng(64)
    codes_bytes = 128 * 128 // 2
    planted = 0
    for t in range(pb.num_tokens):
        r = t // pb.q_per_req
        blocks = sorted(int(b) for b in sel[t] if b >= 0)
        if len(blocks) < 3:
            continue
        b = blocks[2]
        row = int(rng.integers(0, min(128, pb.visible(t) - 128 * b)))
        page = int(pb.block_table[r, b])
        for g in range(pb.num_kv_heads):
            qv = q[t, 16 * g + int(rng.integers(0, 16))]
            nib = np.where(qv < 0, 0xF, 0x7).astype(np.uint8)  # magnitude 6, sign of q
            kv[page, 0, g, row * 64:(row + 1) * 64] = nib[0::2] | (nib[1::2] << 4)
            kv[page, 0, g, codes_bytes + row * 8:codes_bytes + (row + 1) * 8] = 0x30  # E4M3 2^-1
            planted += 1
    assert planted >= pb.num_tokens
    pb.kv_pool = kv
    ref = oracle.decode_step(pb, threads=THREADS)
    assert np.array_equal(ref["selected"], sel)  # the index keys are unchanged
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens),
                           nvfp4_kv=True)
    check_device_ok(dp)
