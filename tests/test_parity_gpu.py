"""Parity of the CUDA path with the CPU oracle, stage by stage and fused.

Tolerances (the workload contract): block scores and selected tables are
bit-exact; the bf16 output is within 4e-3 max abs of the float64 oracle and
the LSE within 1e-4 * max(|lse|, 1).
"""

import os

import numpy as np
import pytest

import oracle
from sparse_attention_decode_msa_gb300 import synth

pytestmark = pytest.mark.gpu

OUT_ATOL = 4e-3
LSE_RTOL = 1e-4
THREADS = max(1, min(32, os.cpu_count() or 1))


def device_problem(pb, **kw):
    from sparse_attention_decode_msa_gb300.runner import DeviceProblem

    return DeviceProblem(pb, **kw)


def assert_scores_equal(pb, gpu_bs, ref_bs, tokens):
    nb = pb.blocks_per_request()
    for i, t in enumerate(tokens):
        n = int(nb[t // pb.q_per_req])
        got, want = gpu_bs[t, :n], ref_bs[i, :n]
        assert np.array_equal(got, want), (t, np.flatnonzero(got != want)[:8])


def half_ulp_bf16(x):
    """Half a bf16 ulp at |x|: the most that rounding the output to bf16 can add."""
    _, e = np.frexp(np.abs(x))
    return np.where(x == 0, 0.0, np.ldexp(1.0, e - 9))


def visible_positions(pb, selected, tokens):
    """Positions each token of `tokens` attends to (the visible positions of
    its selected blocks; the fewest over its selection heads)."""
    sel = np.asarray(selected).reshape(len(tokens), -1, pb.topk)
    out = np.empty(len(tokens), dtype=np.int64)
    for i, t in enumerate(tokens):
        L = int(pb.seq_lens[t // pb.q_per_req]) + t % pb.q_per_req
        b = sel[i].astype(np.int64)
        n = np.where(b >= 0, np.clip(L - 128 * b, 0, 128), 0).sum(axis=-1)
        out[i] = n.min()
    return out


def assert_attention_close(gpu_out, gpu_lse, ref_out, ref_lse, tokens, visible=None,
                           nvfp4_kv=False):
    """|dO| <= 4e-3 and rel |dLSE| <= 1e-4 (the workload contract), with the
    bf16 storage allowance of the design's output-tolerance reading: an
    element may add half a bf16 ulp of the reference where that rounding
    alone can exceed 4e-3 (|O_ref| >= 2, half an ulp >= 7.8e-3), or where the
    token sees at most two positions (`visible`, per token of `tokens`: O is
    then one or two values of V).  nvfp4_kv: NVFP4 values reach 6, the
    allowance holds for every element."""
    tokens = list(tokens)
    out = gpu_out[tokens]
    lse = gpu_lse[tokens]
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    diff = np.abs(out - ref_out)
    allow = np.abs(ref_out) >= 2.0
    if visible is not None:
        few = np.asarray(visible) <= 2
        allow |= few.reshape((-1,) + (1,) * (ref_out.ndim - 1))
    if nvfp4_kv:
        allow[...] = True
    bound = OUT_ATOL + np.where(allow, half_ulp_bf16(ref_out), 0.0)
    excess = (diff - bound).max()
    assert excess <= 0, (f"max |dO| beyond the bound by {excess} (max |dO| = {diff.max()}, "
                         f"{int(allow.sum())} of {allow.size} elements with the bf16 allowance)")
    lerr = (np.abs(lse - ref_lse) / np.maximum(np.abs(ref_lse), 1.0)).max()
    assert lerr <= LSE_RTOL, f"max rel |dLSE| = {lerr}"


def check_device_ok(dp):
    import sparse_attention_decode_msa_gb300 as msa

    assert msa.msa_check_device_status(dp.ws) == msa.MSA_OK


# ---------------------------------------------------------------------------
# stage by stage, small copies of the five workloads


@pytest.mark.parametrize("idx", range(5))
def test_index_score_is_bit_exact(torch_cuda, idx):
    pb = synth.make_small_workload(idx)
    dp = device_problem(pb)
    dp.index_score()
    res = dp.results()
    ref = oracle.decode_step(pb, threads=THREADS)
    assert_scores_equal(pb, res["block_scores"], ref["block_scores"], range(pb.num_tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("nq", [1, 3, 8, 9, 16, 17, 33, 48, 64])
@pytest.mark.parametrize("index_dtype", [synth.BF16, synth.NVFP4])
def test_index_score_across_query_counts(torch_cuda, nq, index_dtype):
    # both scorers (mma.sync for up to 8 query tokens per request or NVFP4
    # keys, tcgen05 above), ragged contexts (cached tokens, >= nq): one
    # position for the first query token, page edges, and a request with more
    # pages than there are CTAs
    ctx = [nq, nq + 127, max(nq, 128), nq + 128, 700, 2000, 40000]
    pb = synth.make_problem(name=f"nq{nq}", contexts=ctx, q_per_req=nq, num_kv_heads=1, topk=4,
                            index_dtype=index_dtype,
                            index_range=(-4, 4) if index_dtype == synth.NVFP4 else (-8, 8),
                            guard_page=True, seed=300 + nq)
    dp = device_problem(pb)
    dp.index_score()
    res = dp.results()
    rng = np.random.default_rng(nq)
    tokens = sorted(set(rng.choice(pb.num_tokens, size=min(pb.num_tokens, 40), replace=False).tolist())
                    | {0, pb.num_tokens - 1})
    nb = pb.blocks_per_request()
    for t in tokens:
        want = oracle.block_scores(pb, t)
        n = int(nb[t // pb.q_per_req])
        assert np.array_equal(res["block_scores"][t, :n], want[:n]), (t, nq)
    check_device_ok(dp)


@pytest.mark.parametrize("nq", [1, 2])
def test_nvfp4_index_score_with_many_requests(torch_cuda, nq):
    # 3000 requests: the per-request page offsets leave no room for the deep
    # page ring of the NVFP4 scorer, which then runs with the shallow one
    rng = np.random.default_rng(40 + nq)
    ctx = rng.integers(nq, 600, size=3000)
    pb = synth.make_problem(name=f"many{nq}", contexts=ctx, q_per_req=nq, num_kv_heads=1, topk=2,
                            index_dtype=synth.NVFP4, index_range=(-4, 4), guard_page=True,
                            seed=500 + nq)
    dp = device_problem(pb)
    dp.index_score()
    res = dp.results()
    tokens = sorted(set(rng.choice(pb.num_tokens, size=40, replace=False).tolist())
                    | {0, pb.num_tokens - 1})
    nb = pb.blocks_per_request()
    for t in tokens:
        want = oracle.block_scores(pb, t)
        n = int(nb[t // pb.q_per_req])
        assert np.array_equal(res["block_scores"][t, :n], want[:n]), (t, nq)
    check_device_ok(dp)


@pytest.mark.parametrize("idx", range(5))
def test_select_is_bit_exact_on_oracle_scores(torch_cuda, idx):
    torch = torch_cuda
    pb = synth.make_small_workload(idx)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    bs = torch.from_numpy(ref["block_scores"][:, None, :].copy()).cuda()
    dp.select(block_scores=bs)
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    check_device_ok(dp)


@pytest.mark.parametrize("idx", range(5))
def test_sparse_decode_matches_oracle_on_oracle_selection(torch_cuda, idx):
    torch = torch_cuda
    pb = synth.make_small_workload(idx)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    sel = torch.from_numpy(ref["selected"][:, None, :].copy()).cuda()
    dp.sparse_decode(selected=sel)
    res = dp.results()
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("jump", [11.5, 24.0])
def test_a_late_large_logit_rescales_the_accumulated_output(torch_cuda, jump):
    """One key per (token, KV head) on the token's third selected page, along
    one query head so that its logit is `jump` in base 2 (the others about
    N(0, 1.44^2)): at 11.5 it passes the running maximum of the first two
    pages (about 4) by less than the decode's rescale slack of 8, so the
    reference stays and P of that position is about 2^7 (it carries about
    half the head's softmax); at 24 by more, so the output accumulated in
    tensor memory so far is rescaled and the position carries the whole
    softmax.  Both must match the oracle."""
    import dataclasses

    pb = synth.make_small_workload(1)
    sel = oracle.decode_step(pb, threads=THREADS)["selected"]
    kv = np.array(pb.kv_pool, copy=True)
    q = synth.bf16_bits_to_f32(pb.q).astype(np.float64)
    rng = np.random.default_rng(31)
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
            alpha = jump / (pb.softmax_scale * np.log2(np.e) * float(qv @ qv))
            kv[page, 0, g, row] = synth.f32_to_bf16_bits((alpha * qv).astype(np.float32))
            planted += 1
    assert planted >= pb.num_tokens
    pb2 = dataclasses.replace(pb, kv_pool=kv)
    ref = oracle.decode_step(pb2, threads=THREADS)
    assert np.array_equal(ref["selected"], sel)  # the index keys are unchanged
    dp = device_problem(pb2)
    dp.decode_step()
    res = dp.results()
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("idx", range(5))
def test_decode_step_matches_oracle(torch_cuda, idx):
    pb = synth.make_small_workload(idx)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    tokens = range(pb.num_tokens)
    assert_scores_equal(pb, res["block_scores"], ref["block_scores"], tokens)
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], tokens)
    check_device_ok(dp)


# ---------------------------------------------------------------------------
# the five workloads at full size, in the launch configuration the benchmark times


@pytest.mark.parametrize("idx", range(5))
def test_full_workload(torch_cuda, idx):
    pb = synth.make_workload(idx)
    dp = device_problem(pb)
    dp.decode_step(keep_intermediates=True)
    res = dp.results()
    # every token: scores, selection; attention on every token of the small
    # workloads and on a seeded sample of the big ones
    T = pb.num_tokens
    rng = np.random.default_rng(1234 + idx)
    tokens = np.arange(T) if T <= 64 else np.sort(rng.choice(T, size=64, replace=False))
    ref = oracle.decode_step(pb, tokens=tokens, threads=THREADS)
    assert_scores_equal(pb, res["block_scores"], ref["block_scores"], tokens)
    assert np.array_equal(res["selected"][tokens], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], tokens)
    assert np.all(np.isfinite(res["out"])) and np.all(np.isfinite(res["lse"]))
    check_device_ok(dp)


# ---------------------------------------------------------------------------
# properties and edge cases


@pytest.mark.parametrize("idx", [1, 3])
@pytest.mark.parametrize("ctas", [1, 2, 5, 37, 152, 600])
def test_result_does_not_depend_on_the_split(torch_cuda, idx, ctas):
    pb = synth.make_small_workload(idx)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb, decode_ctas=ctas)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))
    check_device_ok(dp)


def test_repeated_steps_are_bitwise_identical(torch_cuda):
    pb = synth.make_small_workload(2)
    dp = device_problem(pb)
    dp.decode_step()
    a = dp.results()
    dp.decode_step()
    b = dp.results()
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_select_random_rows_with_heavy_ties(torch_cuda):
    torch = torch_cuda
    import sparse_attention_decode_msa_gb300 as msa

    rng = np.random.default_rng(77)
    # one warp per token (maxB <= 256: 8 keys a lane), four warps per token
    # (maxB <= 2048: 4, 8 or 16 keys a lane) and the radix select of one CTA
    # per token (longer rows); -0.0 and +0.0 are the same score
    for k, maxB, R in [(1, 40, 64), (16, 256, 30), (16, 1024, 48), (32, 1024, 24), (2, 513, 20),
                       (33, 700, 20), (200, 256, 9), (64, 2048, 10), (16, 1500, 7),
                       (256, 3000, 12), (7, 9216, 4)]:
        seq_lens = rng.integers(1, maxB * 128 + 1, size=R).astype(np.int32)
        scores = rng.integers(-3, 4, size=(R, 1, maxB)).astype(np.float32)
        scores[(scores == 0) & (rng.random(scores.shape) < 0.5)] = -0.0
        shape = msa.make_shape(num_requests=R, q_per_req=1, num_kv_heads=1, num_pages=1,
                               max_blocks_per_seq=maxB, topk=k)
        ws_bytes = msa.msa_workspace_bytes(shape)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
        sel = torch.empty((R, 1, k), dtype=torch.int32, device="cuda")
        msa.msa_select_topk(shape, torch.from_numpy(scores).cuda(),
                            torch.from_numpy(seq_lens).cuda(), sel, ws, ws_bytes)
        got = sel.cpu().numpy()[:, 0]
        for r in range(R):
            n = -(-int(seq_lens[r]) // 128)
            order = sorted(range(n), key=lambda b: (-scores[r, 0, b], b))
            want = sorted(order[:k]) + [-1] * max(0, k - n)
            assert got[r].tolist() == want, (k, maxB, r)
        assert msa.msa_check_device_status(ws) == msa.MSA_OK


def test_short_contexts_pad_with_minus_one_and_single_position(torch_cuda):
    pb = synth.make_problem(name="short", contexts=[1, 2, 129, 300, 1000], q_per_req=1,
                            num_kv_heads=2, topk=8, seed=21)
    ref = oracle.decode_step(pb)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert res["selected"][0].tolist() == [0] + [-1] * 7
    assert np.array_equal(res["selected"], ref["selected"])
    tokens = range(pb.num_tokens)
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], tokens,
                           visible=visible_positions(pb, ref["selected"], tokens))


def test_page_aligned_contexts_and_dense_coverage(torch_cuda):
    # contexts that are multiples of 128 and top-k covering every block (dense attention)
    pb = synth.make_problem(name="aligned", contexts=[1024, 2048, 128], q_per_req=2,
                            num_kv_heads=1, topk=16, seed=22)
    ref = oracle.decode_step(pb)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))


def test_all_zero_index_keys_tie_everywhere(torch_cuda):
    pb = synth.make_problem(name="zeros", contexts=[5000, 3000], q_per_req=3, num_kv_heads=1,
                            topk=16, seed=23)
    pb.idxk_pool[:] = 0
    ref = oracle.decode_step(pb)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.all(res["selected"] == np.arange(16))
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))


def test_max_topk_and_wide_block_table(torch_cuda):
    pb = synth.make_problem(name="wide", contexts=[40000], q_per_req=2, num_kv_heads=1,
                            topk=256, max_blocks=4000, seed=24)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))


def test_largest_request_count(torch_cuda):
    # 8192 requests, the most a call takes: the bf16 scorer's page ring then
    # shares shared memory with the largest per-request page offsets (its
    # tightest configuration); every token's scores and selection, attention
    # on a seeded sample
    rng = np.random.default_rng(60)
    ctx = rng.integers(1, 260, size=8192)
    pb = synth.make_problem(name="maxR", contexts=ctx, q_per_req=1, num_kv_heads=1, topk=1,
                            seed=61)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    tokens = np.sort(rng.choice(pb.num_tokens, size=256, replace=False))
    ref = oracle.decode_step(pb, tokens=tokens, threads=THREADS)
    assert_scores_equal(pb, res["block_scores"], ref["block_scores"], tokens)
    assert np.array_equal(res["selected"][tokens], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], tokens,
                           visible=visible_positions(pb, ref["selected"], tokens))
    check_device_ok(dp)


@pytest.mark.parametrize("kv_dtype", [synth.BF16, synth.FP8])
def test_permuting_the_page_pool_changes_nothing(torch_cuda, kv_dtype):
    # pages are data addressed through the block table: moving every page of
    # the pools to another slot and renumbering the table leaves every output
    # bit for bit (no physical page id reaches the arithmetic or the order)
    import dataclasses

    pb = synth.make_problem(name="perm", contexts=[700, 3000, 129, 9000], q_per_req=3,
                            num_kv_heads=2, topk=6, kv_dtype=kv_dtype, guard_page=True, seed=77)
    rng = np.random.default_rng(78)
    perm = rng.permutation(pb.num_pages)  # old page p -> slot perm[p]
    def moved(pool):
        out = np.empty_like(pool)
        out[perm] = pool
        return out
    bt = pb.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    pb2 = dataclasses.replace(pb, kv_pool=moved(pb.kv_pool), idxk_pool=moved(pb.idxk_pool),
                              block_table=bt)
    results = []
    for p in (pb, pb2):
        dp = device_problem(p)
        dp.decode_step()
        results.append(dp.results())
        check_device_ok(dp)
    for key in ("block_scores", "selected", "out", "lse"):
        a, b = results[0][key], results[1][key]
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), key


def test_large_speculative_step(torch_cuda):
    pb = synth.make_problem(name="nq64", contexts=[3000], q_per_req=64, num_kv_heads=1, topk=8,
                            index_range=(-2, 2), seed=25)
    ref = oracle.decode_step(pb, threads=THREADS)
    dp = device_problem(pb)
    dp.decode_step()
    res = dp.results()
    assert_scores_equal(pb, res["block_scores"], ref["block_scores"], range(pb.num_tokens))
    assert np.array_equal(res["selected"], ref["selected"])
    assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"], range(pb.num_tokens))


def test_bad_page_id_is_reported_not_faulted(torch_cuda):
    import sparse_attention_decode_msa_gb300 as msa

    pb = synth.make_problem(name="badpage", contexts=[700], q_per_req=1, num_kv_heads=1, topk=4,
                            seed=26)
    pb.block_table[0, 2] = pb.num_pages + 5   # out of the pool: the kernels must not read it
    dp = device_problem(pb)
    dp.decode_step()
    assert msa.msa_check_device_status(dp.ws) == msa.MSA_ERR_DEVICE_CHECK
    assert msa.msa_check_device_status(dp.ws) == msa.MSA_OK   # the check clears the word


def test_bad_seq_len_is_reported_not_faulted(torch_cuda):
    import sparse_attention_decode_msa_gb300 as msa

    pb = synth.make_problem(name="badlen", contexts=[700, 900], q_per_req=1, num_kv_heads=1,
                            topk=4, seed=27)
    pb.seq_lens[1] = pb.max_blocks * 128 + 1   # more blocks than the table holds
    dp = device_problem(pb)
    dp.decode_step()
    assert msa.msa_check_device_status(dp.ws) == msa.MSA_ERR_DEVICE_CHECK


def test_bad_seq_len_is_reported_by_the_decode_alone(torch_cuda):
    # the decode reads seq_lens itself: called without the scorer and the
    # select, it reports a token whose seq_len does not fit the block table
    torch = torch_cuda
    import sparse_attention_decode_msa_gb300 as msa

    pb = synth.make_problem(name="badlen-decode", contexts=[700, 900], q_per_req=1,
                            num_kv_heads=1, topk=4, seed=28)
    sel = torch.tensor([[[0, 1, 2, 5]], [[0, 1, 2, 3]]], dtype=torch.int32, device="cuda")
    for bad in (0, pb.max_blocks * 128 + 1):
        pb.seq_lens[1] = bad
        dp = device_problem(pb)
        dp.sparse_decode(selected=sel)
        assert msa.msa_check_device_status(dp.ws) == msa.MSA_ERR_DEVICE_CHECK, bad


@pytest.mark.parametrize("kv_dtype", [synth.BF16, synth.FP8, synth.NVFP4])
def test_a_wait_that_runs_out_reports_timeout_and_the_next_call_is_exact(torch_cuda, kv_dtype):
    # With a wait limit of a few clocks the decode gives up at its first wait
    # that is not already complete: every CTA stops, drains its copies and
    # tensor-core work in flight (with the normal limit), frees its tensor
    # memory and exits; the call reports MSA_ERR_TIMEOUT.  After the workspace
    # is re-initialised the same call gives the oracle's result.
    torch = torch_cuda
    import sparse_attention_decode_msa_gb300 as msa

    pb = synth.make_problem(name="timeout", contexts=[3000, 1300, 5000], q_per_req=2,
                            num_kv_heads=2, topk=6, kv_dtype=kv_dtype, seed=29)
    if kv_dtype == synth.NVFP4:
        pb.k_scale, pb.v_scale = 0.75, 0.5
    ref = oracle.decode_step(pb, threads=THREADS)
    sel = torch.from_numpy(ref["selected"][:, None, :].copy()).cuda()
    for ctas in (3, 0):  # split units (the merge path) and the default one CTA per SM
        dp = device_problem(pb, decode_ctas=ctas)
        msa.msa_set_decode_wait_limit(4)
        try:
            dp.sparse_decode(selected=sel)
            status = msa.msa_check_device_status(dp.ws)
        finally:
            msa.msa_set_decode_wait_limit(0)
        assert status == msa.MSA_ERR_TIMEOUT, msa.status_string(status)
        msa.msa_workspace_init(dp.ws, dp.ws_bytes)
        dp.sparse_decode(selected=sel)
        res = dp.results()
        assert_attention_close(res["out"], res["lse"], ref["out"], ref["lse"],
                               range(pb.num_tokens), nvfp4_kv=kv_dtype == synth.NVFP4)
        check_device_ok(dp)
