"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself:
library routines (torch's bf16 / float8 casts, scaled_dot_product_attention
in float64), published tables (tests/golden/), exact integer brute force, and
closed forms of softmax attention.  A plausible slip in the oracle -- a wrong
nibble order, a dropped scale, an off-by-one causal limit, the wrong tie
direction, a wrong query-head to KV-head map, a log in the wrong base --
fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_msa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = synth.PAGE


def bf16_to_f64(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).double().numpy()


def e4m3_to_f64(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).double().numpy()


def f64_to_bf16_bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def load_e2m1_table():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, value = line.split()
            table[int(code)] = float(value)
    return table


def tiny(contexts, nq=1, hkv=1, k=4, **kw):
    kw.setdefault("seed", 7)
    return synth.make_problem(name="pin", contexts=contexts, q_per_req=nq, num_kv_heads=hkv,
                              topk=k, **kw)


def positions(pb, t, sel):
    """(pages, token-in-page) of the visible positions of the selected blocks."""
    r = t // pb.q_per_req
    L = pb.visible(t)
    pages, toks = [], []
    for b in sel:
        if b < 0:
            continue
        for i in range(P):
            if b * P + i < L:
                pages.append(pb.block_table[r, b])
                toks.append(i)
    return np.array(pages), np.array(toks)


def kv_f64(pb, pages, toks):
    """float64 K, V [Hkv, n, D] at the given positions, dequantised by torch."""
    kv = pb.kv_pool[pages, :, :, toks, :]          # [n, 2, Hkv, D]
    if pb.kv_dtype == "fp8":
        K = e4m3_to_f64(kv[:, 0]) * pb.k_scale
        V = e4m3_to_f64(kv[:, 1]) * pb.v_scale
    else:
        K = bf16_to_f64(kv[:, 0])
        V = bf16_to_f64(kv[:, 1])
    return K.transpose(1, 0, 2), V.transpose(1, 0, 2)


def sdpa_f64(pb, t, sel):
    """Attention of token t over the selected positions by torch SDPA (float64)."""
    pages, toks = positions(pb, t, sel)
    K, V = kv_f64(pb, pages, toks)
    G = pb.num_q_heads // pb.num_kv_heads
    q = torch.from_numpy(bf16_to_f64(pb.q[t]))[None, :, None, :]            # [1, Hq, 1, D]
    k = torch.from_numpy(np.repeat(K, G, axis=0))[None]                       # [1, Hq, n, D]
    v = torch.from_numpy(np.repeat(V, G, axis=0))[None]
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=pb.softmax_scale)
    return o[0, :, 0, :].numpy()


# ---------------------------------------------------------------------------
# element decoders


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(0)
    bits = np.concatenate([rng.integers(0, 65536, 4000, dtype=np.uint16),
                           np.array([0, 0x8000, 0x3F80, 0xBF80, 0x7F80, 0xFF80, 0x0001, 0x807F],
                                    dtype=np.uint16)])
    ref = bf16_to_f64(bits)
    got = np.array([oracle.bf16(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = e4m3_to_f64(codes)
    got = np.array([oracle.e4m3(c) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # S.1111.111
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.e4m3(0x7E) == 448.0


def test_e2m1_decode_matches_ocp_table():
    table = load_e2m1_table()
    assert len(table) == 16
    for code, value in table.items():
        got = oracle.e2m1(code)
        assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value), code


def test_power_of_two_scale_codes():
    # The NVFP4 workload stores scales 2^e, e in [-4, 4], as E4M3 codes; torch decodes them.
    for e in range(-4, 5):
        code = (e + 7) << 3
        assert e4m3_to_f64(np.array([code], dtype=np.uint8))[0] == 2.0 ** e
        assert oracle.e4m3(code) == 2.0 ** e


# ---------------------------------------------------------------------------
# (a) index score + block max


def int_scores_bruteforce(pb, t):
    """Exact per-block max of integer index scores by int64 arithmetic."""
    r = t // pb.q_per_req
    L = pb.visible(t)
    q = bf16_to_f64(pb.q_idx[t, 0]).astype(np.int64)
    out = np.full(pb.max_blocks, -np.inf)
    for b in range((L + P - 1) // P):
        page = pb.block_table[r, b]
        keys = bf16_to_f64(pb.idxk_pool[page, 0]).astype(np.int64)   # [P, Di]
        s = keys @ q
        n = min(P, L - b * P)
        out[b] = s[:n].max()
    return out


def test_block_scores_integer_bruteforce():
    pb = tiny([300, 520, 129], nq=3, hkv=1, k=2, num_pages=20)
    for t in range(pb.num_tokens):
        assert np.array_equal(oracle.block_scores(pb, t), int_scores_bruteforce(pb, t)), t


def test_block_scores_nvfp4_exact_integer_arithmetic():
    pb = tiny([400, 257], nq=2, hkv=1, k=2, index_dtype="nvfp4", index_range=(-4, 4), seed=11)
    table = load_e2m1_table()
    twice = np.array([round(2 * table[c]) for c in range(16)], dtype=np.int64)   # 2*e2m1: ints
    for t in range(pb.num_tokens):
        r = t // pb.q_per_req
        L = pb.visible(t)
        q = bf16_to_f64(pb.q_idx[t, 0]).astype(np.int64)
        want = np.full(pb.max_blocks, -np.inf)
        for b in range((L + P - 1) // P):
            page = pb.block_table[r, b]
            by = pb.idxk_pool[page, 0].astype(np.int64)               # [P, 64]
            codes = np.empty((P, 128), dtype=np.int64)
            codes[:, 0::2] = by & 15                                 # dimension 2i: low nibble
            codes[:, 1::2] = by >> 4
            sc = e4m3_to_f64(pb.idxk_scales[page, 0])                # [P, 8] = 2^e
            sc16 = np.round(np.repeat(sc, 16, axis=1) * 16).astype(np.int64)  # 16*2^e: ints
            s = (twice[codes] * sc16) @ q                            # 32 * exact score
            n = min(P, L - b * P)
            want[b] = s[:n].max() / 32.0
        assert np.array_equal(oracle.block_scores(pb, t), want), t


def test_block_scores_are_exact_in_float32():
    for idx in range(5):
        pb = synth.make_small_workload(idx)
        res = oracle.decode_step(pb, tokens=[0, pb.num_tokens - 1], threads=2)
        for i, t in enumerate([0, pb.num_tokens - 1]):
            d = oracle.block_scores(pb, t)
            assert np.array_equal(res["block_scores"][i].astype(np.float64), d)


def test_causal_limit_counts_seq_len_plus_j():
    # All index keys zero except one position; query all ones.  Token j sees
    # positions < seq_len + j: the marked position lights its block only for
    # the tokens that see it.
    pb = tiny([600], nq=4, hkv=1, k=2, num_pages=8)
    pb.q_idx[:] = f64_to_bf16_bits(np.ones(1))[0]
    seq_len = int(pb.seq_lens[0])          # 597
    for j in range(4):
        L = seq_len + j
        for mark, visible in ((L - 1, True), (L, False)):
            pb.idxk_pool[:] = 0
            b, i = divmod(mark, P)
            pb.idxk_pool[pb.block_table[0, b], 0, i, :] = f64_to_bf16_bits(np.ones(1))[0]
            s = oracle.block_scores(pb, j)
            if visible:
                assert s[b] == 128.0
            else:
                assert s[b] in (0.0, -np.inf)
                if mark % P == 0:
                    assert s[b] == -np.inf  # first position of a block nobody sees yet
    # blocks past the visible range are -inf
    s = oracle.block_scores(pb, 0)
    nvis = (seq_len + P - 1) // P
    assert np.all(s[nvis:] == -np.inf) and np.all(np.isfinite(s[:nvis]))


# ---------------------------------------------------------------------------
# (b) selection


def golden_select_cases():
    cases = []
    with open(os.path.join(GOLDEN, "select_ties.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, scores, want = [x.strip() for x in line.split("|")]
            cases.append((int(k), [float(x) for x in scores.split(",")],
                          [int(x) for x in want.split(",")]))
    return cases


@pytest.mark.parametrize("k,scores,want", golden_select_cases())
def test_select_hand_worked_cases(k, scores, want):
    got = oracle.select(np.array(scores), len(scores), k)
    assert got.tolist() == want


def test_select_bruteforce_random_rows_with_ties():
    rng = np.random.default_rng(3)
    for trial in range(400):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 20))
        scores = rng.integers(-3, 4, size=n).astype(np.float64)   # heavy ties
        order = sorted(range(n), key=lambda b: (-scores[b], b))
        want = sorted(order[:k]) + [-1] * max(0, k - n)
        assert oracle.select(scores, n, k).tolist() == want


def test_select_ignores_blocks_past_the_valid_count():
    scores = np.array([1.0, 2.0, 3.0, 100.0, 100.0])
    assert oracle.select(scores, 3, 2).tolist() == [1, 2]


def test_selection_invariant_on_workloads():
    for idx in range(5):
        pb = synth.make_small_workload(idx)
        res = oracle.decode_step(pb, threads=4)
        for i in range(pb.num_tokens):
            n_valid = (pb.visible(i) + P - 1) // P
            bs = res["block_scores"][i][:n_valid]
            sel = res["selected"][i]
            chosen = sel[sel >= 0]
            assert len(chosen) == min(pb.topk, n_valid)
            assert np.all(np.diff(chosen) > 0) and np.all(sel[len(chosen):] == -1)
            rest = np.setdiff1d(np.arange(n_valid), chosen)
            for b in chosen:
                # every chosen block beats every unchosen one: higher score, or equal and smaller
                assert np.all((bs[b] > bs[rest]) | ((bs[b] == bs[rest]) & (b < rest)))


def test_all_zero_index_keys_select_the_first_blocks():
    pb = tiny([2000], nq=2, hkv=1, k=5, num_pages=20)
    pb.idxk_pool[:] = 0
    res = oracle.decode_step(pb)
    assert res["selected"].tolist() == [[0, 1, 2, 3, 4]] * 2
    assert np.all(res["block_scores"][:, :16] == 0.0)


def test_heavy_tie_workload_really_ties_at_kth_place():
    # The long-context workload's small copy: most tokens have a tie that
    # straddles the k-th place, so the tie-break decides the table.
    pb = synth.make_small_workload(2)
    res = oracle.decode_step(pb, threads=4)
    straddle = 0
    for i in range(pb.num_tokens):
        n_valid = (pb.visible(i) + P - 1) // P
        s = np.sort(res["block_scores"][i][:n_valid])[::-1]
        straddle += int(s[pb.topk - 1] == s[pb.topk])
    assert straddle >= pb.num_tokens // 2


# ---------------------------------------------------------------------------
# (c) attention


def test_dense_case_equals_sdpa_bf16():
    # top-k covering every block reduces the method to dense causal attention
    pb = tiny([700, 333], nq=3, hkv=2, k=8, seed=5)
    res = oracle.decode_step(pb)
    for t in range(pb.num_tokens):
        n_valid = (pb.visible(t) + P - 1) // P
        assert res["selected"][t].tolist() == list(range(n_valid)) + [-1] * (8 - n_valid)
        ref = sdpa_f64(pb, t, range(n_valid))
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-12)


def test_sparse_case_equals_sdpa_over_selected_positions():
    pb = synth.make_small_workload(1)
    res = oracle.decode_step(pb, threads=4)
    for t in range(pb.num_tokens):
        ref = sdpa_f64(pb, t, res["selected"][t])
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-12)


def test_fp8_kv_equals_sdpa_on_torch_decoded_values_with_separate_scales():
    pb = tiny([900], nq=2, hkv=2, k=3, kv_dtype="fp8", seed=9)
    pb.k_scale, pb.v_scale = 0.0125, 0.03   # distinct scales: each must be applied to its own tensor
    res = oracle.decode_step(pb)
    for t in range(pb.num_tokens):
        ref = sdpa_f64(pb, t, res["selected"][t])
        np.testing.assert_allclose(res["out"][t], ref, rtol=0, atol=1e-12)


def test_zero_keys_give_uniform_weights():
    pb = tiny([1000], nq=2, hkv=1, k=3, seed=4)
    pb.kv_pool[:, 0] = 0                      # K = 0: every logit 0
    res = oracle.decode_step(pb)
    for t in range(pb.num_tokens):
        pages, toks = positions(pb, t, res["selected"][t])
        V = bf16_to_f64(pb.kv_pool[pages, 1, 0, toks, :])      # [n, D]
        np.testing.assert_allclose(res["out"][t], np.broadcast_to(V.mean(0), (16, 128)),
                                   rtol=0, atol=1e-13)
        np.testing.assert_allclose(res["lse"][t], np.full(16, math.log(len(pages))), atol=1e-13)


def test_constant_values_give_that_value():
    pb = tiny([800], nq=1, hkv=2, k=3, seed=8)
    pb.kv_pool[:, 1, 0] = f64_to_bf16_bits(np.full(1, 1.5))[0]
    pb.kv_pool[:, 1, 1] = f64_to_bf16_bits(np.full(1, -0.75))[0]
    res = oracle.decode_step(pb)
    # query heads 0..15 use KV head 0, heads 16..31 KV head 1
    np.testing.assert_allclose(res["out"][0, :16], 1.5, atol=1e-14)
    np.testing.assert_allclose(res["out"][0, 16:], -0.75, atol=1e-14)


def test_single_visible_position():
    pb = tiny([1], nq=1, hkv=1, k=2, seed=2)
    pb.softmax_scale = 1.0
    page = pb.block_table[0, 0]
    pb.q[0] = 0
    pb.q[0, :, 5] = f64_to_bf16_bits(np.full(1, 2.0))[0]
    pb.kv_pool[page, 0, 0, 0] = 0
    pb.kv_pool[page, 0, 0, 0, 5] = f64_to_bf16_bits(np.full(1, 1.25))[0]
    res = oracle.decode_step(pb)
    v0 = bf16_to_f64(pb.kv_pool[page, 1, 0, 0])
    assert res["selected"][0].tolist() == [0, -1]
    np.testing.assert_array_equal(res["out"][0], np.broadcast_to(v0, (16, 128)))
    np.testing.assert_allclose(res["lse"][0], 2.5, atol=0)      # z = 2 * 1.25, one term


def test_two_positions_logsumexp_closed_form():
    pb = tiny([2], nq=1, hkv=1, k=1, seed=6)
    pb.softmax_scale = 1.0
    page = pb.block_table[0, 0]
    pb.q[0] = 0
    pb.q[0, :, 0] = f64_to_bf16_bits(np.ones(1))[0]
    pb.kv_pool[page, 0, 0, :2] = 0
    a, b = 0.5, -1.75
    pb.kv_pool[page, 0, 0, 0, 0] = f64_to_bf16_bits(np.full(1, a))[0]
    pb.kv_pool[page, 0, 0, 1, 0] = f64_to_bf16_bits(np.full(1, b))[0]
    pb.kv_pool[page, 1, 0, 0] = f64_to_bf16_bits(np.full(1, 3.0))[0]
    pb.kv_pool[page, 1, 0, 1] = f64_to_bf16_bits(np.full(1, -1.0))[0]
    res = oracle.decode_step(pb)
    lse = math.log(math.exp(a) + math.exp(b))      # natural log of the softmax denominator
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(res["lse"][0], lse, atol=1e-15)
    np.testing.assert_allclose(res["out"][0], 3.0 * wa - 1.0 * (1 - wa), atol=1e-15)


def test_query_head_to_kv_head_map_is_consecutive_groups_of_16():
    pb = tiny([300], nq=1, hkv=4, k=3, seed=12)
    for g in range(4):
        pb.kv_pool[:, 1, g] = f64_to_bf16_bits(np.full(1, float(g + 1)))[0]
    res = oracle.decode_step(pb)
    for h in range(64):
        np.testing.assert_allclose(res["out"][0, h], h // 16 + 1, atol=1e-14)


def test_attention_causal_limit():
    pb = tiny([520], nq=4, hkv=1, k=5, seed=13)   # 5 blocks, k covers them all
    base = oracle.decode_step(pb)
    for j in range(4):
        L = pb.visible(j)
        for pos, changes in ((L, False), (L - 1, True)):
            mod = tiny([520], nq=4, hkv=1, k=5, seed=13)
            b, i = divmod(pos, P)
            page = mod.block_table[0, b]
            mod.kv_pool[page, 1, 0, i] = f64_to_bf16_bits(np.full(1, 50.0))[0]
            out = oracle.decode_step(mod)["out"][j]
            assert (not np.array_equal(out, base["out"][j])) == changes, (j, pos)


@pytest.mark.parametrize("kv_dtype", [synth.BF16, synth.FP8, synth.NVFP4])
def test_pages_are_reached_only_through_the_block_table(kv_dtype):
    # moving every page of the pools to another slot and renumbering the
    # block table changes no result: a page read by its block number, or a
    # table entry used for the wrong request, breaks this
    import dataclasses

    pb = synth.make_problem(name="perm", contexts=[300, 1000, 129], q_per_req=2, num_kv_heads=2,
                            topk=4, kv_dtype=kv_dtype, guard_page=True, seed=91)
    perm = np.random.default_rng(92).permutation(pb.num_pages)

    def moved(pool):
        out = np.empty_like(pool)
        out[perm] = pool
        return out

    bt = pb.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    assert not np.array_equal(bt, pb.block_table)
    pb2 = dataclasses.replace(pb, kv_pool=moved(pb.kv_pool), idxk_pool=moved(pb.idxk_pool),
                              block_table=bt)
    r1 = oracle.decode_step(pb, threads=2)
    r2 = oracle.decode_step(pb2, threads=2)
    for key in ("block_scores", "selected", "out", "lse"):
        assert np.array_equal(r1[key], r2[key]), key
    # and a table that points at the wrong pages does change the result
    bt_bad = pb.block_table.copy()
    bt_bad[0, :2] = bt_bad[0, 1::-1]
    r3 = oracle.decode_step(dataclasses.replace(pb, block_table=bt_bad), threads=2)
    assert not np.array_equal(r3["block_scores"], r1["block_scores"])


def test_decode_step_matches_stagewise_calls():
    pb = synth.make_small_workload(4)
    res = oracle.decode_step(pb, threads=3)
    for t in range(pb.num_tokens):
        bs = oracle.block_scores(pb, t)
        n_valid = (pb.visible(t) + P - 1) // P
        sel = oracle.select(bs, n_valid, pb.topk)
        out, lse = oracle.attend(pb, t, sel)
        assert np.array_equal(res["selected"][t], sel)
        assert np.array_equal(res["out"][t], out) and np.array_equal(res["lse"][t], lse)


def test_out_of_range_page_is_reported():
    pb = tiny([300], nq=1, hkv=1, k=2, num_pages=4)
    pb.block_table[0, 1] = 99
    with pytest.raises(oracle.OracleError):
        oracle.decode_step(pb)
