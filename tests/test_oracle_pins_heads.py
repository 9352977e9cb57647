"""Pins of the oracle's selection variants (no GPU needed): init / local
block forcing and several index heads, one selection table per KV head.

Each test checks the oracle against facts it does not compute itself:
hand-worked tables (tests/golden/select_forced.txt), exact integer brute
force of the per-head scores, an invariant every valid table must satisfy,
and a closed form of attention that only holds when each KV head reads its
own table.
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


def f64_to_bf16_bits(x):
    t = torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def golden_forced_cases():
    cases = []
    with open(os.path.join(GOLDEN, "select_forced.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, init, local, scores, want = [x.strip() for x in line.split("|")]
            cases.append((int(k), int(init), int(local), [float(x) for x in scores.split(",")],
                          [int(x) for x in want.split(",")]))
    return cases


@pytest.mark.parametrize("k,init,local,scores,want", golden_forced_cases())
def test_forced_select_hand_worked_cases(k, init, local, scores, want):
    assert oracle.select(np.array(scores), len(scores), k, init, local).tolist() == want


def check_forced_table(scores, n_valid, k, init, local, sel):
    """Every property a valid forced table has, checked from its definition."""
    forced = {b for b in range(n_valid) if b < init or b >= n_valid - local}
    chosen = [int(b) for b in sel if b >= 0]
    assert chosen == sorted(set(chosen)), "ascending, no repeats"
    assert all(b == -1 for b in sel[len(chosen):]), "-1 padding after the blocks"
    assert len(chosen) == min(k, n_valid)
    assert forced <= set(chosen)
    free_in = [b for b in chosen if b not in forced]
    free_out = [b for b in range(n_valid) if b not in forced and b not in chosen]
    for a in free_in:
        for b in free_out:
            assert scores[a] > scores[b] or (scores[a] == scores[b] and a < b)


def test_forced_select_invariant_on_random_rows_with_ties():
    rng = np.random.default_rng(5)
    for trial in range(500):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 20))
        init = int(rng.integers(0, k + 1))
        local = int(rng.integers(0, k - init + 1))
        scores = rng.integers(-3, 4, size=n).astype(np.float64)
        sel = oracle.select(scores, n, k, init, local)
        check_forced_table(scores, n, k, init, local, sel.tolist())


def test_forcing_nothing_is_the_plain_select():
    rng = np.random.default_rng(6)
    for trial in range(100):
        n = int(rng.integers(1, 30))
        k = int(rng.integers(1, 12))
        scores = rng.integers(-2, 3, size=n).astype(np.float64)
        order = sorted(range(n), key=lambda b: (-scores[b], b))
        want = sorted(order[:k]) + [-1] * max(0, k - n)
        assert oracle.select(scores, n, k, 0, 0).tolist() == want


def test_more_forced_blocks_than_places_is_refused():
    with pytest.raises(oracle.OracleError):
        oracle.select(np.zeros(10), 10, 3, 2, 2)


def int_head_scores(pb, t, head):
    """Block maxima of index head `head` by exact int64 arithmetic."""
    r = t // pb.q_per_req
    L = pb.visible(t)
    q = bf16_to_f64(pb.q_idx[t, head]).astype(np.int64)
    out = np.full(pb.max_blocks, -np.inf)
    for b in range((L + P - 1) // P):
        keys = bf16_to_f64(pb.idxk_pool[pb.block_table[r, b], head]).astype(np.int64)
        s = keys @ q
        out[b] = s[: min(P, L - b * P)].max()
    return out


@pytest.mark.parametrize("hkv,hi", [(1, 2), (2, 2), (2, 4)])
def test_per_head_scores_and_group_max_selection_bruteforce(hkv, hi):
    pb = synth.make_problem(name="heads", contexts=[700, 1300], q_per_req=2, num_kv_heads=hkv,
                            topk=3, seed=21, num_index_heads=hi, index_range=(-2, 2),
                            init_blocks=1, local_blocks=1)
    res = oracle.decode_step(pb)
    hs = 1 if hi == 1 else hkv
    assert res["block_scores"].shape == (pb.num_tokens, hi, pb.max_blocks)
    assert res["selected"].shape == (pb.num_tokens, hs, pb.topk)
    for t in range(pb.num_tokens):
        per_head = np.stack([int_head_scores(pb, t, i) for i in range(hi)])
        n_valid = (pb.visible(t) + P - 1) // P
        assert np.array_equal(res["block_scores"][t, :, :n_valid], per_head[:, :n_valid])
        r = hi // hs
        for gs in range(hs):
            red = per_head[gs * r:(gs + 1) * r].max(axis=0)[:n_valid]
            forced = [b for b in range(n_valid) if b < 1 or b >= n_valid - 1]
            rest = sorted((b for b in range(n_valid) if b not in forced),
                          key=lambda b: (-red[b], b))
            want = sorted(forced + rest[: pb.topk - len(forced)])
            want += [-1] * (pb.topk - len(want))
            assert res["selected"][t, gs].tolist() == want, (t, gs)


def test_each_kv_head_attends_over_its_own_table():
    # Two KV heads with one index head each and top-1.  Index head 0 lights
    # only block 0, index head 1 only block 2, so the tables are {0} and {2}.
    # Main keys are zero (uniform weights); V is c_g on the block KV head g
    # selected and 7 everywhere else.  Then every query head of group g gets
    # O = c_g exactly and LSE = ln(positions of that block), and any mix-up of
    # the tables shows as a 7 or the other head's constant.
    pb = synth.make_problem(name="own-table", contexts=[3 * P], q_per_req=1, num_kv_heads=2,
                            topk=1, seed=3, num_index_heads=2)
    pb.q_idx[:] = f64_to_bf16_bits(1.0)
    pb.idxk_pool[:] = 0
    pages = pb.block_table[0, :3]
    pb.idxk_pool[pages[0], 0] = f64_to_bf16_bits(1.0)
    pb.idxk_pool[pages[2], 1] = f64_to_bf16_bits(1.0)
    pb.kv_pool[:, 0] = 0                                   # K = 0
    pb.kv_pool[:, 1] = f64_to_bf16_bits(7.0)               # V = 7 by default
    c = {0: 0.5, 1: -2.0}
    pb.kv_pool[pages[0], 1, 0] = f64_to_bf16_bits(c[0])
    pb.kv_pool[pages[2], 1, 1] = f64_to_bf16_bits(c[1])
    res = oracle.decode_step(pb)
    assert res["selected"][0].tolist() == [[0], [2]]
    L = pb.visible(0)
    for h in range(pb.num_q_heads):
        g = h // 16
        assert np.all(res["out"][0, h] == c[g]), h
        n_pos = P if g == 0 else L - 2 * P
        assert math.isclose(res["lse"][0, h], math.log(n_pos), rel_tol=0, abs_tol=1e-12), h


def test_one_index_head_keeps_the_shared_table_layout():
    pb = synth.make_small_workload(1)
    res = oracle.decode_step(pb, tokens=[0, 1])
    assert res["block_scores"].shape == (2, pb.max_blocks)
    assert res["selected"].shape == (2, pb.topk)


# ---------------------------------------------------------------------------
# many query rows from a head-major score buffer (the prefill select tile)

def test_row_select_hand_worked_causal_rows():
    # three rows seeing 2, 4 and 5 blocks of one head; k = 2
    scores = np.array([[[1, 1, 1],      # block 0
                        [5, 0, 0],      # block 1
                        [9, 3, 3],      # block 2 (row 0 cannot see it)
                        [0, 3, 7],      # block 3
                        [0, 0, 7]]],    # block 4 (only row 2 sees it)
                      dtype=np.float64)
    sel = oracle.select_rows(scores, [2, 4, 5], 2)
    assert sel[:, 0].tolist() == [[0, 1], [2, 3], [3, 4]]


def test_row_select_is_the_per_token_select_of_each_row():
    # The pages: the tile select gives the same table bit for bit as the
    # per-token select, including tie order and forcing.  Checked against
    # an independent brute force of each row.
    rng = np.random.default_rng(8)
    hs, maxb, n = 2, 40, 19
    scores = rng.integers(-2, 3, size=(hs, maxb, n)).astype(np.float64)
    nvis = rng.integers(1, maxb + 1, size=n).astype(np.int32)
    k, init, local = 6, 1, 2
    sel = oracle.select_rows(scores, nvis, k, init, local)
    for t in range(n):
        for gs in range(hs):
            nv = int(nvis[t])
            row = scores[gs, :nv, t]
            forced = [b for b in range(nv) if b < init or b >= nv - local]
            rest = sorted((b for b in range(nv) if b not in forced), key=lambda b: (-row[b], b))
            want = sorted(forced + rest[: k - len(forced)])
            want += [-1] * (k - len(want))
            assert sel[t, gs].tolist() == want, (t, gs)
