"""Pins of the oracle's KV / index-key update (no GPU needed): where each new
token lands, the E4M3 and E2M1 encoders, and the NVFP4 group quantiser.

Checks come from outside the oracle: torch's float8_e4m3fn cast (round to
nearest even), the OCP e2m1 table (tests/golden/e2m1_ocp_mx.txt) with the
nearest value found by brute force, hand-worked groups
(tests/golden/nvfp4_groups.txt), and numpy indexing of the pools.
"""

import os

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_decode_msa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = synth.PAGE


def e2m1_table():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                code, value = line.split()
                table[int(code)] = float(value)
    return table


def torch_e4m3_codes(x32):
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def torch_e4m3_values(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).double().numpy()


def test_e4m3_encoder_matches_torch_on_every_bf16_value_in_range():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    x = synth.bf16_bits_to_f32(bits)
    keep = np.isfinite(x) & (np.abs(x) < 464)          # below the saturation boundary
    x = x[keep]
    want = torch_e4m3_codes(x)
    got = np.array([oracle.encode_e4m3(v) for v in x], dtype=np.uint8)
    zero = torch_e4m3_values(want) == 0                # torch keeps -0; the update stores +0
    assert np.array_equal(got[~zero], want[~zero])
    assert np.all(got[zero] == 0)


def test_e4m3_encoder_saturates():
    assert oracle.encode_e4m3(448.0) == 0x7E
    assert oracle.encode_e4m3(1e6) == 0x7E
    assert oracle.encode_e4m3(-1e6) == 0xFE


def test_e2m1_encoder_nearest_value_of_the_ocp_table():
    table = e2m1_table()
    mags = [(c, table[c]) for c in range(8)]
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.uniform(-8, 8, 3000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0],
                         [-0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0]])
    for x in xs:
        a = abs(x)
        # nearest magnitude, ties to the even code, saturating at 6
        best = min(mags, key=lambda cv: (abs(cv[1] - a), cv[0] & 1))[0] if a < 6 else 7
        want = 0 if best == 0 else (best | (8 if x < 0 else 0))
        assert oracle.encode_e2m1(x) == want, x
    for code, value in table.items():
        if value != 0:
            assert oracle.encode_e2m1(value) == code


def golden_groups():
    cases = []
    with open(os.path.join(GOLDEN, "nvfp4_groups.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                xs, sc, codes = [p.strip() for p in line.split("|")]
                cases.append(([float(v) for v in xs.split(",")], int(sc),
                              [int(v) for v in codes.split(",")]))
    return cases


def one_token_nvfp4_problem():
    return synth.make_problem(name="upd", contexts=[300], q_per_req=1, num_kv_heads=1, topk=2,
                              index_dtype=synth.NVFP4, seed=9)


@pytest.mark.parametrize("xs,scale_code,codes", golden_groups())
def test_nvfp4_group_quantisation_hand_worked(xs, scale_code, codes):
    pb = one_token_nvfp4_problem()
    idxk_new = np.zeros((1, 1, 128), dtype=np.uint16)
    idxk_new[0, 0, 32:48] = synth.f32_to_bf16_bits(np.array(xs, dtype=np.float32))   # group 2
    zeros = np.zeros((1, 1, 128), dtype=np.uint16)
    res = oracle.kv_update(pb, zeros, zeros, idxk_new)
    pos = int(pb.seq_lens[0]) - 1
    page, row = pb.block_table[0, pos // P], pos % P
    assert int(res["idxk_scales"][page, 0, row, 2]) == scale_code
    by = res["idxk_pool"][page, 0, row, 16:24].astype(int)
    got = [(b >> (4 * h)) & 15 for b in by for h in (0, 1)]     # dimension 2i: low nibble
    assert got == codes


def new_positions(pb):
    """(t, page, row) of every new token: position seq_len - 1 + j."""
    out = []
    for t in range(pb.num_tokens):
        r, j = divmod(t, pb.q_per_req)
        pos = int(pb.seq_lens[r]) - 1 + j
        out.append((t, pb.block_table[r, pos // P], pos % P))
    return out


def test_bf16_update_writes_exactly_the_new_rows():
    pb = synth.make_problem(name="upd", contexts=[300, 1000, 129], q_per_req=3, num_kv_heads=2,
                            topk=2, num_index_heads=2, seed=12)
    upd = synth.make_update(pb)
    res = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    kv, ik = pb.kv_pool.copy(), pb.idxk_pool.copy()
    for t, page, row in new_positions(pb):
        kv[page, 0, :, row] = upd["k_new"][t]
        kv[page, 1, :, row] = upd["v_new"][t]
        ik[page, :, row] = upd["idxk_new"][t]
    assert np.array_equal(res["kv_pool"], kv)
    assert np.array_equal(res["idxk_pool"], ik)


def test_fp8_update_matches_torch_cast_of_the_float32_quotient():
    pb = synth.make_problem(name="upd8", contexts=[700, 260], q_per_req=2, num_kv_heads=2,
                            topk=2, kv_dtype=synth.FP8, seed=13)
    pb.v_scale = pb.k_scale * 0.75      # separate scales
    upd = synth.make_update(pb)
    res = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    kv = pb.kv_pool.copy()
    for t, page, row in new_positions(pb):
        for kvi, name, scale in ((0, "k_new", pb.k_scale), (1, "v_new", pb.v_scale)):
            x = synth.bf16_bits_to_f32(upd[name][t]) / np.float32(scale)
            codes = torch_e4m3_codes(x)
            codes[torch_e4m3_values(codes) == 0] = 0
            # torch's cast overflows to NaN; the update saturates at 448 (code 0x7E)
            big = np.abs(x) >= 464
            codes[big] = np.where(x[big] < 0, 0xFE, 0x7E)
            kv[page, kvi, :, row] = codes
    assert np.array_equal(res["kv_pool"], kv)


def test_nvfp4_update_of_representable_values_is_lossless():
    pb = synth.make_problem(name="upd4", contexts=[500, 900], q_per_req=2, num_kv_heads=1,
                            topk=2, index_dtype=synth.NVFP4, num_index_heads=2, seed=14)
    upd = synth.make_update(pb, exact_nvfp4=True)
    res = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    table = e2m1_table()
    for t, page, row in new_positions(pb):
        for i in range(pb.num_index_heads):
            by = res["idxk_pool"][page, i, row].astype(int)
            codes = np.empty(128, dtype=int)
            codes[0::2], codes[1::2] = by & 15, by >> 4
            scale = np.repeat(torch_e4m3_values(res["idxk_scales"][page, i, row]), 16)
            vals = np.array([table[c] for c in codes]) * scale
            assert np.array_equal(vals, synth.bf16_bits_to_f32(upd["idxk_new"][t, i]))
    # every other page row is untouched
    mask = np.ones(pb.idxk_pool.shape[:3], dtype=bool)
    for t, page, row in new_positions(pb):
        mask[page, :, row] = False
    assert np.array_equal(res["idxk_pool"][mask], pb.idxk_pool[mask])
    assert np.array_equal(res["idxk_scales"][mask], pb.idxk_scales[mask])


# ---------------------------------------------------------------------------
# NVFP4 K / V (decode and update)

def nvfp4_kv_f64(pb, page, kv, g):
    """[128, 128] float64 values of one NVFP4 K or V tile, decoded with the
    OCP e2m1 table and torch's E4M3 decode, times the tensor scale."""
    table = e2m1_table()
    tile = pb.kv_pool[page, kv, g]
    by = tile[: P * 64].reshape(P, 64).astype(int)
    codes = np.empty((P, 128), dtype=int)
    codes[:, 0::2], codes[:, 1::2] = by & 15, by >> 4
    sc = torch_e4m3_values(tile[P * 64:].reshape(P, 8))
    vals = np.vectorize(table.get)(codes).astype(np.float64) * np.repeat(sc, 16, axis=1)
    return vals * (pb.v_scale if kv else pb.k_scale)


def test_nvfp4_kv_dense_attention_equals_sdpa():
    # k >= visible blocks: dense causal attention over torch-decoded K and V
    pb = synth.make_problem(name="f4kv", contexts=[700, 300], q_per_req=2, num_kv_heads=2,
                            topk=8, kv_dtype=synth.NVFP4, seed=15)
    pb.k_scale, pb.v_scale = 0.5, 2.0
    res = oracle.decode_step(pb)
    for t in range(pb.num_tokens):
        r = t // pb.q_per_req
        L = pb.visible(t)
        nb = (L + P - 1) // P
        for h in range(pb.num_q_heads):
            g = h // 16
            K = np.concatenate([nvfp4_kv_f64(pb, pb.block_table[r, b], 0, g) for b in range(nb)])[:L]
            V = np.concatenate([nvfp4_kv_f64(pb, pb.block_table[r, b], 1, g) for b in range(nb)])[:L]
            q = torch.from_numpy(synth.bf16_bits_to_f32(pb.q[t, h]).astype(np.float64))
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, None], torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None],
                scale=pb.softmax_scale)[0, 0, 0].numpy()
            assert np.allclose(res["out"][t, h], o, rtol=0, atol=1e-12), (t, h)


def test_nvfp4_kv_update_of_representable_values_is_lossless():
    pb = synth.make_problem(name="f4upd", contexts=[500, 129], q_per_req=2, num_kv_heads=2,
                            topk=2, kv_dtype=synth.NVFP4, seed=16)
    pb.k_scale, pb.v_scale = 0.25, 4.0
    upd = synth.make_update(pb, exact_nvfp4=True)
    # K / V inputs the format holds exactly after division by the tensor scale
    rng = np.random.default_rng(3)
    for name, scale in (("k_new", pb.k_scale), ("v_new", pb.v_scale)):
        groups = upd[name].shape[:-1] + (8, 16)
        mag = synth._E2M1_MAGNITUDES[rng.integers(0, 8, size=groups)]
        mag[..., 0] = 6.0
        x = mag * np.exp2(rng.integers(-4, 5, size=groups[:-1] + (1,))) * scale
        upd[name] = synth.f32_to_bf16_bits(x.reshape(upd[name].shape).astype(np.float32))
    new = oracle.kv_update(pb, upd["k_new"], upd["v_new"], upd["idxk_new"])
    after = synth.Problem(**{**pb.__dict__, "kv_pool": new["kv_pool"]})
    for t, page, row in new_positions(pb):
        for kv, name in ((0, "k_new"), (1, "v_new")):
            for g in range(pb.num_kv_heads):
                got = nvfp4_kv_f64(after, page, kv, g)[row]
                assert np.array_equal(got, synth.bf16_bits_to_f32(upd[name][t, g])), (t, kv, g)
