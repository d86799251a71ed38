"""Pins for the fp64 oracle, against things other than the oracle itself.

* the pages' worked example (golden fixture, printed to 4 decimals);
* the pages' cache-size figures (closed form);
* library routines: torch's float16 / bfloat16 / float8_e4m3fn / float8_e5m2
  conversions and
  torch's scaled_dot_product_attention (``enable_gqa=True``) in float64, on
  fixed workloads and on random small shapes (hypothesis, derandomized);
* structural facts the pages state: G = 1 is MHA, GQA equals MHA on a
  repeat_kv-expanded cache, query head h reads KV head floor(h / G), heads that
  share K/V still differ, softmax weights sum to 1;
* special cases with a closed form: one token returns its V row, identical keys
  (or a zero query) return the mean of V, a dominant key returns its V row, a
  uniform score shift or a token permutation changes nothing.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

from grouped_query_attention_11_b300.workloads import (Workload, make_inputs,
                                                       small_variant, WORKLOADS)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden",
                      "worked_example_2.txt")


def _read_golden(path):
    meta, k, v, q, w, out = {}, {}, {}, {}, {}, {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tag, *rest = line.split()
            if tag in ("Hq", "Hkv", "D", "S"):
                meta[tag] = int(rest[0])
            elif tag in ("scale_inv_sqrt", "tol"):
                meta[tag] = float(rest[0])
            elif tag in ("k", "v"):
                (k if tag == "k" else v)[(int(rest[0]), int(rest[1]))] = \
                    [float(x) for x in rest[2:]]
            elif tag in ("q", "w", "out"):
                {"q": q, "w": w, "out": out}[tag][int(rest[0])] = \
                    [float(x) for x in rest[1:]]
    Hq, Hkv, D, S = meta["Hq"], meta["Hkv"], meta["D"], meta["S"]
    K = np.zeros((1, Hkv, S, D))
    V = np.zeros((1, Hkv, S, D))
    for (j, t), vals in k.items():
        K[0, j, t] = vals
    for (j, t), vals in v.items():
        V[0, j, t] = vals
    Q = np.array([[q[h] for h in range(Hq)]])
    W = np.array([w[h] for h in range(Hq)])
    O = np.array([out[h] for h in range(Hq)])
    scale = 1.0 / math.sqrt(meta["scale_inv_sqrt"])
    return Q, K, V, scale, W, O, meta["tol"]


# ------------------------------------------------------------- worked example

def test_worked_example_2_outputs(oracle_mod):
    Q, K, V, scale, W, O, tol = _read_golden(GOLDEN)
    out = oracle_mod.gqa_decode(Q, K, V, [K.shape[2]], scale)
    assert np.max(np.abs(out[0] - O)) <= tol + 1e-12


def test_worked_example_2_weights(oracle_mod):
    Q, K, V, scale, W, O, tol = _read_golden(GOLDEN)
    for h in range(Q.shape[1]):
        w, row = oracle_mod.gqa_weights(Q, K, V, [K.shape[2]], scale, 0, h)
        assert np.max(np.abs(w - W[h])) <= tol + 1e-12
        assert abs(w.sum() - 1.0) < 1e-12


def test_worked_example_2_shared_kv_heads_differ(oracle_mod):
    # Heads 0 and 1 read the same K/V but their outputs differ (the page's
    # "misconception" section): the softmax follows each head's own query.
    Q, K, V, scale, *_ = _read_golden(GOLDEN)
    out = oracle_mod.gqa_decode(Q, K, V, [2], scale)
    assert np.max(np.abs(out[0, 0] - out[0, 1])) > 0.5
    np.testing.assert_allclose(out[0, 0], out[0, 1][::-1], atol=1e-12)


# --------------------------------------------------------------- cache sizes

@pytest.mark.parametrize("args,expected", [
    ((80, 8, 128, 2), 327_680),      # 70B GQA-8: 320 KiB/token
    ((80, 64, 128, 2), 2_621_440),   # 70B as MHA: 2.5 MiB/token
    ((80, 1, 128, 2), 40_960),       # 70B as MQA: 40 KiB/token
    ((32, 32, 128, 2), 524_288),     # 8B-class MHA: 512 KiB
    ((32, 8, 128, 2), 131_072),      # 8B-class GQA-8: 128 KiB
    ((32, 1, 128, 2), 16_384),       # 8B-class MQA: 16 KiB
    ((32, 8, 128, 1), 65_536),       # GQA-8 with FP8 cache: 64 KiB
    ((40, 40, 128, 2), 819_200),     # 40-layer, 40-head example, MHA
    ((40, 8, 128, 2), 163_840),      # same at GQA-8 (5x smaller)
])
def test_kv_bytes_per_token(oracle_mod, args, expected):
    assert oracle_mod.kv_bytes_per_token(*args) == expected


def test_kv_cache_totals(oracle_mod):
    # 70B, 16 sequences x 4096 tokens: 171.799 GB (MHA), 21.475 GB (GQA-8).
    per = oracle_mod.kv_bytes_per_token
    assert round(per(80, 64, 128, 2) * 4096 * 16 / 1e9, 3) == 171.799
    assert round(per(80, 8, 128, 2) * 4096 * 16 / 1e9, 3) == 21.475
    # 32 -> 8 KV heads saves 384 KiB/token, 8 -> 1 saves 112 KiB more.
    assert (per(32, 32, 128, 2) - per(32, 8, 128, 2)) == 384 * 1024
    assert (per(32, 8, 128, 2) - per(32, 1, 128, 2)) == 112 * 1024
    # 8B at 128k context: 16 GiB per request.
    assert per(32, 8, 128, 2) * 131_072 == 16 * 1024 ** 3


# ------------------------------------------------------------------ decoders

def test_f16_decoder_matches_torch(oracle_mod):
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.float16).copy()).double().numpy()
    ours = np.array([oracle_mod.f16_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


def test_bf16_decoder_matches_torch(oracle_mod):
    codes = torch.arange(65536, dtype=torch.int32).to(torch.uint16)
    ref = codes.view(torch.bfloat16).double().numpy()
    ours = np.array([oracle_mod.bf16_to_f64(int(c)) for c in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e4m3_decoder_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([oracle_mod.e4m3_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 2                      # 0x7F and 0xFF only
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle_mod.e4m3_to_f64(0x7E) == 448.0
    assert oracle_mod.e4m3_to_f64(0x01) == 2.0 ** -9


def test_e5m2_decoder_matches_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e5m2).double().numpy()
    ours = np.array([oracle_mod.e5m2_to_f64(c) for c in range(256)])
    nan = np.isnan(ref)
    assert nan.sum() == 6                      # S.11111.{01,10,11}
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle_mod.e5m2_to_f64(0x7B) == 57344.0
    assert oracle_mod.e5m2_to_f64(0x7C) == np.inf
    assert oracle_mod.e5m2_to_f64(0x01) == 2.0 ** -16


# ------------------------------------------------- library routine: SDPA

def _sdpa_gqa(inp):
    """torch SDPA (enable_gqa) per sequence, float64, valid tokens only."""
    q, k, v = inp["q"].double(), inp["k"].double(), inp["v"].double()
    if inp.get("k_scale") is not None:
        k = k * inp["k_scale"].double()[:, :, None, None]
        v = v * inp["v_scale"].double()[:, :, None, None]
    B, Hq, D = q.shape
    out = torch.zeros((B, Hq, D), dtype=torch.float64)
    for b in range(B):
        L = int(inp["seq_lens"][b])
        if L == 0:
            continue
        o = F.scaled_dot_product_attention(
            q[b:b + 1, :, None, :], k[b:b + 1, :, :L], v[b:b + 1, :, :L],
            scale=inp["scale"], enable_gqa=True)
        out[b] = o[0, :, 0, :]
    return out.numpy()


SMALL = [
    Workload("t_g4", 2, 8, 2, 64, 37, "f16", lens=("list", 37, 5), seed=7),
    Workload("t_g8", 2, 16, 2, 128, 70, "bf16", lens=("ragged", 1, 70), seed=8),
    Workload("t_mha", 1, 4, 4, 64, 33, "bf16", seed=9),
    Workload("t_mqa", 2, 16, 1, 64, 50, "bf16", lens=("ragged", 1, 50), seed=10),
    Workload("t_fp8", 3, 8, 2, 128, 90, "bf16", kv="e4m3",
             lens=("ragged", 1, 90), seed=11),
    Workload("t_e5m2", 3, 8, 2, 128, 90, "bf16", kv="e5m2",
             lens=("ragged", 1, 90), seed=12),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_oracle_matches_torch_sdpa_enable_gqa(oracle_mod, w):
    inp = make_inputs(w, pad="nan")
    ours = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"], k_scale=inp["k_scale"],
                                 v_scale=inp["v_scale"])
    ref = _sdpa_gqa(inp)
    assert not np.isnan(ours).any()
    np.testing.assert_allclose(ours, ref, rtol=0, atol=1e-12)


@settings(max_examples=60, deadline=None, derandomize=True,
          suppress_health_check=[HealthCheck.function_scoped_fixture])
@given(B=st.integers(1, 3), Hkv=st.sampled_from([1, 2, 3]),
       G=st.sampled_from([1, 2, 3, 5, 8]), D=st.sampled_from([8, 16, 64, 128]),
       Smax=st.integers(1, 48), dtype=st.sampled_from(["f16", "bf16"]),
       kv=st.sampled_from(["same", "e4m3", "e5m2"]), seed=st.integers(0, 999))
def test_oracle_matches_torch_sdpa_on_random_shapes(oracle_mod, B, Hkv, G, D,
                                                    Smax, dtype, kv, seed):
    """Any group size, head dim, cache type and length mix (empty sequences
    included): the oracle equals torch's SDPA with enable_gqa in float64."""
    w = Workload("hyp", B, G * Hkv, Hkv, D, Smax, dtype, kv=kv,
                 lens=("ragged", 0, Smax), seed=seed)
    inp = make_inputs(w, pad="nan")
    ours = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"], k_scale=inp["k_scale"],
                                 v_scale=inp["v_scale"])
    assert not np.isnan(ours).any()
    np.testing.assert_allclose(ours, _sdpa_gqa(inp), rtol=0, atol=1e-12)


def test_g1_is_per_head_mha(oracle_mod):
    w = Workload("mha", 2, 6, 6, 64, 40, "bf16", lens=("list", 40, 17), seed=12)
    inp = make_inputs(w)
    ours = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"])
    for b in range(w.B):
        L = int(inp["seq_lens"][b])
        o = F.scaled_dot_product_attention(
            inp["q"].double()[b:b + 1, :, None], inp["k"].double()[b:b + 1, :, :L],
            inp["v"].double()[b:b + 1, :, :L], scale=inp["scale"])
        np.testing.assert_allclose(ours[b], o[0, :, 0].numpy(), atol=1e-12,
                                   rtol=0)


# --------------------------------------------------------------- structure

def test_gqa_equals_mha_on_expanded_cache(oracle_mod):
    w = Workload("exp", 2, 16, 4, 64, 45, "bf16", lens=("list", 45, 12), seed=13)
    inp = make_inputs(w)
    gqa = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                inp["scale"])
    # explicit expansion: KV head j copied to query heads jG .. jG+G-1
    kx = np.repeat(inp["k"].double().numpy(), w.G, axis=1)
    vx = np.repeat(inp["v"].double().numpy(), w.G, axis=1)
    mha = oracle_mod.gqa_decode(inp["q"].double().numpy(), kx, vx,
                                inp["seq_lens"], inp["scale"])
    assert np.array_equal(gqa, mha)


def test_head_mapping_is_contiguous(oracle_mod):
    w = Workload("map", 1, 12, 3, 64, 20, "bf16", seed=14)
    inp = make_inputs(w)
    base = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"])
    for j in range(w.Hkv):
        k2 = inp["k"].clone()
        v2 = inp["v"].clone()
        k2[:, j] = k2[:, j] * 1.5
        v2[:, j] = -v2[:, j]
        out = oracle_mod.gqa_decode(inp["q"], k2, v2, inp["seq_lens"],
                                    inp["scale"])
        changed = np.abs(out - base).max(axis=2)[0] > 0
        expect = np.zeros(w.Hq, dtype=bool)
        expect[j * w.G:(j + 1) * w.G] = True
        assert np.array_equal(changed, expect), (j, changed)


def test_softmax_weights_sum_to_one(oracle_mod):
    w = Workload("sum", 2, 8, 2, 128, 300, "bf16", lens=("list", 300, 1), seed=15)
    inp = make_inputs(w)
    for b in range(2):
        for h in range(8):
            wt, _ = oracle_mod.gqa_weights(inp["q"], inp["k"], inp["v"],
                                           inp["seq_lens"], inp["scale"], b, h)
            assert len(wt) == int(inp["seq_lens"][b])
            assert abs(wt.sum() - 1.0) < 1e-12
            assert (wt > 0).all()


# ------------------------------------------------------------ special cases

def test_single_token_returns_its_value_row(oracle_mod):
    w = Workload("s1", 3, 8, 2, 64, 9, "bf16", lens=("list", 1, 1, 1), seed=16)
    inp = make_inputs(w)
    out = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                inp["scale"])
    for b in range(3):
        for h in range(8):
            assert np.array_equal(out[b, h],
                                  inp["v"][b, h // 4, 0].double().numpy())


def test_identical_keys_return_mean_of_values(oracle_mod):
    w = Workload("idk", 2, 8, 2, 64, 33, "bf16", lens=("list", 33, 20), seed=17)
    inp = make_inputs(w)
    k = inp["k"].clone()
    k[:, :, :, :] = k[:, :, :1, :]          # every token gets token 0's key
    out = oracle_mod.gqa_decode(inp["q"], k, inp["v"], inp["seq_lens"],
                                inp["scale"])
    for b in range(2):
        L = int(inp["seq_lens"][b])
        mean = inp["v"][b, :, :L].double().mean(dim=1).numpy()   # [Hkv, D]
        for h in range(8):
            np.testing.assert_allclose(out[b, h], mean[h // 4], atol=1e-13,
                                       rtol=0)


def test_zero_query_returns_mean_of_values(oracle_mod):
    w = Workload("q0", 1, 4, 1, 64, 25, "f16", seed=18)
    inp = make_inputs(w)
    out = oracle_mod.gqa_decode(torch.zeros_like(inp["q"]), inp["k"], inp["v"],
                                inp["seq_lens"], inp["scale"])
    mean = inp["v"][0, 0].double().mean(dim=0).numpy()
    for h in range(4):
        np.testing.assert_allclose(out[0, h], mean, atol=1e-13, rtol=0)


def test_dominant_key_returns_its_value_row(oracle_mod):
    w = Workload("dom", 1, 4, 1, 64, 40, "bf16", seed=19)
    inp = make_inputs(w)
    q = inp["q"].double().numpy()
    k = inp["k"].double().numpy()
    t_star = 23
    # key t* aligned with every query head's direction, scores >= 50 above rest
    k[0, 0, t_star] = 100.0 * q[0].sum(axis=0) / np.linalg.norm(q[0].sum(axis=0))
    k[0, 0, t_star] *= 8.0
    out = oracle_mod.gqa_decode(q, k, inp["v"].double().numpy(),
                                inp["seq_lens"], inp["scale"])
    s = inp["scale"] * np.einsum("hd,td->ht", q[0], k[0, 0])
    gap = s[:, t_star] - np.delete(s, t_star, axis=1).max(axis=1)
    assert (gap > 50).all()
    for h in range(4):
        # the other 39 tokens carry weight <= 39 * exp(-50) in total
        np.testing.assert_allclose(out[0, h], inp["v"][0, 0, t_star].double(),
                                   atol=1e-15, rtol=0)


def test_uniform_score_shift_leaves_output_unchanged(oracle_mod):
    w = Workload("shift", 1, 8, 2, 64, 64, "bf16", seed=20)
    inp = make_inputs(w)
    q = inp["q"].double().numpy()
    k = inp["k"].double().numpy()
    v = inp["v"].double().numpy()
    base = oracle_mod.gqa_decode(q, k, v, inp["seq_lens"], inp["scale"])
    u = np.zeros(64)
    u[5] = 1.0
    k2 = k + 300.0 * u                      # scores shift by 300*q[5]*scale
    out = oracle_mod.gqa_decode(q, k2, v, inp["seq_lens"], inp["scale"])
    np.testing.assert_allclose(out, base, atol=1e-11, rtol=0)


def test_token_permutation_leaves_output_unchanged(oracle_mod):
    w = Workload("perm", 1, 8, 2, 64, 50, "bf16", seed=21)
    inp = make_inputs(w)
    perm = torch.randperm(50, generator=torch.Generator().manual_seed(3))
    out = oracle_mod.gqa_decode(inp["q"], inp["k"][:, :, perm],
                                inp["v"][:, :, perm], inp["seq_lens"],
                                inp["scale"])
    base = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"])
    np.testing.assert_allclose(out, base, atol=1e-13, rtol=0)


def test_empty_sequence_gives_zero_output_and_padding_is_ignored(oracle_mod):
    w = Workload("e", 3, 4, 2, 64, 16, "bf16", lens=("list", 0, 16, 3), seed=22)
    inp = make_inputs(w, pad="nan")
    out = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                inp["scale"])
    assert not np.isnan(out).any()
    assert np.array_equal(out[0], np.zeros((4, 64)))


def test_fp8_cache_equals_dequantised_values(oracle_mod):
    w = small_variant(WORKLOADS["ragged_fp8_b64_h32_kv8_l500_30000"], B=3,
                      Smax=77, lens=("ragged", 1, 77), seed=23)
    inp = make_inputs(w, pad="nan")
    fp8 = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                inp["scale"], k_scale=inp["k_scale"],
                                v_scale=inp["v_scale"])
    kd = inp["k"].double() * inp["k_scale"].double()[:, :, None, None]
    vd = inp["v"].double() * inp["v_scale"].double()[:, :, None, None]
    ref = oracle_mod.gqa_decode(inp["q"], kd.numpy(), vd.numpy(),
                                inp["seq_lens"], inp["scale"])
    assert np.array_equal(fp8, ref)
    # K and V scales are distinct per (sequence, KV head): swapping them must
    # change the result.
    swapped = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"],
                                    inp["seq_lens"], inp["scale"],
                                    k_scale=inp["v_scale"],
                                    v_scale=inp["k_scale"])
    assert np.abs(swapped - fp8).max() > 1e-6


def test_sampled_rows_match_full_decode(oracle_mod):
    w = Workload("rows", 3, 8, 2, 64, 40, "bf16", lens=("ragged", 0, 40),
                 seed=24)
    inp = make_inputs(w)
    full = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                                 inp["scale"])
    bh = [(2, 7), (0, 0), (1, 3)]
    rows = oracle_mod.gqa_decode_rows(inp["q"], inp["k"], inp["v"],
                                      inp["seq_lens"], inp["scale"], bh)
    for i, (b, h) in enumerate(bh):
        assert np.array_equal(rows[i], full[b, h])


# ------------------------------------------------- paged cache (gather step)

def test_paged_oracle_on_worked_example_in_reversed_pages(oracle_mod):
    """The worked example's two cached tokens stored in a page pool in
    reverse order (page size 1, so token t of KV head j sits in page 1 - t)
    give the printed outputs."""
    Q, K, V, scale, W, O, tol = _read_golden(GOLDEN)
    # pool [num_pages=2, Hkv=2, page_size=1, D=2]: page p holds token 1 - p
    kp = np.zeros((2, 2, 1, 2))
    vp = np.zeros((2, 2, 1, 2))
    for t in range(2):
        kp[1 - t, :, 0] = K[0, :, t]
        vp[1 - t, :, 0] = V[0, :, t]
    table = np.array([[1, 0]], dtype=np.int32)
    out = oracle_mod.gqa_decode_paged(Q, kp, vp, table, np.array([2]), scale)
    assert np.abs(out[0] - O).max() <= tol


@pytest.mark.parametrize("page_size", [64, 128])
def test_paged_oracle_is_invariant_to_page_placement(oracle_mod, page_size):
    """Any placement of the pages in the pool, and any content of pages no
    sequence uses, gives the contiguous result."""
    w = Workload("pg", 3, 16, 2, 64, 300, "bf16", lens=("list", 300, 1, 129),
                 seed=5, page_size=page_size)
    inp = make_inputs(w, pad="nan")
    a = oracle_mod.gqa_decode_paged(inp["q"], inp["k"], inp["v"],
                                    inp["block_table"], inp["seq_lens"],
                                    inp["scale"])
    b = oracle_mod.gqa_decode(inp["q"], inp["k_contig"], inp["v_contig"],
                              inp["seq_lens"], inp["scale"])
    assert np.array_equal(a, b)
    table = inp["block_table"].numpy()
    used = set(int(x) for x in table.ravel() if x >= 0)
    assert len(used) == int(sum((int(L) + page_size - 1) // page_size
                                for L in inp["seq_lens"]))


# ------------------------------------------ FP8 encoder (cache append step)

@pytest.mark.parametrize("kind,dtype,maxv", [
    (2, torch.float8_e4m3fn, 448.0), (4, torch.float8_e5m2, 57344.0)])
def test_fp8_encoder_matches_torch_in_range(oracle_mod, kind, dtype, maxv):
    """Round-to-nearest-even onto the 8-bit grid, checked against torch's
    cast on every finite code, every midpoint between neighbouring codes
    (the ties), random values and subnormals, all within the finite range."""
    rng = np.random.default_rng(kind)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(dtype)
    vals = codes.float()
    vals = vals[torch.isfinite(vals) & (vals.abs() <= maxv)]
    s = torch.sort(vals).values
    x = torch.cat([vals, (s[1:] + s[:-1]) / 2,
                   torch.tensor(rng.uniform(-maxv, maxv, 4000),
                                dtype=torch.float32),
                   torch.tensor(rng.uniform(-0.01, 0.01, 4000),
                                dtype=torch.float32)])
    ref = x.to(dtype).view(torch.uint8).numpy()
    ours = np.array([oracle_mod.f32_to_fp8(v, kind) for v in x.tolist()],
                    dtype=np.uint8)
    assert np.array_equal(ref, ours)


def test_fp8_encoder_clamps_beyond_the_largest_value(oracle_mod):
    assert oracle_mod.f32_to_fp8(1e6, 2) == 0x7E       # +448
    assert oracle_mod.f32_to_fp8(-500.0, 2) == 0xFE    # -448
    assert oracle_mod.f32_to_fp8(1e9, 4) == 0x7B       # +57344
    assert oracle_mod.f32_to_fp8(-70000.0, 4) == 0xFB


# ------------------------------------------------- cache append (the oracle)

def _append_case(cache_kind, seed, B=3, Hkv=2, Smax=40, D=64, lens=(5, 0, 39),
                 scale_mul=None):
    """Random caches with lens[b] valid tokens, new rows, and scales."""
    g = torch.Generator().manual_seed(seed)
    kn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = (3.0 * torch.randn((B, Hkv, D), generator=g)).to(torch.bfloat16)
    seq = torch.tensor(lens, dtype=torch.int32)
    if cache_kind == "bf16":
        kc = torch.randn((B, Hkv, Smax, D), generator=g).to(torch.bfloat16)
        vc = torch.randn((B, Hkv, Smax, D), generator=g).to(torch.bfloat16)
        return kn, vn, kc, vc, seq, None, None
    dt = torch.float8_e4m3fn if cache_kind == "e4m3" else torch.float8_e5m2
    kc = torch.randn((B, Hkv, Smax, D), generator=g).mul(50).to(dt)
    vc = torch.randn((B, Hkv, Smax, D), generator=g).mul(50).to(dt)
    ks = torch.rand((B, Hkv), generator=g).add(0.5).mul(scale_mul)
    vs = torch.rand((B, Hkv), generator=g).add(0.5).mul(scale_mul)
    return kn, vn, kc, vc, seq, ks.float(), vs.float()


def test_append_16bit_copies_the_row(oracle_mod):
    kn, vn, kc, vc, seq, _, _ = _append_case("bf16", 1)
    k2, v2, _, _, lens, flags = oracle_mod.append_kv(kn, vn, kc, vc, seq)
    assert flags == 0 and list(lens) == [6, 1, 40]
    k2 = torch.from_numpy(k2).view(torch.bfloat16)
    v2 = torch.from_numpy(v2).view(torch.bfloat16)
    for b, L in enumerate(seq.tolist()):
        assert torch.equal(k2[b, :, L], kn[b])
        assert torch.equal(v2[b, :, L], vn[b])
        mask = torch.ones(k2.shape[2], dtype=torch.bool)
        mask[L] = False
        assert torch.equal(k2[b, :, mask], kc[b, :, mask])


@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
@pytest.mark.parametrize("scale_mul", [10.0, 1e-5, 0.0])
def test_append_fp8_quantise_and_rescale(oracle_mod, kind, scale_mul):
    """Against float32 arithmetic and torch's casts: the scale (kept,
    doubled until the new row fits, or set from the row when unset), the
    re-encoded earlier codes and the new row's codes."""
    dt = torch.float8_e4m3fn if kind == "e4m3" else torch.float8_e5m2
    M = np.float32(448.0 if kind == "e4m3" else 57344.0)
    kn, vn, kc, vc, seq, ks, vs = _append_case(kind, 2, scale_mul=scale_mul)
    k2, v2, ks2, vs2, lens, flags = oracle_mod.append_kv(
        kn, vn, kc, vc, seq, k_scale=ks, v_scale=vs)
    assert flags == 0 and list(lens) == [6, 1, 40]
    for new, old, sc, got, sc2 in ((kn, kc, ks, k2, ks2), (vn, vc, vs, v2, vs2)):
        got = torch.from_numpy(got).view(dt)
        for b, L in enumerate(seq.tolist()):
            for j in range(new.shape[1]):
                x = new[b, j].float().numpy()
                a = np.float32(np.abs(x).max())
                s = np.float32(sc[b, j])
                if not s > 0:
                    s2 = np.float32(a / M) if a > 0 else np.float32(1.0)
                    prev = old[b, j, :L]
                else:
                    s2 = s
                    while np.float32(a / s2) > M:
                        s2 = np.float32(s2 * np.float32(2.0))
                    ratio = np.float32(s / s2)
                    prev = (old[b, j, :L].float() *
                            torch.tensor(ratio)).to(dt) if s2 != s \
                        else old[b, j, :L]
                assert np.float32(sc2[b, j]) == s2
                assert torch.equal(got[b, j, :L].view(torch.uint8),
                                   prev.view(torch.uint8))
                row = (torch.from_numpy(x) / torch.tensor(s2)).to(dt)
                assert torch.equal(got[b, j, L].view(torch.uint8),
                                   row.view(torch.uint8))
                if scale_mul == 1e-5:
                    assert s2 > s          # the tiny scales had to grow


def test_append_full_cache_is_flagged_and_left_alone(oracle_mod):
    kn, vn, kc, vc, seq, _, _ = _append_case("bf16", 3, lens=(40, 2, -3))
    k2, _, _, _, lens, flags = oracle_mod.append_kv(kn, vn, kc, vc, seq)
    assert flags == 4
    assert list(lens) == [40, 3, 1]      # full, appended, negative as 0
    assert torch.equal(torch.from_numpy(k2).view(torch.bfloat16)[0], kc[0])


# ---------------------------------- multi-token causal step (chunk oracle)

def test_chunk_with_one_token_is_the_decode_step(oracle_mod):
    w = Workload("c1", 3, 16, 4, 64, 90, "bf16", lens=("list", 90, 1, 33),
                 seed=21)
    inp = make_inputs(w, pad="nan")
    a = oracle_mod.gqa_decode(inp["q"], inp["k"], inp["v"], inp["seq_lens"],
                              inp["scale"])
    c = oracle_mod.gqa_decode_chunk(inp["q"][:, :, None, :], inp["k"],
                                    inp["v"], inp["seq_lens"], inp["scale"])
    assert np.array_equal(a, c[:, :, 0, :])


def test_chunk_token_i_is_a_decode_over_its_prefix(oracle_mod):
    """New token i of a T-token chunk sees exactly the first L - T + i + 1
    cached tokens: the same as a one-token step with that length."""
    w = Workload("c4", 2, 16, 2, 128, 200, "f16", lens=("list", 200, 77),
                 seed=22, T=5)
    inp = make_inputs(w, pad="nan")
    c = oracle_mod.gqa_decode_chunk(inp["q"], inp["k"], inp["v"],
                                    inp["seq_lens"], inp["scale"])
    for i in range(5):
        lens_i = inp["seq_lens"] - 5 + i + 1
        d = oracle_mod.gqa_decode(inp["q"][:, :, i, :].contiguous(), inp["k"],
                                  inp["v"], lens_i, inp["scale"])
        assert np.array_equal(c[:, :, i, :], d)


def test_chunk_longer_than_the_cache_gives_zero_rows(oracle_mod):
    w = Workload("c_short", 1, 4, 2, 64, 8, "bf16", lens=("list", 3), seed=23,
                 T=5)
    inp = make_inputs(w, pad="nan")
    c = oracle_mod.gqa_decode_chunk(inp["q"], inp["k"], inp["v"],
                                    inp["seq_lens"], inp["scale"])
    assert np.count_nonzero(c[0, :, :2]) == 0     # tokens 0, 1 see nothing
    assert np.isfinite(c).all() and np.count_nonzero(c[0, :, 2:]) > 0


def test_full_causal_prefill_matches_torch_sdpa(oracle_mod):
    """T = L (the whole cache is new): the causal GQA attention of the
    pages' SDPA call, scaled_dot_product_attention(q, k, v, is_causal=True,
    enable_gqa=True), in float64."""
    for Hq, Hkv in ((8, 2), (4, 4), (8, 1)):
        w = Workload("pf", 2, Hq, Hkv, 64, 40, "bf16", seed=24 + Hkv, T=40)
        inp = make_inputs(w, pad="nan")
        c = oracle_mod.gqa_decode_chunk(inp["q"], inp["k"], inp["v"],
                                        inp["seq_lens"], inp["scale"])
        ref = F.scaled_dot_product_attention(
            inp["q"].double(), inp["k"].double(), inp["v"].double(),
            scale=inp["scale"], is_causal=True, enable_gqa=True)
        assert np.abs(c - ref.numpy()).max() <= 1e-12
