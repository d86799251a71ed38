"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, on
seeded inputs at sizes the oracle finishes in seconds.  Each case spans several
64-token tiles and ends in a ragged tail; cache padding is NaN so any read past
a sequence's valid prefix poisons the output."""
import math
import os

import numpy as np
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import (WORKLOADS, Workload,
                                                       make_inputs,
                                                       small_variant)

from gpu_util import (assert_close, assert_contract, oracle_full, run_cuda,
                      to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)
    yield
    gq.gqa_set_num_ctas(0)


CASES = [
    # name, B, Hq, Hkv, D, Smax, dtype, kv, lens
    ("f16_g4_d64_tiny_shape", 1, 8, 2, 64, 128, "f16", "same", ("uniform",)),
    ("bf16_g4_d128_ragged", 3, 32, 8, 128, 300, "bf16", "same",
     ("list", 300, 1, 129)),
    ("bf16_g8_d128_ragged", 2, 64, 8, 128, 515, "bf16", "same",
     ("list", 515, 200)),
    ("f16_g8_d128", 2, 16, 2, 128, 257, "f16", "same", ("list", 257, 64)),
    ("bf16_mha_g1", 2, 8, 8, 128, 190, "bf16", "same", ("list", 190, 77)),
    ("bf16_mqa_g64", 2, 64, 1, 128, 200, "bf16", "same", ("list", 200, 33)),
    ("bf16_g32_d64", 2, 32, 1, 64, 150, "bf16", "same", ("list", 150, 65)),
    ("bf16_g48_two_kv", 1, 96, 2, 128, 100, "bf16", "same", ("uniform",)),
    ("bf16_g80_two_chunks", 1, 80, 1, 64, 130, "bf16", "same", ("uniform",)),
    ("f16_g128_two_chunks", 2, 128, 1, 64, 70, "f16", "same", ("list", 70, 3)),
    ("bf16_g2_d64", 3, 4, 2, 64, 64, "bf16", "same", ("list", 64, 63, 65 - 1)),
    ("bf16_empty_sequences", 4, 16, 4, 128, 100, "bf16", "same",
     ("list", 0, 5, 0, 100)),
    ("bf16_smax_not_tile_multiple", 2, 16, 2, 128, 100, "bf16", "same",
     ("uniform",)),
    ("fp8_g4_d128_ragged", 4, 32, 8, 128, 400, "bf16", "e4m3",
     ("list", 400, 1, 70, 333)),
    ("fp8_g8_d128", 2, 64, 8, 128, 260, "bf16", "e4m3", ("list", 260, 129)),
    ("fp8_g4_d64", 3, 8, 2, 64, 200, "bf16", "e4m3", ("list", 200, 64, 9)),
    ("fp8_f16_q_g4", 2, 16, 4, 128, 150, "f16", "e4m3", ("list", 150, 80)),
    ("fp8_mqa_g64", 1, 64, 1, 128, 300, "bf16", "e4m3", ("uniform",)),
    ("fp8_mha_g1", 2, 4, 4, 64, 99, "bf16", "e4m3", ("list", 99, 17)),
    ("e5m2_g4_d128_ragged", 4, 32, 8, 128, 400, "bf16", "e5m2",
     ("list", 400, 1, 70, 333)),
    ("e5m2_g8_d64_f16", 2, 16, 2, 64, 300, "f16", "e5m2", ("list", 300, 129)),
    ("e5m2_mqa_g64", 1, 64, 1, 128, 200, "bf16", "e5m2", ("uniform",)),
    # 8-bit caches with 9..16 rows per unit: the wide one-head-block path
    # (groups of <= 8 rows take the narrow-row path)
    ("fp8_g16_d128_wide", 2, 32, 2, 128, 300, "bf16", "e4m3",
     ("list", 300, 77)),
    ("e5m2_g12_d64_wide", 2, 24, 2, 64, 200, "f16", "e5m2", ("list", 130, 200)),
    ("e5m2_g16_d128_wide", 2, 32, 2, 128, 260, "bf16", "e5m2",
     ("list", 260, 100)),
    # 8-bit caches with 17..32 rows per unit: two head blocks per warp group
    ("fp8_g32_d128_two_blocks", 2, 64, 2, 128, 300, "bf16", "e4m3",
     ("list", 300, 77)),
    ("e5m2_g24_d64_two_blocks", 2, 48, 2, 64, 200, "f16", "e5m2",
     ("list", 200, 129)),
    ("fp8_g2_d128_narrow", 3, 8, 4, 128, 333, "bf16", "e4m3",
     ("list", 333, 1, 64)),
    # more sequences than threads per block: the general scheduler prologue
    ("bf16_many_sequences", 300, 8, 2, 64, 70, "bf16", "same",
     ("ragged", 0, 70)),
    ("fp8_many_sequences", 290, 8, 2, 128, 80, "bf16", "e4m3",
     ("ragged", 0, 80)),
    ("bf16_more_sequences_than_threads", 400, 8, 2, 64, 60, "bf16", "same",
     ("ragged", 0, 60)),
]


def _workload(c, seed):
    name, B, Hq, Hkv, D, Smax, dt, kv, lens = c
    return Workload(name, B, Hq, Hkv, D, Smax, dt, kv=kv, lens=lens, seed=seed)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_small(oracle_mod, case):
    w = _workload(case, 2000 + CASES.index(case))
    inp = make_inputs(w, pad="nan")
    out = run_cuda(inp)
    ref = oracle_full(oracle_mod, inp)
    assert_close(out, ref, w.name)
    for b in range(w.B):
        if int(inp["seq_lens"][b]) == 0:
            assert torch.count_nonzero(out[b]).item() == 0


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_parity_config_shaped_small(oracle_mod, name):
    """Every named workload's head layout and dtypes at a reduced size, with
    the contract tolerance exactly."""
    w = WORKLOADS[name]
    small = small_variant(w, B=min(w.B, 3), Smax=min(w.Smax, 700),
                          lens=("ragged", 1, min(w.Smax, 700)) if
                          w.lens[0] == "ragged" else ("uniform",),
                          seed=w.seed + 50)
    inp = make_inputs(small, pad="nan")
    out = run_cuda(inp)
    ref = oracle_full(oracle_mod, inp)
    assert_contract(out, ref, small.name)


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 37, 148, 1000])
def test_split_invariance(oracle_mod, num_ctas):
    """Any split of the sequence axis between blocks gives the same result up
    to fp32 rounding: one block (no split), a few, many more than units."""
    w = Workload("split", 2, 32, 4, 128, 1000, "bf16",
                 lens=("list", 1000, 777), seed=31)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    try:
        gq.gqa_set_num_ctas(num_ctas)
        out = run_cuda(inp)
    finally:
        gq.gqa_set_num_ctas(0)
    assert_contract(out, ref, f"ctas={num_ctas}")


def test_split_invariance_fp8(oracle_mod):
    w = Workload("split8", 3, 32, 8, 128, 900, "bf16", kv="e4m3",
                 lens=("list", 900, 1, 450), seed=32)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    for n in (1, 3, 64, 500):
        try:
            gq.gqa_set_num_ctas(n)
            out = run_cuda(inp)
        finally:
            gq.gqa_set_num_ctas(0)
        assert_contract(out, ref, f"fp8 ctas={n}")


@pytest.mark.parametrize("kv", ["e4m3", "e5m2"])
def test_fp8_per_tensor_scales(oracle_mod, kv):
    """One scale for each whole tensor (K, V): every (sequence, KV head)
    entry set to the tensor's largest.  Both sides dequantise code x scale,
    so parity holds whatever the scales; the largest keeps values O(1)."""
    w = Workload("per_tensor_" + kv, 3, 32, 8, 128, 400, "bf16", kv=kv,
                 lens=("list", 400, 3, 200), seed=33)
    inp = make_inputs(w, pad="nan")
    inp["k_scale"] = torch.full_like(inp["k_scale"],
                                     float(inp["k_scale"].max()))
    inp["v_scale"] = torch.full_like(inp["v_scale"],
                                     float(inp["v_scale"].max()))
    out = run_cuda(inp)
    ref = oracle_full(oracle_mod, inp)
    assert_close(out, ref, w.name)


def test_deterministic_bitwise():
    w = Workload("det", 4, 64, 8, 128, 800, "bf16", lens=("ragged", 1, 800),
                 seed=33)
    dev = to_device(make_inputs(w, pad="nan"))
    a = gq.decode_inputs(dev).clone()
    b = gq.decode_inputs(dev).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_worked_example_2_zero_padded(oracle_mod):
    """The pages' worked example (4 heads, head_dim 2, 2 KV heads, 2 tokens)
    with head_dim zero-padded to 64 and fp16 I/O: every input is exact in fp16,
    so the first two columns must match the printed values and the rest must
    be exactly zero."""
    from test_oracle_pins import GOLDEN, _read_golden
    Q, K, V, scale, W, O, tol = _read_golden(GOLDEN)
    D = 64
    q = torch.zeros((1, 4, D), dtype=torch.float16)
    k = torch.zeros((1, 2, 2, D), dtype=torch.float16)
    v = torch.zeros((1, 2, 2, D), dtype=torch.float16)
    q[..., :2] = torch.from_numpy(Q).half()
    k[..., :2] = torch.from_numpy(K).half()
    v[..., :2] = torch.from_numpy(V).half()
    inp = {"q": q, "k": k, "v": v, "k_scale": None, "v_scale": None,
           "seq_lens": torch.tensor([2], dtype=torch.int32), "scale": scale}
    out = run_cuda(inp).double().cpu().numpy()
    # printed to 4 decimals (+-5e-5); fp16 probabilities and fp16 output
    # rounding at |out| < 4 add at most ~3e-3
    assert np.abs(out[0, :, :2] - O).max() <= tol + 4e-3
    assert np.count_nonzero(out[0, :, 2:]) == 0
    ref = oracle_full(oracle_mod, inp)
    assert np.abs(out - ref).max() <= 4e-3


def test_single_token_returns_value_row():
    w = Workload("s1", 3, 32, 8, 128, 64, "bf16", lens=("list", 1, 1, 1),
                 seed=34)
    inp = make_inputs(w, pad="nan")
    out = run_cuda(inp).cpu()
    for b in range(3):
        for h in range(32):
            assert torch.equal(out[b, h], inp["v"][b, h // 4, 0])


def test_identical_keys_return_mean_of_values(oracle_mod):
    w = Workload("idk", 2, 16, 2, 128, 300, "bf16", lens=("list", 300, 97),
                 seed=35)
    inp = make_inputs(w, pad="nan")
    k = inp["k"].clone()
    k[:, :, :, :] = k[:, :, :1, :]
    inp["k"] = k
    out = run_cuda(inp).double().cpu().numpy()
    for b in range(2):
        L = int(inp["seq_lens"][b])
        mean = inp["v"][b, :, :L].double().mean(dim=1).numpy()
        for h in range(16):
            assert np.abs(out[b, h] - mean[h // 8]).max() <= 2e-3


def test_dominant_key_returns_its_value_row():
    w = Workload("dom", 1, 8, 1, 128, 500, "f16", seed=36)
    inp = make_inputs(w, pad="nan")
    q = inp["q"].double()
    t_star = 311
    direction = q[0].sum(dim=0)
    k = inp["k"].clone()
    k[0, 0, t_star] = (direction / direction.norm() * 300).half()
    inp["k"] = k
    s = inp["scale"] * torch.einsum("hd,td->ht", q[0], k[0, 0].double())
    gap = s[:, t_star] - torch.cat([s[:, :t_star], s[:, t_star + 1:]], 1).amax(1)
    assert (gap > 50).all()
    out = run_cuda(inp).double().cpu()
    for h in range(8):
        assert torch.allclose(out[0, h], inp["v"][0, 0, t_star].double(),
                              atol=2.0 ** -11 * 4, rtol=0)


def test_score_shift_invariance(oracle_mod):
    """Adding the same vector u to every key shifts each head's scores by a
    constant (q.u*scale); the online softmax must not care, even when the
    shift is large."""
    w = Workload("shift", 2, 16, 2, 64, 400, "f16", lens=("list", 400, 150),
                 seed=37)
    inp = make_inputs(w, pad="zero")
    u = torch.zeros(64, dtype=torch.float64)
    u[3] = 24.0
    k2 = (inp["k"].double() + u).half()
    inp2 = dict(inp, k=k2)
    ref = oracle_full(oracle_mod, inp2)
    out = run_cuda(inp2)
    assert_close(out, ref, "shifted")


def test_gqa_equals_mha_on_expanded_cache(oracle_mod):
    """GQA over Hkv heads equals MHA (G = 1) over the cache expanded to Hq heads
    (KV head j copied to query heads jG .. jG+G-1): on the GPU and against the
    oracle."""
    for Hkv in (8, 1):
        w = Workload("exp", 2, 64, Hkv, 128, 300, "bf16",
                     lens=("list", 300, 129), seed=38 + Hkv)
        inp = make_inputs(w, pad="nan")
        gqa = run_cuda(inp)
        G = w.Hq // Hkv
        inp_x = dict(inp, k=inp["k"].repeat_interleave(G, dim=1).contiguous(),
                     v=inp["v"].repeat_interleave(G, dim=1).contiguous())
        mha = run_cuda(inp_x)
        ref = oracle_full(oracle_mod, inp)
        ref_x = oracle_full(oracle_mod, inp_x)
        assert np.array_equal(ref, ref_x)
        assert_contract(gqa, ref, "gqa")
        assert_contract(mha, ref_x, "mha on expanded")
        d = (gqa.double() - mha.double()).abs().max().item()
        assert d <= 2 * 2.0 ** -8 * 4


def test_head_mapping_on_gpu():
    """Perturbing KV head j changes exactly query heads jG .. jG+G-1."""
    w = Workload("map", 1, 32, 4, 128, 130, "bf16", seed=40)
    inp = make_inputs(w, pad="nan")
    base = run_cuda(inp).cpu()
    for j in range(4):
        v2 = inp["v"].clone()
        v2[:, j, :130] = -v2[:, j, :130] - 1
        out = run_cuda(dict(inp, v=v2)).cpu()
        changed = (out != base).flatten(2).any(dim=2)[0]
        expect = torch.zeros(32, dtype=torch.bool)
        expect[j * 8:(j + 1) * 8] = True
        assert torch.equal(changed, expect)


def test_seq_lens_beyond_smax_are_clamped(oracle_mod):
    w = Workload("clamp", 2, 16, 2, 128, 90, "bf16", seed=41)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)          # uses 90 for both
    inp2 = dict(inp, seq_lens=torch.tensor([1000, -5], dtype=torch.int32))
    out = run_cuda(inp2)
    assert_close(out[0:1], ref[0:1], "clamped high")
    assert torch.count_nonzero(out[1]).item() == 0


def test_output_written_in_place_and_stream_respected():
    w = Workload("stream", 2, 32, 8, 128, 256, "bf16", seed=42)
    dev = to_device(make_inputs(w, pad="nan"))
    s = torch.cuda.Stream()
    out = torch.full_like(dev["q"], float("nan"))
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gq.decode_inputs(dev, out=out, stream=s)
    s.synchronize()
    assert torch.isfinite(out).all()
    assert gq.gqa_device_errors(s) == 0


def test_scratch_reuse_across_unit_counts(oracle_mod):
    """Calls on one stream whose unit counts go up and down: the split-combine
    counters of a call with many units must not pick up the partial results a
    call with few units left behind in the library's scratch."""
    shapes = [
        # B, Hq, Hkv, D, Smax, lens  (units = B * Hkv)
        (2, 64, 1, 128, 900, ("list", 900, 700)),       # 2 units, many splits
        (3, 64, 64, 128, 700, ("uniform",)),            # 192 units
        (1, 32, 2, 128, 1000, ("uniform",)),            # 2 units
        (4, 16, 16, 64, 500, ("list", 500, 3, 250, 499)),  # 64 units
        (3, 64, 64, 128, 700, ("uniform",)),
    ]
    for i, (B, Hq, Hkv, D, Smax, lens) in enumerate(shapes):
        w = Workload(f"reuse{i}", B, Hq, Hkv, D, Smax, "bf16", lens=lens,
                     seed=60 + i)
        inp = make_inputs(w, pad="nan")
        out = run_cuda(inp)
        assert_contract(out, oracle_full(oracle_mod, inp), w.name)


PAGED = [
    # name, B, Hq, Hkv, D, Smax, dtype, page_size, lens
    ("paged64_bf16_g8", 3, 64, 8, 128, 700, "bf16", 64, ("list", 700, 1, 333)),
    ("paged128_f16_g4", 4, 16, 4, 64, 500, "f16", 128,
     ("list", 500, 0, 129, 255)),
    ("paged256_bf16_mqa", 2, 64, 1, 128, 1024, "bf16", 256,
     ("list", 1024, 257)),
    ("paged64_bf16_mha", 2, 8, 8, 128, 200, "bf16", 64, ("list", 200, 64)),
]


@pytest.mark.parametrize("case", PAGED, ids=[c[0] for c in PAGED])
def test_parity_paged(oracle_mod, case):
    name, B, Hq, Hkv, D, Smax, dt, ps, lens = case
    w = Workload(name, B, Hq, Hkv, D, Smax, dt, lens=lens,
                 seed=3000 + PAGED.index(case), page_size=ps)
    inp = make_inputs(w, pad="nan")
    out = run_cuda(inp)
    ref = oracle_mod.gqa_decode_paged(inp["q"], inp["k"], inp["v"],
                                      inp["block_table"], inp["seq_lens"],
                                      inp["scale"])
    assert_close(out, ref, name)
    # the same cache laid out contiguously gives the same bits
    flat = {k: v for k, v in inp.items() if k != "block_table"}
    flat["k"], flat["v"] = inp["k_contig"], inp["v_contig"]
    assert torch.equal(run_cuda(flat).view(torch.int16),
                       out.view(torch.int16))


def test_paged_bad_block_table_entry_is_flagged():
    w = Workload("pgbad", 2, 16, 2, 64, 256, "bf16", lens=("list", 256, 200),
                 seed=3100, page_size=64)
    inp = make_inputs(w, pad="nan")
    inp["block_table"] = inp["block_table"].clone()
    inp["block_table"][1, 2] = 10 ** 6     # read: tokens 128..191 of seq 1
    dev = to_device(inp)
    gq.decode_inputs(dev)
    assert gq.gqa_device_errors() & 2
    assert gq.gqa_device_errors() == 0     # the query cleared it


CHUNKS = [
    # name, B, Hq, Hkv, D, Smax, dtype, T, lens
    ("chunk4_bf16_g8", 3, 64, 8, 128, 700, "bf16", 4, ("list", 700, 4, 333)),
    ("chunk16_f16_g4", 2, 16, 4, 64, 300, "f16", 16, ("list", 300, 70)),
    ("chunk8_bf16_mqa", 2, 16, 1, 128, 200, "bf16", 8, ("list", 200, 130)),
    ("chunk64_bf16_g2", 1, 4, 2, 64, 150, "bf16", 64, ("uniform",)),
    ("chunk3_bf16_short", 3, 8, 2, 128, 64, "bf16", 3, ("list", 2, 0, 64)),
    ("chunk1_is_decode", 2, 32, 8, 128, 257, "bf16", 1, ("list", 257, 9)),
]


@pytest.mark.parametrize("case", CHUNKS, ids=[c[0] for c in CHUNKS])
def test_parity_chunk(oracle_mod, case):
    name, B, Hq, Hkv, D, Smax, dt, T, lens = case
    w = Workload(name, B, Hq, Hkv, D, Smax, dt, lens=lens,
                 seed=4000 + CHUNKS.index(case), T=T)
    inp = make_inputs(w, pad="nan")
    if T == 1:
        inp["q"] = inp["q"][:, :, None, :].contiguous()
    dev = to_device(inp)
    out = gq.gqa_decode_chunk(dev["q"], dev["k"], dev["v"], dev["seq_lens"],
                              dev["scale"])
    assert gq.gqa_last_launch_count() == 1
    assert gq.gqa_device_errors() == 0
    ref = oracle_mod.gqa_decode_chunk(inp["q"], inp["k"], inp["v"],
                                      inp["seq_lens"], inp["scale"])
    assert_close(out, ref, name)
    if T == 1:   # the same bits as the decode step
        d = gq.gqa_decode(dev["q"][:, :, 0].contiguous(), dev["k"], dev["v"],
                          dev["seq_lens"], dev["scale"])
        assert torch.equal(d.view(torch.int16), out[:, :, 0].view(torch.int16))
