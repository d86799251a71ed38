"""GPU parity of the tensor-core (tcgen05) decode kernel with the fp64 oracle.

The kernel serves units of 33 to 64 query rows per KV head (multi-query
attention, wide groups, multi-token causal chunks of wide groups) with a
16-bit cache and head_dim 128 by default; gqa_set_kernel_path(2) also sends
units of up to 32 rows to it (its 32-column variant), and
gqa_set_kernel_path(1) sends everything to the warp-level mma kernel.
Each case runs under all three settings against the same oracle output, on
NaN-padded caches, with sequences that end inside a tile, empty sequences,
units split between blocks and row chunks of a KV head (more than 64 rows)."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import assert_close, assert_contract, oracle_full, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _paths():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)
    gq.gqa_set_kernel_path(0)
    yield
    gq.gqa_set_kernel_path(0)
    gq.gqa_set_num_ctas(0)


CASES = [
    # name, B, Hq, Hkv, Smax, dtype, lens, T   (D = 128)
    ("mqa_g64", 3, 64, 1, 700, "bf16", ("list", 700, 129, 1), 1),
    ("g32_f16", 2, 64, 2, 500, "f16", ("list", 500, 300), 1),
    ("g48", 2, 96, 2, 300, "bf16", ("list", 300, 65), 1),
    ("g80_two_row_chunks", 1, 80, 1, 260, "bf16", ("uniform",), 1),
    ("g128_f16_two_row_chunks", 2, 128, 1, 190, "f16", ("list", 190, 3), 1),
    ("g8_chunk4", 3, 64, 8, 600, "bf16", ("list", 600, 4, 333), 4),
    ("g4_chunk8_f16", 2, 16, 4, 300, "f16", ("list", 300, 70), 8),
    ("mqa_chunk3", 2, 16, 1, 200, "bf16", ("list", 200, 2), 3),
    ("g16_chunk5_row_chunks", 2, 32, 2, 200, "bf16", ("list", 200, 130), 5),
    ("short_and_empty", 4, 64, 1, 128, "bf16", ("list", 0, 1, 64, 65), 1),
    ("whole_tiles", 2, 64, 2, 256, "bf16", ("uniform",), 1),
    ("smax_not_tile_multiple", 2, 64, 1, 100, "bf16", ("uniform",), 1),
    ("many_sequences", 300, 32, 1, 90, "bf16", ("ragged", 0, 90), 1),
    # units of at most 32 rows: the tensor-core kernel only under path 2
    ("g8_small", 2, 64, 8, 515, "bf16", ("list", 515, 200), 1),
    ("g4_f16_small", 3, 32, 8, 300, "f16", ("list", 300, 1, 129), 1),
    ("mha_g1", 2, 8, 8, 190, "bf16", ("list", 190, 77), 1),
]


def _run(inp, T):
    if T == 1:
        return run_cuda(inp)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in inp.items()}
    out = gq.gqa_decode_chunk(dev["q"], dev["k"], dev["v"], dev["seq_lens"],
                              dev["scale"])
    assert gq.gqa_device_errors() == 0
    return out


@pytest.mark.parametrize("path", [0, 1, 2])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_parity_every_kernel_path(oracle_mod, case, path):
    name, B, Hq, Hkv, Smax, dt, lens, T = case
    w = Workload(name, B, Hq, Hkv, 128, Smax, dt, lens=lens,
                 seed=5000 + CASES.index(case), T=T)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    gq.gqa_set_kernel_path(path)
    out = _run(inp, T)
    assert_close(out, ref, f"{name} path {path}")
    for b in range(B):
        if int(inp["seq_lens"][b]) == 0:
            assert torch.count_nonzero(out[b]).item() == 0


@pytest.mark.parametrize("num_ctas", [1, 2, 7, 37, 148, 1000])
def test_split_invariance(oracle_mod, num_ctas):
    """Any split of the 128-token tiles between blocks: one block, a few,
    more blocks than tiles (units cut anywhere, the split combine)."""
    w = Workload("umma_split", 2, 64, 1, 128, 1500, "bf16",
                 lens=("list", 1500, 777), seed=5100)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    gq.gqa_set_num_ctas(num_ctas)
    out = run_cuda(inp)
    assert_contract(out, ref, f"ctas={num_ctas}")


def test_chunk_split_invariance(oracle_mod):
    w = Workload("umma_chunk_split", 2, 64, 8, 128, 900, "bf16",
                 lens=("list", 900, 455), seed=5101, T=4)
    inp = make_inputs(w, pad="nan")
    ref = oracle_full(oracle_mod, inp)
    for n in (1, 5, 64, 300):
        gq.gqa_set_num_ctas(n)
        assert_contract(_run(inp, 4), ref, f"chunk ctas={n}")


def test_lazy_rescale_large_score_growth(oracle_mod):
    """Scores that keep growing along the sequence (every tile's maximum far
    above the previous one) force a rescale of O and L on every tile; and a
    single huge score late in the sequence."""
    w = Workload("umma_grow", 2, 64, 1, 128, 1024, "f16", seed=5102)
    inp = make_inputs(w, pad="zero")
    k = inp["k"].double()
    ramp = torch.linspace(0.0, 600.0, 1024, dtype=torch.float64)
    u = inp["q"][0].double().mean(dim=0)
    u = u / u.norm()
    k2 = k + ramp[None, None, :, None] * u[None, None, None, :]
    k2[1, 0, 900] = u * 400.0
    inp["k"] = k2.half()
    ref = oracle_full(oracle_mod, inp)
    for path in (1, 2):
        gq.gqa_set_kernel_path(path)
        assert_close(run_cuda(inp), ref, f"growing scores path {path}")


def test_deterministic_bitwise():
    w = Workload("umma_det", 4, 64, 1, 128, 1100, "bf16",
                 lens=("ragged", 1, 1100), seed=5103)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in make_inputs(w, pad="nan").items()}
    a = gq.decode_inputs(dev).clone()
    b = gq.decode_inputs(dev).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_tensor_core_kernel_launched():
    """The automatic choice sends a 64-row unit to the tensor-core kernel
    (one launch) and it leaves no fault flag."""
    w = Workload("umma_launch", 2, 64, 1, 128, 300, "bf16", seed=5104)
    dev = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
           for k, v in make_inputs(w, pad="nan").items()}
    gq.decode_inputs(dev)
    assert gq.gqa_last_launch_count() == 1
    assert gq.gqa_device_errors() == 0


PAGED = [
    # name, B, Hq, Hkv, Smax, dtype, page_size, lens
    # 64-token pages: the two halves of each 128-token tile come from
    # different pages (shuffled in the pool)
    ("mqa_pages64", 3, 64, 1, 640, "bf16", 64, ("list", 640, 129, 1)),
    ("mqa_pages128_f16", 2, 64, 1, 512, "f16", 128, ("list", 512, 300)),
    ("g48_pages64_uniform", 4, 96, 2, 384, "bf16", 64, ("uniform",)),
]


@pytest.mark.parametrize("path", [0, 2])
@pytest.mark.parametrize("case", PAGED, ids=[c[0] for c in PAGED])
def test_paged_tensor_core_kernel(oracle_mod, case, path):
    """Paged caches on the tensor-core kernel (page of each 64-token box
    looked up in the block table): the oracle's output, and the same bits as
    the contiguous cache."""
    name, B, Hq, Hkv, Smax, dt, ps, lens = case
    w = Workload(name, B, Hq, Hkv, 128, Smax, dt, lens=lens,
                 seed=5200 + PAGED.index(case), page_size=ps)
    inp = make_inputs(w, pad="nan")
    ref = oracle_mod.gqa_decode_paged(inp["q"], inp["k"], inp["v"],
                                      inp["block_table"], inp["seq_lens"],
                                      inp["scale"])
    gq.gqa_set_kernel_path(path)
    out = run_cuda(inp)
    assert_close(out, ref, f"{name} path {path}")
    flat = {k: v for k, v in inp.items() if k != "block_table"}
    flat["k"], flat["v"] = inp["k_contig"], inp["v_contig"]
    assert torch.equal(run_cuda(flat).view(torch.int16),
                       out.view(torch.int16))
