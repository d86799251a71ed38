"""gqa_decode_static: the decode step for callers that cannot let the library
allocate device memory (engines that own the whole memory pool, loops where an
allocation could stall).  Its scratch is one fixed array in the library's
static device memory, shared by every call.

Called through the C ABI and compared with gqa_decode on the same inputs, two
calls in a row (the second one sees what the first left in the shared array),
plus a refused oversized request.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300.workloads import Workload, make_inputs

from gpu_util import MAX_ABS, MEAN_ABS, assert_contract, oracle_full, to_device

pytestmark = pytest.mark.gpu


def _call_static(d, out, stream):
    q, k = d["q"], d["k"]
    B, Hq, D = q.shape
    _, Hkv, Smax, _ = k.shape
    dt = gq.GQA_BF16 if q.dtype == torch.bfloat16 else gq.GQA_F16
    return gq.lib().gqa_decode_static(
        q.data_ptr(), k.data_ptr(), d["v"].data_ptr(),
        d["seq_lens"].data_ptr(), float(d["scale"]), out.data_ptr(), B, Hq,
        Hkv, Smax, D, dt, stream.cuda_stream)


def _check_pair(got, ref):
    e = (got.double() - ref.double()).abs()
    assert torch.isfinite(got).all()
    assert e.max().item() <= MAX_ABS and e.mean().item() <= MEAN_ABS


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    gq.gqa_set_num_ctas(0)


def test_static_scratch_matches_gqa_decode_twice(oracle_mod):
    stream = torch.cuda.current_stream()
    # first a split-heavy shape (few units, many blocks per unit), then one
    # with many units and ragged lengths: the second call finds the first
    # call's partials and counters region in the shared array
    shapes = [
        Workload("static_a", 2, 64, 8, 128, 1500, "bf16",
                 lens=("list", 1500, 777), seed=71),
        Workload("static_b", 5, 32, 8, 128, 900, "bf16",
                 lens=("list", 900, 1, 450, 0, 899), seed=72),
    ]
    for w in shapes:
        inp = make_inputs(w, pad="nan")
        d = to_device(inp)
        ref = gq.gqa_decode(d["q"], d["k"], d["v"], d["seq_lens"], d["scale"])
        out = torch.full_like(d["q"], float("nan"))
        assert _call_static(d, out, stream) == gq.GQA_OK
        torch.cuda.synchronize()
        _check_pair(out, ref)
        assert_contract(out, oracle_full(oracle_mod, inp), w.name)


def test_static_scratch_two_calls_in_a_row_same_inputs():
    stream = torch.cuda.current_stream()
    w = Workload("static_c", 8, 64, 8, 128, 2048, "f16",
                 lens=("ragged", 1, 2048), seed=73)
    d = to_device(make_inputs(w, pad="nan"))
    ref = gq.gqa_decode(d["q"], d["k"], d["v"], d["seq_lens"], d["scale"])
    o1 = torch.empty_like(d["q"])
    o2 = torch.empty_like(d["q"])
    assert _call_static(d, o1, stream) == gq.GQA_OK
    assert _call_static(d, o2, stream) == gq.GQA_OK
    torch.cuda.synchronize()
    _check_pair(o1, ref)
    _check_pair(o2, ref)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def _pool_used_bytes(device: int) -> int:
    """Bytes in use from the device's default memory pool, the pool the
    library's stream-ordered scratch allocations come from."""
    from cuda.bindings import runtime as rt
    err, pool = rt.cudaDeviceGetDefaultMemPool(device)
    assert err == rt.cudaError_t.cudaSuccess, err
    err, v = rt.cudaMemPoolGetAttribute(
        pool, rt.cudaMemPoolAttr.cudaMemPoolAttrUsedMemCurrent)
    assert err == rt.cudaError_t.cudaSuccess, err
    return int(v)


def test_static_entry_point_allocates_nothing():
    """On a stream the allocating entry point has never seen, two calls of
    gqa_decode_static leave the device pool's usage unchanged (no per-stream
    scratch is created), and still match gqa_decode.  Control: the first
    gqa_decode call on a new stream does take its scratch from that pool, so
    the measurement would see an allocation."""
    w = Workload("static_d", 3, 64, 8, 128, 1200, "bf16",
                 lens=("list", 1200, 5, 640), seed=74)
    d = to_device(make_inputs(w, pad="nan"))
    ref = gq.gqa_decode(d["q"], d["k"], d["v"], d["seq_lens"], d["scale"])
    out = torch.empty_like(d["q"])
    torch.cuda.synchronize()
    dev = torch.cuda.current_device()
    fresh = torch.cuda.Stream()
    before = _pool_used_bytes(dev)
    for _ in range(2):
        assert _call_static(d, out, fresh) == gq.GQA_OK
    fresh.synchronize()
    assert _pool_used_bytes(dev) == before
    _check_pair(out, ref)

    other = torch.cuda.Stream()
    gq.gqa_decode(d["q"], d["k"], d["v"], d["seq_lens"], d["scale"],
                  out=out, stream=other)
    other.synchronize()
    assert _pool_used_bytes(dev) > before


def test_static_scratch_refuses_oversized_request():
    # B=32, Hq=Hkv=64, D=128 needs about 18 MB of scratch: refused with
    # GQA_ERR_UNSUPPORTED before anything is enqueued (the pointers are
    # never dereferenced)
    q = torch.empty((32, 64, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((32, 64, 64, 128), dtype=torch.bfloat16, device="cuda")
    lens = torch.full((32,), 64, dtype=torch.int32, device="cuda")
    st = gq.lib().gqa_decode_static(q.data_ptr(), k.data_ptr(), k.data_ptr(),
                                    lens.data_ptr(), 0.1, q.data_ptr(), 32, 64,
                                    64, 64, 128, gq.GQA_BF16,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == gq.GQA_ERR_UNSUPPORTED
    assert gq.gqa_last_launch_count() == 0
