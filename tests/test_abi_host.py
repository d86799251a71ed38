"""Host-only checks of the C-ABI library: it loads without a GPU, exports every
function include/gqa.h declares, and rejects bad arguments on the host before
any CUDA call (so these run on a machine with no GPU)."""
import ctypes
import math
import os
import re

import pytest

import grouped_query_attention_11_b300 as gq
from grouped_query_attention_11_b300 import build as gq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")


@pytest.fixture(scope="module")
def L():
    gq_build.build()
    return gq.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert {"gqa_decode", "gqa_decode_fp8", "gqa_kv_bytes_per_token",
            "gqa_status_string"} <= set(names)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in gq.SIGNATURES, name


@pytest.mark.parametrize("args,expected", [
    ((80, 8, 128, 2), 327_680), ((80, 64, 128, 2), 2_621_440),
    ((80, 1, 128, 2), 40_960), ((32, 32, 128, 2), 524_288),
    ((32, 8, 128, 2), 131_072), ((32, 1, 128, 2), 16_384),
    ((32, 8, 128, 1), 65_536), ((40, 40, 128, 2), 819_200),
    ((40, 8, 128, 2), 163_840), ((0, 8, 128, 2), 0), ((80, -1, 128, 2), 0),
])
def test_kv_bytes_per_token(L, args, expected):
    # the pages' cache-size figures (cache-size formula, 2 x layers x kv_heads
    # x head_dim x bytes per element)
    assert gq.gqa_kv_bytes_per_token(*args) == expected


def test_status_strings(L):
    for st in range(5):
        assert gq.gqa_status_string(st)
    assert gq.gqa_status_string(99) == "unknown status"


# Fake, well-aligned "device" addresses: the library must reject the call on
# the host before it ever dereferences or hands them to CUDA.
A = 1 << 20


def _call(q=A, k=A * 2, v=A * 3, lens=A * 4, scale=0.125, out=A * 5, B=2,
          Hq=8, Hkv=2, Smax=128, D=64, dtype=gq.GQA_BF16):
    return gq.lib().gqa_decode(q, k, v, lens, scale, out, B, Hq, Hkv, Smax, D,
                               dtype, None)


def _call8(q=A, k=A * 2, v=A * 3, ks=A * 6, vs=A * 7, lens=A * 4, scale=0.125,
           out=A * 5, B=2, Hq=8, Hkv=2, Smax=128, D=64, kv=gq.GQA_E4M3,
           dtype=gq.GQA_BF16):
    return gq.lib().gqa_decode_fp8(q, k, v, ks, vs, lens, scale, out, B, Hq,
                                   Hkv, Smax, D, kv, dtype, None)


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(k=None), dict(v=None), dict(lens=None), dict(out=None),
    dict(q=A + 8), dict(k=A * 2 + 2), dict(out=A * 5 + 4), dict(lens=A * 4 + 2),
    dict(B=0), dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(Hq=8, Hkv=3),
    dict(Smax=0), dict(scale=0.0), dict(scale=-1.0), dict(scale=math.inf),
    dict(scale=math.nan), dict(dtype=gq.GQA_E4M3), dict(dtype=7),
])
def test_decode_rejects_invalid_arguments(L, kw):
    gq.lib().gqa_set_num_ctas(0)
    assert _call(**kw) == gq.GQA_ERR_INVALID_ARG
    assert gq.gqa_last_launch_count() == 0


@pytest.mark.parametrize("kw", [dict(D=96), dict(D=256), dict(D=32)])
def test_decode_unsupported_head_dim(L, kw):
    assert _call(**kw) == gq.GQA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kw", [
    dict(ks=None), dict(vs=None), dict(ks=A * 6 + 2), dict(q=None),
    dict(dtype=gq.GQA_E4M3), dict(Hq=6, Hkv=4), dict(scale=0.0),
    dict(kv=gq.GQA_BF16), dict(kv=gq.GQA_F16), dict(kv=9),
    dict(kv=gq.GQA_E5M2, ks=None), dict(kv=gq.GQA_E5M2, B=0),
])
def test_decode_fp8_rejects_invalid_arguments(L, kw):
    assert _call8(**kw) == gq.GQA_ERR_INVALID_ARG


def test_device_errors_rejects_null_flags(L):
    assert gq.lib().gqa_device_errors(None, None) == gq.GQA_ERR_INVALID_ARG


def test_product_path_has_no_oracle_dependency():
    # The CUDA library and its binding never import or link the oracle.
    pkg = os.path.join(ROOT, "grouped_query_attention_11_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text
                assert "liboracle" not in text and "gqa_oracle" not in text


def _callp(q=A, k=A * 2, v=A * 3, bt=A * 8, lens=A * 4, scale=0.125,
           out=A * 5, B=2, Hq=8, Hkv=2, num_pages=16, page_size=64,
           max_pages=4, D=64, dtype=gq.GQA_BF16):
    return gq.lib().gqa_decode_paged(q, k, v, bt, lens, scale, out, B, Hq, Hkv,
                                     num_pages, page_size, max_pages, D, dtype,
                                     None)


@pytest.mark.parametrize("kw", [
    dict(bt=None), dict(bt=A * 8 + 2), dict(num_pages=0), dict(max_pages=0),
    dict(page_size=0), dict(q=None), dict(dtype=gq.GQA_E4M3), dict(Hq=6, Hkv=4),
    dict(scale=0.0), dict(B=0),
])
def test_decode_paged_rejects_invalid_arguments(L, kw):
    assert _callp(**kw) == gq.GQA_ERR_INVALID_ARG
    assert gq.gqa_last_launch_count() == 0


@pytest.mark.parametrize("kw", [dict(page_size=32), dict(page_size=100),
                                dict(D=96)])
def test_decode_paged_unsupported(L, kw):
    assert _callp(**kw) == gq.GQA_ERR_UNSUPPORTED


def _calla(kn=A, vn=A * 2, kc=A * 3, vc=A * 4, ks=A * 6, vs=A * 7, lens=A * 5,
           B=2, Hkv=2, Smax=64, D=64, ind=gq.GQA_BF16, cd=gq.GQA_E4M3):
    return gq.lib().gqa_append_kv(kn, vn, kc, vc, ks, vs, lens, B, Hkv, Smax,
                                  D, ind, cd, None)


@pytest.mark.parametrize("kw", [
    dict(kn=None), dict(vc=None), dict(lens=None), dict(kn=A + 8),
    dict(lens=A * 5 + 2), dict(ks=None), dict(vs=A * 7 + 1), dict(B=0),
    dict(Hkv=0), dict(Smax=0), dict(ind=gq.GQA_E4M3),
    dict(ind=gq.GQA_F16, cd=gq.GQA_BF16), dict(cd=9),
])
def test_append_rejects_invalid_arguments(L, kw):
    assert _calla(**kw) == gq.GQA_ERR_INVALID_ARG
    assert gq.gqa_last_launch_count() == 0


def test_append_unsupported_head_dim(L):
    assert _calla(D=96) == gq.GQA_ERR_UNSUPPORTED


def test_decode_chunk_rejects_invalid_arguments(L):
    lib = gq.lib()
    assert lib.gqa_decode_chunk(A, A * 2, A * 3, A * 4, 0.125, A * 5, 2, 8, 2,
                                0, 64, 64, gq.GQA_BF16, None) == \
        gq.GQA_ERR_INVALID_ARG
    assert lib.gqa_decode_chunk(A, A * 2, A * 3, A * 4, 0.125, A * 5, 2, 8, 3,
                                2, 64, 64, gq.GQA_BF16, None) == \
        gq.GQA_ERR_INVALID_ARG
    assert lib.gqa_decode_chunk(A, A * 2, A * 3, A * 4, 0.125, A * 5, 2, 8, 2,
                                2, 64, 96, gq.GQA_BF16, None) == \
        gq.GQA_ERR_UNSUPPORTED


def header_enum(prefix):
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return {k: int(v) for k, v in re.findall(
        rf"\b({prefix}[A-Z0-9_]+)\s*=\s*(\d+)", text)}


def test_binding_constants_match_the_header():
    for prefix in ("GQA_TUNE_", "GQA_ERR_", "GQA_E", "GQA_F16", "GQA_BF16"):
        for name, value in header_enum(prefix).items():
            assert getattr(gq, name) == value, name
    assert set(header_enum("GQA_TUNE_")) == {
        "GQA_TUNE_NO_L2_WARMUP", "GQA_TUNE_NO_CLUSTER",
        "GQA_TUNE_NO_NARROW_ROWS"}


def test_tuning_and_release_need_no_gpu(L):
    # host-only settings; releasing a stream the library never used is a
    # no-op (it touches no device)
    L.gqa_set_tuning(7)
    L.gqa_set_tuning(0)
    assert L.gqa_release_stream(None) == gq.GQA_OK
