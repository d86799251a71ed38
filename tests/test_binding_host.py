"""Host checks of the Python binding's argument validation (no GPU): tensors
whose shapes, dtypes or devices disagree are rejected with ValueError before
the C call, because the library sizes every device access from q's and the
cache's dimensions.  The C library is replaced by a recorder, and the
CUDA-tensor check by a no-op, so CPU tensors stand in for device ones."""
import pytest
import torch

import grouped_query_attention_11_b300 as gq


class _Recorder:
    """Stands in for the loaded library: every entry point returns GQA_OK and
    records that it was reached."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            return gq.GQA_OK
        fn.__name__ = name
        return fn


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(gq, "lib", lambda: r)
    monkeypatch.setattr(gq, "_check_dev", lambda name, t: None)
    return r


B, HQ, HKV, S, D = 2, 8, 2, 64, 64
BF = torch.bfloat16


def _base():
    return dict(q=torch.zeros(B, HQ, D, dtype=BF),
                k=torch.zeros(B, HKV, S, D, dtype=BF),
                v=torch.zeros(B, HKV, S, D, dtype=BF),
                lens=torch.zeros(B, dtype=torch.int32),
                out=torch.zeros(B, HQ, D, dtype=BF))


def _decode(fn, a):
    return fn(a["q"], a["k"], a["v"], a["lens"], 0.125, out=a["out"],
              stream=0)


BAD = {
    "v_smaller": ("v", torch.zeros(B, HKV, S // 2, D, dtype=BF)),
    "out_smaller": ("out", torch.zeros(B, HQ - 1, D, dtype=BF)),
    "out_dtype": ("out", torch.zeros(B, HQ, D, dtype=torch.float16)),
    "lens_short": ("lens", torch.zeros(B - 1, dtype=torch.int32)),
    "k_batch": ("k", torch.zeros(B + 1, HKV, S, D, dtype=BF)),
    "k_head_dim": ("k", torch.zeros(B, HKV, S, D // 2, dtype=BF)),
    "q_rank": ("q", torch.zeros(B, HQ, 1, D, dtype=BF)),
}


@pytest.mark.parametrize("entry", ["gqa_decode", "gqa_decode_static"])
def test_decode_accepts_consistent_tensors(rec, entry):
    _decode(getattr(gq, entry), _base())
    assert rec.calls == [entry]


@pytest.mark.parametrize("entry", ["gqa_decode", "gqa_decode_static"])
@pytest.mark.parametrize("bad", list(BAD))
def test_decode_rejects_inconsistent_tensors(rec, entry, bad):
    a = _base()
    key, t = BAD[bad]
    a[key] = t
    with pytest.raises(ValueError):
        _decode(getattr(gq, entry), a)
    assert rec.calls == []


def _fp8_args():
    a = _base()
    a["k"] = a["k"].to(torch.float8_e4m3fn)
    a["v"] = a["v"].to(torch.float8_e4m3fn)
    a["ks"] = torch.ones(B, HKV)
    a["vs"] = torch.ones(B, HKV)
    return a


def _fp8(a):
    return gq.gqa_decode_fp8(a["q"], a["k"], a["v"], a["ks"], a["vs"],
                             a["lens"], 0.125, out=a["out"], stream=0)


def test_decode_fp8_checks_scales_and_out(rec):
    _fp8(_fp8_args())
    assert rec.calls == ["gqa_decode_fp8"]
    for key, t in (("ks", torch.ones(B, HKV + 1)), ("vs", torch.ones(B)),
                   ("out", torch.zeros(B, HQ, D, dtype=torch.float16)),
                   ("v", torch.zeros(B, HKV, S - 1, D,
                                     dtype=torch.float8_e4m3fn))):
        a = _fp8_args()
        a[key] = t
        with pytest.raises(ValueError):
            _fp8(a)
    assert rec.calls == ["gqa_decode_fp8"]


def test_decode_chunk_checks_shapes(rec):
    T = 3
    q = torch.zeros(B, HQ, T, D, dtype=BF)
    k = torch.zeros(B, HKV, S, D, dtype=BF)
    lens = torch.zeros(B, dtype=torch.int32)
    gq.gqa_decode_chunk(q, k, k.clone(), lens, 0.1, out=torch.zeros_like(q),
                        stream=0)
    assert rec.calls == ["gqa_decode_chunk"]
    with pytest.raises(ValueError):
        gq.gqa_decode_chunk(q, k, k.clone(), lens, 0.1,
                            out=torch.zeros(B, HQ, T - 1, D, dtype=BF),
                            stream=0)
    with pytest.raises(ValueError):
        gq.gqa_decode_chunk(q[:, :, 0], k, k.clone(), lens, 0.1, stream=0)
    assert rec.calls == ["gqa_decode_chunk"]


def test_decode_paged_checks_shapes(rec):
    pages = torch.zeros(7, HKV, 64, D, dtype=BF)
    q = torch.zeros(B, HQ, D, dtype=BF)
    table = torch.zeros(B, 3, dtype=torch.int32)
    lens = torch.zeros(B, dtype=torch.int32)
    gq.gqa_decode_paged(q, pages, pages.clone(), table, lens, 0.1, stream=0)
    assert rec.calls == ["gqa_decode_paged"]
    for kw in (dict(block_table=torch.zeros(B + 1, 3, dtype=torch.int32)),
               dict(v_pages=torch.zeros(6, HKV, 64, D, dtype=BF)),
               dict(seq_lens=torch.zeros(B + 2, dtype=torch.int32))):
        args = dict(q=q, k_pages=pages, v_pages=pages.clone(),
                    block_table=table, seq_lens=lens)
        args.update(kw)
        with pytest.raises(ValueError):
            gq.gqa_decode_paged(args["q"], args["k_pages"], args["v_pages"],
                                args["block_table"], args["seq_lens"], 0.1,
                                stream=0)
    assert rec.calls == ["gqa_decode_paged"]


def test_append_checks_shapes(rec):
    kc = torch.zeros(B, HKV, S, D, dtype=torch.float8_e4m3fn)
    kn = torch.zeros(B, HKV, D, dtype=BF)
    lens = torch.zeros(B, dtype=torch.int32)
    sc = torch.ones(B, HKV)
    gq.gqa_append_kv(kn, kn.clone(), kc, kc.clone(), lens, k_scale=sc,
                     v_scale=sc.clone(), stream=0)
    assert rec.calls == ["gqa_append_kv"]
    bad = [dict(v_new=torch.zeros(B, HKV, D - 8, dtype=BF)),
           dict(v_cache=torch.zeros(B, HKV, S - 1, D,
                                    dtype=torch.float8_e4m3fn)),
           dict(seq_lens=torch.zeros(B + 1, dtype=torch.int32)),
           dict(k_scale=torch.ones(B))]
    for kw in bad:
        args = dict(k_new=kn, v_new=kn.clone(), k_cache=kc,
                    v_cache=kc.clone(), seq_lens=lens, k_scale=sc,
                    v_scale=sc.clone())
        args.update(kw)
        with pytest.raises(ValueError):
            gq.gqa_append_kv(args["k_new"], args["v_new"], args["k_cache"],
                             args["v_cache"], args["seq_lens"],
                             k_scale=args["k_scale"], v_scale=args["v_scale"],
                             stream=0)
    assert rec.calls == ["gqa_append_kv"]
