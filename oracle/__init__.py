"""fp64 CPU oracle for the GQA decode step — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The CUDA library never links or calls
it, and this package imports nothing from the CUDA library: the two meet only
through the seeded inputs the tests generate.

The arithmetic lives in ``gqa_oracle.c`` (plain C, fp64, plain loops); this
module only builds it with gcc and marshals numpy arrays through ctypes.  The
method it follows, with the passages it restates, is described in the C file's
header: scaled dot-product attention per query head, query head h reading KV
head floor(h / G), softmax over the valid cached tokens, optional FP8 E4M3 /
E5M2 cache values times a per-(sequence, KV head) scale.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16, E4M3, F64, E5M2 = 0, 1, 2, 3, 4

_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc -O2 (no fast-math) and OpenMP."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    vp, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.oracle_gqa_decode.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, f64, vp,
                                      i32, i32, i32, i32, i32, i32]
    lib.oracle_gqa_decode.restype = i32
    lib.oracle_gqa_decode_rows.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, f64,
                                           vp, i32, vp, i32, i32, i32, i32, i32,
                                           i32]
    lib.oracle_gqa_decode_rows.restype = i32
    lib.oracle_gqa_weights.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, f64,
                                       i32, i32, vp, vp, i32, i32, i32, i32, i32]
    lib.oracle_gqa_weights.restype = i32
    lib.oracle_kv_bytes_per_token.argtypes = [i32, i32, i32, i32]
    lib.oracle_kv_bytes_per_token.restype = ctypes.c_uint64
    lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_f64.restype = f64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = f64
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = f64
    lib.oracle_e5m2_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_to_f64.restype = f64
    lib.oracle_gqa_decode_chunk.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp,
                                            f64, vp, i32, i32, i32, i32, i32,
                                            i32, i32]
    lib.oracle_gqa_decode_chunk.restype = i32
    lib.oracle_f32_to_fp8.argtypes = [ctypes.c_float, i32]
    lib.oracle_f32_to_fp8.restype = ctypes.c_uint8
    lib.oracle_append_kv.argtypes = [vp, vp, i32, vp, vp, i32, vp, vp, vp,
                                     i32, i32, i32, i32]
    lib.oracle_append_kv.restype = i32
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    _lib = lib
    return lib


# --------------------------------------------------------------- marshalling

def _as_raw(x, what):
    """numpy/torch CPU array -> (contiguous numpy array, element type code).

    16-bit floats travel as their raw bit patterns (uint16) and FP8 as raw
    bytes (uint8); the oracle decodes them itself.
    """
    try:  # accept torch CPU tensors without making torch a hard dependency
        import torch
        if isinstance(x, torch.Tensor):
            if x.is_cuda:
                raise ValueError(f"{what}: the oracle takes host tensors only")
            x = x.contiguous()
            if x.dtype == torch.float16:
                return x.view(torch.uint16).numpy(), F16
            if x.dtype == torch.bfloat16:
                return x.view(torch.uint16).numpy(), BF16
            if x.dtype == torch.float8_e4m3fn:
                return x.view(torch.uint8).numpy(), E4M3
            if x.dtype == torch.float8_e5m2:
                return x.view(torch.uint8).numpy(), E5M2
            if x.dtype == torch.uint8:
                return x.numpy(), E4M3
            x = x.double().numpy()
    except ImportError:
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16), F16
    if x.dtype == np.uint8:
        return x, E4M3
    return np.ascontiguousarray(x, dtype=np.float64), F64


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _scales(s):
    if s is None:
        return None
    try:
        import torch
        if isinstance(s, torch.Tensor):
            s = s.double().numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(s, dtype=np.float64)


def _lens(seq_lens):
    try:
        import torch
        if isinstance(seq_lens, torch.Tensor):
            seq_lens = seq_lens.cpu().numpy()
    except ImportError:
        pass
    return np.ascontiguousarray(seq_lens, dtype=np.int32)


def gqa_decode(q, k, v, seq_lens, scale, *, k_scale=None, v_scale=None,
               nthreads: int = 0) -> np.ndarray:
    """out[B, Hq, D] (float64) of one GQA decode step.

    q: [B, Hq, D]; k, v: [B, Hkv, Smax, D] (float16/bfloat16/float64 values, or
    FP8 E4M3 / E5M2 codes with ``k_scale``/``v_scale`` of shape [B, Hkv]);
    seq_lens: [B] valid cached tokens per sequence.
    """
    lib = _load()
    qa, qt = _as_raw(q, "q")
    ka, kt = _as_raw(k, "k")
    va, vt = _as_raw(v, "v")
    if kt != vt:
        raise ValueError("k and v must share an element type")
    B, Hq, D = qa.shape
    _, Hkv, Smax, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    lens = _lens(seq_lens)
    ks, vs = _scales(k_scale), _scales(v_scale)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = lib.oracle_gqa_decode(_ptr(qa), qt, _ptr(ka), _ptr(va), kt, _ptr(ks),
                               _ptr(vs), _ptr(lens), float(scale), _ptr(out),
                               B, Hq, Hkv, Smax, D, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gqa_decode rejected its arguments")
    return out


def gqa_decode_chunk(q, k, v, seq_lens, scale, *, k_scale=None,
                     v_scale=None, nthreads: int = 0) -> np.ndarray:
    """out[B, Hq, T, D] (float64) for T new tokens per sequence (the last T
    of its seq_lens[b] cached tokens), each attending causally: token i sees
    cached tokens t <= seq_lens[b] - T + i.  q: [B, Hq, T, D]."""
    lib = _load()
    qa, qt = _as_raw(q, "q")
    ka, kt = _as_raw(k, "k")
    va, vt = _as_raw(v, "v")
    if kt != vt:
        raise ValueError("k and v must share an element type")
    B, Hq, T, D = qa.shape
    _, Hkv, Smax, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    lens = _lens(seq_lens)
    ks, vs = _scales(k_scale), _scales(v_scale)
    out = np.zeros((B, Hq, T, D), dtype=np.float64)
    rc = lib.oracle_gqa_decode_chunk(_ptr(qa), qt, _ptr(ka), _ptr(va), kt,
                                     _ptr(ks), _ptr(vs), _ptr(lens),
                                     float(scale), _ptr(out), B, Hq, Hkv, T,
                                     Smax, D, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gqa_decode_chunk rejected its arguments")
    return out


def gqa_decode_paged(q, k_pages, v_pages, block_table, seq_lens, scale, *,
                     nthreads: int = 0) -> np.ndarray:
    """out[B, Hq, D] (float64) of one decode step over a paged cache.

    k_pages, v_pages: [num_pages, Hkv, page_size, D]; block_table: [B,
    max_pages], entry (b, i) the page of tokens [i*page_size, (i+1)*page_size)
    of sequence b.  The pages of each sequence are gathered back into a
    contiguous cache (tokens in order) and the contiguous oracle runs on it.
    """
    ka, kt = _as_raw(k_pages, "k_pages")
    va, vt = _as_raw(v_pages, "v_pages")
    table = block_table.cpu().numpy() if hasattr(block_table, "cpu") \
        else np.asarray(block_table)
    table = np.ascontiguousarray(table, dtype=np.int32)
    lens = _lens(seq_lens)
    _, Hkv, page_size, D = ka.shape
    B, max_pages = table.shape
    Smax = max_pages * page_size
    kc = np.zeros((B, Hkv, Smax, D), dtype=ka.dtype)
    vc = np.zeros((B, Hkv, Smax, D), dtype=va.dtype)
    for b in range(B):
        L = min(max(int(lens[b]), 0), Smax)
        for i in range(-(-L // page_size)):
            pg = int(table[b, i])
            if not 0 <= pg < ka.shape[0]:
                raise ValueError(f"block_table[{b}, {i}] = {pg} out of range")
            kc[b, :, i * page_size:(i + 1) * page_size] = ka[pg]
            vc[b, :, i * page_size:(i + 1) * page_size] = va[pg]
    qa, qt = _as_raw(q, "q")
    lib = _load()
    B2, Hq, D2 = qa.shape
    out = np.zeros((B2, Hq, D2), dtype=np.float64)
    lens_c = np.minimum(np.maximum(lens, 0), Smax).astype(np.int32)
    rc = lib.oracle_gqa_decode(_ptr(qa), qt, _ptr(kc), _ptr(vc), kt, None,
                               None, _ptr(lens_c), float(scale), _ptr(out),
                               B2, Hq, Hkv, Smax, D2, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gqa_decode rejected its arguments")
    return out


def gqa_decode_rows(q, k, v, seq_lens, scale, bh, *, k_scale=None,
                    v_scale=None, nthreads: int = 0) -> np.ndarray:
    """Output rows [n, D] (float64) for the (b, h) pairs in ``bh`` ([n, 2])."""
    lib = _load()
    qa, qt = _as_raw(q, "q")
    ka, kt = _as_raw(k, "k")
    va, vt = _as_raw(v, "v")
    B, Hq, D = qa.shape
    _, Hkv, Smax, _ = ka.shape
    pairs = np.ascontiguousarray(np.asarray(bh, dtype=np.int32).reshape(-1, 2))
    n = pairs.shape[0]
    lens = _lens(seq_lens)
    ks, vs = _scales(k_scale), _scales(v_scale)
    out = np.zeros((n, D), dtype=np.float64)
    rc = lib.oracle_gqa_decode_rows(_ptr(qa), qt, _ptr(ka), _ptr(va), kt,
                                    _ptr(ks), _ptr(vs), _ptr(lens), float(scale),
                                    _ptr(pairs), n, _ptr(out), B, Hq, Hkv, Smax,
                                    D, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gqa_decode_rows rejected its arguments")
    return out


def gqa_weights(q, k, v, seq_lens, scale, b, h, *, k_scale=None,
                v_scale=None):
    """(weights[L], out_row[D]) of one (b, h) row: the debug entry."""
    lib = _load()
    qa, qt = _as_raw(q, "q")
    ka, kt = _as_raw(k, "k")
    va, _ = _as_raw(v, "v")
    B, Hq, D = qa.shape
    _, Hkv, Smax, _ = ka.shape
    lens = _lens(seq_lens)
    ks, vs = _scales(k_scale), _scales(v_scale)
    w = np.zeros(Smax, dtype=np.float64)
    row = np.zeros(D, dtype=np.float64)
    L = lib.oracle_gqa_weights(_ptr(qa), qt, _ptr(ka), _ptr(va), kt, _ptr(ks),
                               _ptr(vs), _ptr(lens), float(scale), int(b), int(h),
                               _ptr(w), _ptr(row), B, Hq, Hkv, Smax, D)
    if L < 0:
        raise ValueError("oracle_gqa_weights rejected its arguments")
    return w[:L].copy(), row


def f32_to_fp8(v: float, kind: int) -> int:
    """The oracle's fp32 -> 8-bit code (E4M3 or E5M2), RNE, clamped."""
    return int(_load().oracle_f32_to_fp8(float(v), int(kind)))


def append_kv(k_new, v_new, k_cache, v_cache, seq_lens, *, k_scale=None,
              v_scale=None):
    """One cache append on host copies: returns (k_cache, v_cache, k_scale,
    v_scale, seq_lens, flags) after writing the new rows.  k_new / v_new
    [B, Hkv, D] float16 / bfloat16; caches [B, Hkv, Smax, D] in the same
    16-bit type or FP8 E4M3 / E5M2 (then k_scale / v_scale [B, Hkv] fp32)."""
    import torch
    lib = _load()
    kn, it = _as_raw(k_new, "k_new")
    vn, _ = _as_raw(v_new, "v_new")
    kc, ct = _as_raw(k_cache.clone(), "k_cache")
    vc, _ = _as_raw(v_cache.clone(), "v_cache")
    kc, vc = kc.copy(), vc.copy()
    B, Hkv, Smax, D = kc.shape
    lens = np.ascontiguousarray(_lens(seq_lens).copy())
    ks = vs = None
    if k_scale is not None:
        ks = np.ascontiguousarray(k_scale.numpy().astype(np.float32).copy())
        vs = np.ascontiguousarray(v_scale.numpy().astype(np.float32).copy())
    flags = lib.oracle_append_kv(_ptr(kn), _ptr(vn), it, _ptr(kc), _ptr(vc),
                                 ct, _ptr(ks), _ptr(vs), _ptr(lens), B, Hkv,
                                 Smax, D)
    return kc, vc, ks, vs, lens, int(flags)


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                       bytes_per_elem: int) -> int:
    return int(_load().oracle_kv_bytes_per_token(layers, kv_heads, head_dim,
                                                 bytes_per_elem))


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(bits: int) -> float:
    return _load().oracle_e4m3_to_f64(bits)


def e5m2_to_f64(bits: int) -> float:
    return _load().oracle_e5m2_to_f64(bits)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def timed_decode(*args, **kwargs):
    """(out, seconds) of gqa_decode, wall clock, for the CPU baseline."""
    t0 = time.perf_counter()
    out = gqa_decode(*args, **kwargs)
    return out, time.perf_counter() - t0
