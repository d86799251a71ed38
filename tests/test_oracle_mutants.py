"""The oracle's pins catch plausible mistakes.

Each mutant below plants one slip of the kind a hand-written oracle could
carry (a wrong index, a dropped term or factor, a swapped operand, an
off-by-one bound, a wrong bias or width in a decoder, truncation instead of
rounding) into a private copy of the oracle, builds that copy with gcc and
runs the pin suite (tests/test_oracle_pins.py) against it.  The copy must
fail at least one pin; an unmutated copy, run the same way, must pass.  The
mistakes are planted on the CPU, in copies under a temporary directory: the
oracle in the tree is never changed."""
import concurrent.futures
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
C_SRC = "oracle/gqa_oracle.c"
PY_SRC = "oracle/__init__.py"

# name -> list of (file, exact text, replacement); each text occurs once
MUTANTS = {
    "head_mapping_interleaved": [
        (C_SRC, "const int kvh = h / G;", "const int kvh = h % p->Hkv;")],
    "chunk_head_mapping_interleaved": [
        (C_SRC, "attend(&p, b, h / G, (size_t)r * D,",
         "attend(&p, b, h % Hkv, (size_t)r * D,")],
    "score_scale_dropped": [
        (C_SRC, "scores[t] = p->scale * dot;", "scores[t] = dot;")],
    "score_sign_flipped": [
        (C_SRC, "dot += qd * kd;", "dot -= qd * kd;")],
    "softmax_not_normalised": [
        (C_SRC, "for (int t = 0; t < n; ++t) scores[t] /= z;", "(void)z;")],
    "values_read_from_keys": [
        (C_SRC, "load_elem(p->v, kv_off + (size_t)t * p->D + d, p->kv_dtype)",
         "load_elem(p->k, kv_off + (size_t)t * p->D + d, p->kv_dtype)")],
    "key_scale_dropped": [
        (C_SRC, "(size_t)t * p->D + d, p->kv_dtype) * ks;",
         "(size_t)t * p->D + d, p->kv_dtype);")],
    "key_value_scales_swapped": [
        (C_SRC, "const double ks = p->k_scale ? p->k_scale[",
         "const double ks = p->v_scale ? p->v_scale["),
        (C_SRC, "const double vs = p->v_scale ? p->v_scale[",
         "const double vs = p->k_scale ? p->k_scale[")],
    "last_token_dropped": [
        (C_SRC, "q_off, clamped_len(p, b), out", "q_off, clamped_len(p, b) - 1, out")],
    "kv_slab_index_transposed": [
        (C_SRC, "((size_t)b * p->Hkv + kvh) * (size_t)p->Smax",
         "((size_t)kvh * p->B + b) * (size_t)p->Smax")],
    "query_row_index_transposed": [
        (C_SRC, "((size_t)b * p->Hq + h) * p->D;",
         "((size_t)h * p->B + b) * p->D;")],
    "causal_bound_off_by_one": [
        (C_SRC, "int n = L - T + i + 1;", "int n = L - T + i;")],
    "e4m3_exponent_bias": [
        (C_SRC, "(double)f / 8.0, e - 7);", "(double)f / 8.0, e - 8);")],
    "e4m3_subnormal_scale": [
        (C_SRC, "mag = ldexp((double)f, -9);", "mag = ldexp((double)f, -10);")],
    "e5m2_fraction_width": [
        (C_SRC, "(double)f / 4.0, e - 15);", "(double)f / 8.0, e - 15);")],
    "f16_exponent_bias": [
        (C_SRC, "(double)f / 1024.0, e - 15);", "(double)f / 1024.0, e - 14);")],
    "bf16_fraction_width": [
        (C_SRC, "(double)f / 128.0, e - 127);", "(double)f / 256.0, e - 127);")],
    "cache_bytes_without_k_and_v": [
        (C_SRC, "return 2ull * (uint64_t)layers", "return 1ull * (uint64_t)layers")],
    "encoder_truncates": [
        (C_SRC, "double r = nearbyint((a / ldexp(1.0, e) - 1.0)",
         "double r = floor((a / ldexp(1.0, e) - 1.0)")],
    "append_rescale_ratio_inverted": [
        (C_SRC, "const float ratio = s / s2;", "const float ratio = s2 / s;")],
    "append_quantises_by_multiplying": [
        (C_SRC, "oracle_f32_to_fp8(x / s2, cache_dtype);",
         "oracle_f32_to_fp8(x * s2, cache_dtype);")],
    "paged_gather_reads_first_page": [
        (PY_SRC, "pg = int(table[b, i])", "pg = int(table[b, 0])")],
}


def _copy_tree(dst):
    """The oracle, the pins and what they import, without built files."""
    for d in ("oracle", "tests/golden"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d),
                        ignore=shutil.ignore_patterns("*.so", "*.o",
                                                      "__pycache__"))
    for f in ("tests/conftest.py", "tests/test_oracle_pins.py",
              "grouped_query_attention_11_b300/__init__.py",
              "grouped_query_attention_11_b300/workloads.py"):
        os.makedirs(os.path.dirname(os.path.join(dst, f)), exist_ok=True)
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))


def _plant(dst, edits):
    for path, old, new in edits:
        full = os.path.join(dst, path)
        text = open(full).read()
        assert text.count(old) == 1, (path, old)
        with open(full, "w") as f:
            f.write(text.replace(old, new))


def _run_pins(dst):
    """Builds the copy's oracle, then runs its pins; (return code, failed
    test names)."""
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    "-o", os.path.join(dst, "oracle", "liboracle.so"),
                    os.path.join(dst, C_SRC), "-lm"], check=True)
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest",
                        "tests/test_oracle_pins.py", "-q", "-x",
                        "-p", "no:cacheprovider", "-m", "not gpu"],
                       cwd=dst, env=env, capture_output=True, text=True,
                       timeout=600)
    failed = re.findall(r"FAILED tests/test_oracle_pins.py::(\S+)", r.stdout)
    return r.returncode, failed, r.stdout[-2000:]


def _case(tmp_root, name, edits):
    dst = os.path.join(tmp_root, name)
    _copy_tree(dst)
    _plant(dst, edits)
    return name, _run_pins(dst)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    cases = [("unmutated", [])] + list(MUTANTS.items())
    workers = max(1, min(8, (os.cpu_count() or 2) // 2))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = dict(ex.map(lambda c: _case(str(tmp_path), *c), cases))
    rc, failed, tail = results.pop("unmutated")
    assert rc == 0, "the unmutated copy must pass its pins:\n" + tail
    survivors = [n for n, (rc, failed, _) in results.items()
                 if rc != 1 or not failed]
    assert not survivors, "mutants no pin caught: " + ", ".join(
        f"{n} (rc {results[n][0]})" for n in survivors)
