"""Host-side checks of bench.py (no GPU): the source hash that ties profiled
DRAM traffic to the kernel code, and the JSON line of the reference arm (the
CPU oracle), which runs anywhere."""
import json
import os
import shutil
import subprocess
import sys


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_layout():
    a = 'int x = 1;  // one\n/* block\n comment */ float y;\n'
    b = 'int x = 1;\nfloat   y;'
    assert bench._code_only(a) == bench._code_only(b)
    # literals survive, including comment markers and quotes inside them
    s = 'const char* p = "a//b /*c*/"; char q = \'"\';'
    assert bench._code_only(s) == s
    # a code change does not
    assert bench._code_only("int x = 1;") != bench._code_only("int x = 2;")


def _fake_root(tmp_path, traffic, sha):
    csrc = tmp_path / "grouped_query_attention_11_b300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(ROOT, "grouped_query_attention_11_b300",
                                 "csrc", name), csrc / name)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / bench.TRAFFIC_SUMMARY).write_text(
        "# summary\n\n"
        f"- traffic_bytes_per_launch w: `{traffic}` for `1000` algorithmic "
        "bytes\n"
        f"- kernel_sources_sha256: `{sha}`\n")
    return str(tmp_path)


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    sha = bench.kernel_sources_sha256()
    monkeypatch.setattr(bench, "ROOT", _fake_root(tmp_path, 12345, sha))
    assert bench.kernel_sources_sha256() == sha
    assert bench.profiled_traffic("w") == 12345
    assert bench.profiled_traffic("w", 1000) == 12345
    # another draw of the workload: scaled by its algorithmic bytes
    assert bench.profiled_traffic("w", 2000) == 24690
    assert bench.profiled_traffic("missing") is None
    # a comment added to a kernel source keeps the summary valid ...
    src = tmp_path / "grouped_query_attention_11_b300" / "csrc" / \
        bench.KERNEL_SOURCES[0]
    src.write_text(src.read_text() + "\n// a note\n")
    assert bench.profiled_traffic("w") == 12345
    # ... a code change does not
    src.write_text(src.read_text() + "\nstatic int changed = 1;\n")
    assert bench.profiled_traffic("w") is None


def test_reference_arm_json_line():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--workload", "tiny_b1_h8_kv2_d64_s128_f16", "--steps",
         "2", "--warmup", "3"],
        capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
              "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
              "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["warmup"] >= 3
    assert d["higher_is_better"] is False
    assert d["value"] > 0 and d["unit"] == "us/step"
    assert d["config"]["workload"] == "tiny_b1_h8_kv2_d64_s128_f16"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_committed_traffic_covers_every_workload_of_these_sources():
    """The committed ncu summary was taken from the kernel code in the tree
    (its hash matches) and gives a DRAM figure for every workload bench.py
    reports, so no line of the bench carries a null traffic; a kernel change
    without a new capture fails here."""
    from grouped_query_attention_11_b300.workloads import WORKLOADS
    missing = [n for n in WORKLOADS if bench.profiled_traffic(n) is None]
    assert not missing, (
        "DRAM-traffic summary is stale or incomplete for: " + ", ".join(missing))
    text = open(os.path.join(ROOT, bench.TRAFFIC_SUMMARY)).read()
    for name in WORKLOADS:
        line = next(x for x in text.splitlines()
                    if f"traffic_bytes_per_launch {name}:" in x)
        traffic, algo = [int(x) for x in line.split("`") if x.isdigit()]
        if algo < (1 << 20):
            # a 67 KB step: fixed per-launch bytes (seq_lens, the error
            # word, partial sectors) are of the same order as the data
            continue
        # one launch moves its algorithmic bytes once, plus the partials and
        # error words it writes: no re-reads (ncu's counts can fall a little
        # short where a few lines were still in L2)
        assert 0.99 * algo <= traffic <= 1.02 * algo, (name, traffic, algo)
