"""bench.py's reference arm (the CPU oracle) keeps the JSON-line contract; runs
on the host only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.timeout(600)
def test_reference_arm_prints_one_json_line(tmp_path):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
           "--steps", "2", "--warmup", "1", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=str(tmp_path), timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["value"] > 0 and out["unit"] == "GB/s" and out["steps"] == 2
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == out["value"]
    assert out["e2e"]["h2d_bytes_per_step"] == 0 and out["e2e"]["value"] == out["value"]


def test_whole_job_rate_and_peak_helpers():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.whole_job_gbs(4, 1e9, 500.0) == pytest.approx(8.0)
    peak, kind = bench._peak_hbm()
    assert peak > 0 and kind in ("measured", "fallback")


def test_kernel_source_hash_ignores_comments_only(tmp_path):
    """The traffic record stays valid across comment edits and is voided by code edits."""
    sys.path.insert(0, ROOT)
    import bench

    src = os.path.join(ROOT, "e8_lattice_vector_gb300", "csrc")
    for name in ("a", "b", "c"):
        (tmp_path / name).mkdir()
    for f in sorted(os.listdir(src)):
        text = open(os.path.join(src, f), encoding="utf-8").read()
        (tmp_path / "a" / f).write_text(text, encoding="utf-8")
        (tmp_path / "b" / f).write_text("// a new comment line\n" + text.replace("\n", "  // note\n", 1),
                                        encoding="utf-8")
        (tmp_path / "c" / f).write_text(text + ("\nint extra_symbol = 1;\n" if f.endswith(".cu") else ""),
                                        encoding="utf-8")
    ha, hb, hc = (bench._kernel_src_hash(str(tmp_path / n)) for n in ("a", "b", "c"))
    assert ha == bench._kernel_src_hash()
    assert hb == ha
    assert hc != ha


def test_mode_selection_by_code_widths_and_parity():
    """--bits picks a config's mode by its code widths, --strict / --joint by its
    parity, --delta-chunk overrides the restart interval; a width pair the
    config does not serve is an error."""
    sys.path.insert(0, ROOT)
    import argparse

    import bench
    from e8_lattice_vector_gb300.synth import CONFIGS

    def pick(name, **kw):
        a = argparse.Namespace(strict=False, joint=False, delta_chunk=None, bits=None)
        for k, v in kw.items():
            setattr(a, k, v)
        return bench._pick_params(CONFIGS[name], a)

    p = pick("qwen25_14b")
    assert (p.key_bits, p.value_bits, p.strict, p.delta_chunk) == (3, 2, 0, 256)
    p = pick("qwen25_14b", bits="2,2", strict=True)
    assert (p.key_bits, p.value_bits, p.strict) == (2, 2, 1)
    p = pick("llama31_8b", joint=True, delta_chunk=32768)
    assert (p.key_bits, p.value_bits, p.strict, p.delta_chunk) == (2, 2, 2, 32768)
    with pytest.raises(SystemExit):
        pick("llama31_8b", bits="4,4")
