"""bench.py's reference arm (the FP64 oracle timed on the host cores) prints the
one JSON line the bench contract asks for.  CPU only: a short sample."""
import json
import os
import subprocess
import sys

from gdn_testutil import ROOT


def test_reference_arm_json_line():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-seconds", "0.3"], capture_output=True, text=True, cwd=ROOT, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.strip().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["higher_is_better"] is False and d["n_gpus"] == 1
    assert d["unit"] == "µs/token/layer" and d["value"] > 0 and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("gdn-prefill")


def test_profile_tables_parse_and_follow_the_sources(tmp_path, monkeypatch):
    """The bench reads the recorded DRAM bytes and instruction counts only while a
    row's source hash matches the kernel file; a changed file gives None."""
    sys.path.insert(0, ROOT)
    import bench

    csrc = os.path.join(ROOT, "linear_attention_recurrence_gb300", "csrc")
    rows = [ln for ln in open(os.path.join(ROOT, "profiles", "flop_counts.md")) if "csrc/gdn_chunk_tmem.cu" in ln]
    assert rows, "the tensor-memory kernel has a counts row"
    counts = bench.captured_counts("gdn_chunk_tmem.cu")
    if counts is not None:  # the row matches the current source: tcgen05 ops are counted
        cells = [c.strip() for c in rows[0].strip().strip("|").split("|")]
        assert counts["tensor_flop"] == int(cells[9]) * 2048 + int(cells[10])
        assert bench.captured_traffic("gdn_chunk_tmem.cu") is not None

    # a copy of the tree whose kernel source differs from the recorded hash
    fake = tmp_path / "repo"
    (fake / "profiles").mkdir(parents=True)
    (fake / "linear_attention_recurrence_gb300" / "csrc").mkdir(parents=True)
    for name in ("flop_counts.md", "dram_traffic.md"):
        (fake / "profiles" / name).write_text(open(os.path.join(ROOT, "profiles", name)).read())
    src = open(os.path.join(csrc, "gdn_chunk_tmem.cu")).read()
    (fake / "linear_attention_recurrence_gb300" / "csrc" / "gdn_chunk_tmem.cu").write_text(src + "\n// edited\n")
    monkeypatch.setattr(bench, "ROOT", str(fake))
    assert bench.captured_counts("gdn_chunk_tmem.cu") is None
    assert bench.captured_traffic("gdn_chunk_tmem.cu") is None
