"""bench.py's host side without a GPU: the command line parses, the algorithmic bytes of
the headline workload follow from its shapes, and the committed profile summary is read
only while the CUDA sources hash to the profiled ones."""
import os
import re
import subprocess
import sys

import bench
from speculative_decoding_token_temp_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_help_parses():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    for opt in ("--gpus", "--steps", "--warmup", "--impl", "--offset", "--multi"):
        assert opt in r.stdout


def test_headline_algorithmic_bytes():
    # every target and draft logit once plus one (target, draft) row pair per sequence,
    # plus tokens and both uniforms: the headline's 1247.69 MB
    w = synth.HEADLINE.make()
    ab = bench.algorithmic_bytes(w)
    B, g, V = 256, 8, 128256
    logits = (B * (g + 1) + B * g) * V * 2
    pairs = B * 2 * V * 2
    small = B * g * 4 * 2 + B * 4
    assert ab["stochastic"] == logits + pairs + small
    assert ab["greedy"] >= B * (g + 1) * V * 2


def test_profile_traffic_tracks_the_sources(tmp_path, monkeypatch):
    sha = bench.kernel_sources_sha256()
    assert re.fullmatch(r"[0-9a-f]{64}", sha)
    good = tmp_path / "good.md"
    good.write_text(f"x\n    sources_sha256: {sha}\n    traffic_bytes_per_call: 1234\n")
    monkeypatch.setattr(bench, "PROFILE", str(good))
    assert bench.profiled_traffic() == 1234
    stale = tmp_path / "stale.md"
    stale.write_text("    sources_sha256: " + "0" * 64 + "\n    traffic_bytes_per_call: 1234\n")
    monkeypatch.setattr(bench, "PROFILE", str(stale))
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE", str(tmp_path / "missing.md"))
    assert bench.profiled_traffic() is None
