"""Repository hygiene: the design notes stay readable and name files that
exist, and no source file names a path of the build machine."""
import collections
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tracked(exts):
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:
        files = []
        for d, _, fs in os.walk(ROOT):
            if "/." in d or "/_work" in d or "gpurun_out" in d:
                continue
            files += [os.path.relpath(os.path.join(d, f), ROOT) for f in fs]
    else:
        files = out.stdout.split()
    return [f for f in files if f.endswith(exts)]


def test_design_notes_have_no_repeated_lines():
    with open(os.path.join(ROOT, "DESIGN.md"), encoding="utf-8") as f:
        lines = [l for l in f.read().split("\n") if len(l) > 40]
    counts = collections.Counter(lines)
    worst = counts.most_common(1)[0] if counts else ("", 0)
    assert worst[1] <= 2, f"line repeated {worst[1]} times: {worst[0][:80]}"
    assert len(lines) < 2000


def test_design_file_map_names_existing_files():
    with open(os.path.join(ROOT, "DESIGN.md"), encoding="utf-8") as f:
        text = f.read()
    names = set(re.findall(r"`((?:csrc|tests|oracle|include|profiles|synth)/[\w./-]+)`", text))
    assert names
    pkg = "global_attention_sinks_swa_b300"
    for n in names:
        cands = [os.path.join(ROOT, n), os.path.join(ROOT, pkg, n)]
        assert any(os.path.exists(c.rstrip("/")) for c in cands), n


def test_sources_name_no_machine_path():
    bad = re.compile("/" + "root/")
    me = os.path.relpath(os.path.abspath(__file__), ROOT)
    for rel in _tracked((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
        if rel == me:
            continue
        with open(os.path.join(ROOT, rel), encoding="utf-8", errors="replace") as f:
            for i, line in enumerate(f, 1):
                assert not bad.search(line), f"{rel}:{i}: {line.strip()}"
