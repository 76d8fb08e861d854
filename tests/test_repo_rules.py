"""Rules of the repository that hold without a GPU.

The product path (the package: its Python binding and its CUDA sources) never reaches
the oracle, which is test infrastructure only; nothing committed uses the scratch
folder; every profiler command recorded under profiles/ leaves the GPU's clocks as it
found them; the working folders stay out of the commits.
"""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "aux_loss_free_gb300")


def _files(top, exts):
    for dirpath, dirnames, filenames in os.walk(top):
        dirnames[:] = [d for d in dirnames if not d.startswith((".", "_build", "__pycache__"))]
        for name in filenames:
            if name.endswith(exts):
                yield os.path.join(dirpath, name)


def test_the_product_path_does_not_reach_the_oracle():
    bad = []
    pat = re.compile(r"^\s*(from\s+oracle\b|import\s+oracle\b)|\boracle[/\\]")
    for path in _files(PKG, (".py", ".cu", ".cuh", ".h", ".cpp")):
        with open(path, encoding="utf-8") as fh:
            for n, line in enumerate(fh, 1):
                if pat.search(line):
                    bad.append(f"{os.path.relpath(path, ROOT)}:{n}: {line.strip()}")
    assert not bad, "\n".join(bad)


def test_nothing_committed_uses_the_scratch_folder():
    bad = []
    tops = [PKG, os.path.join(ROOT, "tests"), os.path.join(ROOT, "oracle"), os.path.join(ROOT, "synth")]
    files = [p for t in tops for p in _files(t, (".py", ".cu", ".cuh", ".h"))]
    files += [os.path.join(ROOT, f) for f in ("bench.py", "__graft_entry__.py")]
    me = os.path.abspath(__file__)
    for path in files:
        if os.path.abspath(path) == me:
            continue
        with open(path, encoding="utf-8") as fh:
            text = fh.read()
        if re.search(r"['\"/]_work[/'\"]", text):
            bad.append(os.path.relpath(path, ROOT))
    assert not bad, bad


def test_profiler_commands_leave_the_clocks_alone():
    prof = os.path.join(ROOT, "profiles")
    bad = []
    for path in _files(prof, (".md", ".txt")):
        with open(path, encoding="utf-8") as fh:
            for n, line in enumerate(fh, 1):
                if re.search(r"(^|[\s`'\"])ncu\s+--(set|metrics|section)", line) and "--clock-control none" not in line:
                    bad.append(f"{os.path.relpath(path, ROOT)}:{n}")
    assert not bad, bad


def test_the_scratch_folder_is_ignored():
    with open(os.path.join(ROOT, ".gitignore"), encoding="utf-8") as fh:
        lines = {ln.strip().rstrip("/") for ln in fh if ln.strip() and not ln.startswith("#")}
    assert "_work" in lines or "/_work" in lines
