"""Repository rules that the code must keep (no GPU needed): committed files never reach into the
git-ignored scratch folder, sources stand on their own, and profiles/ holds text summaries only."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELF = os.path.relpath(os.path.abspath(__file__), ROOT)


def _tracked():
    try:
        out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True, check=True).stdout
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("git is not available")
    return [f for f in out.splitlines() if os.path.isfile(os.path.join(ROOT, f))]


def _text(path):
    try:
        with open(os.path.join(ROOT, path), encoding="utf-8") as f:
            return f.read()
    except UnicodeDecodeError:
        return ""


def test_nothing_committed_uses_the_scratch_folder():
    scratch = "_" + "work/"
    for f in _tracked():
        if f.endswith(".md") or f in (".gitignore", ".gpurunignore", SELF):
            continue
        assert scratch not in _text(f), f"{f} refers to the scratch folder"


def test_sources_do_not_point_at_the_build_notes():
    names = ["DESIGN" + ".md", "SURVEY" + ".md", "PAPER" + ".md", "VERDICT" + ".md", "ADVICE" + ".md"]
    exts = (".py", ".cu", ".cuh", ".h", ".c")
    for f in _tracked():
        if not f.endswith(exts) or f == SELF:
            continue
        text = _text(f)
        for n in names:
            assert n not in text, f"{f} names {n}"


def test_profiles_hold_text_only():
    for f in _tracked():
        if f.startswith("profiles/"):
            assert f.endswith((".md", ".txt")), f"{f}: profiles/ holds text summaries only"
