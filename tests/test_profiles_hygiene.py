"""The ncu summaries under profiles/ state the commands that made them; those
commands must leave the GPU's clocks alone and run files of this repository."""
import json
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _summaries():
    return sorted(f for f in os.listdir(PROFILES) if f.endswith(".md"))


def _ncu_lines(text):
    """The ncu command lines inside the summary's fenced code blocks."""
    out, fenced = [], False
    for ln in text.splitlines():
        if ln.strip().startswith("```"):
            fenced = not fenced
        elif fenced and re.match(r"\s*ncu\s", ln):
            out.append(ln.strip())
    return out


def test_every_summary_states_its_commands():
    for name in _summaries():
        text = open(os.path.join(PROFILES, name)).read()
        assert _ncu_lines(text), f"{name}: no ncu command"


def test_ncu_commands_keep_clocks_and_run_committed_files():
    assert os.path.exists(os.path.join(ROOT, "bench.py"))
    for name in _summaries():
        for ln in _ncu_lines(open(os.path.join(PROFILES, name)).read()):
            assert "--clock-control none" in ln, (name, ln)
            # the profiled program is this repository's bench.py
            assert re.search(r"\spython\s+bench\.py(\s|$)", ln), (name, ln)


def test_stored_traffic_entries_are_well_formed():
    tr = json.load(open(os.path.join(PROFILES, "traffic.json")))
    assert tr
    for kernel, ent in tr.items():
        assert ent["bytes_per_launch"] > 0, kernel
        assert re.fullmatch(r"[0-9a-f]{16}", ent["source_hash"]), kernel
        assert ent["workload"], kernel
