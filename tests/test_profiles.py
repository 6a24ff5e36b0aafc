"""The committed ncu summaries match the kernels they describe.

`bench.py` reports a kernel's measured DRAM traffic (`roofline.traffic`)
from the summary of its workload under `profiles/`, and only while the
summary's `sources` line equals the hash of the current CUDA sources.  These
checks make a stale summary fail the CPU suite instead of silently turning the
bench's traffic into null: every summary names the sources it was captured on,
carries a traffic line per kernel, and records a capture of one kernel and one
launch, with the clocks left alone.
"""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

import bench  # noqa: E402  (its hash and summary reader need no GPU)

SUMMARIES = sorted(glob.glob(os.path.join(ROOT, "profiles", "kernels_*.md")))


def _lines(path):
    with open(path) as f:
        return f.read().splitlines()


def test_summaries_exist():
    names = {os.path.basename(p) for p in SUMMARIES}
    # the bench's default workload, one workload per other head dim, and LMSD
    for want in ("kernels_recsys_full.md", "kernels_skewed_full.md", "kernels_full_full.md"):
        assert want in names
    assert any(n.startswith("kernels_lmsd_") for n in names)


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_summary_is_current(path):
    lines = _lines(path)
    src = [l.split()[1] for l in lines if l.startswith("sources ")]
    assert src == [bench.kernel_sources_sha()], (
        f"{os.path.basename(path)} was captured on other kernel sources; recapture it")


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_summary_traffic_lines(path):
    traffic = [l.split() for l in _lines(path) if l.startswith("traffic ")]
    assert len(traffic) == 2  # the two kernels of the summary
    for _, kernel, nbytes in traffic:
        assert kernel.startswith("hstu_")
        assert int(nbytes) > 0
    # the bench reads the same figures back
    for _, kernel, nbytes in traffic:
        assert bench.summary_traffic(path, kernel) == int(nbytes)


@pytest.mark.parametrize("path", SUMMARIES, ids=os.path.basename)
def test_capture_commands(path):
    text = "\n".join(_lines(path))
    # command lines (continued with a trailing backslash), not prose
    cmds = re.findall(r"^\s*ncu -[^\n]*(?:\\\n[^\n]*)*", text, flags=re.M)
    captures = [c for c in cmds if "--set full" in c]
    assert captures, "no full-set capture recorded"
    for c in cmds:
        if "-i " in c:  # reading a report back
            continue
        assert "--clock-control none" in c
    for c in captures:
        assert re.search(r"-k regex:\S+", c), c   # one kernel per capture
        assert re.search(r"-c 1\b", c), c         # one launch


def test_launch_list_command():
    path = os.path.join(ROOT, "profiles", "launches_recsys_fwd_bwd.md")
    text = "\n".join(_lines(path))
    cmds = re.findall(r"^\s*ncu -[^\n]*(?:\\\n[^\n]*)*", text, flags=re.M)
    assert cmds and all("--clock-control none" in c for c in cmds)
    # the launch list is the single-pass metric only
    assert all("--metrics gpu__time_duration.sum" in c for c in cmds)
