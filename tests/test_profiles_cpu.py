"""The ncu summaries under profiles/ quote the commands that produced them:
every `python bench.py ...` command there must be one the current bench.py
accepts, and every summary names the source hash its counters belong to."""
import glob
import os
import re
import shlex

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md")))


def _bench_commands(text):
    """bench.py argument lists in the summary's code blocks (variables such
    as P="python bench.py ..." and continued lines resolved)."""
    cmds = []
    for block in re.findall(r"```\n(.*?)```", text, flags=re.S):
        joined = block.replace("\\\n", " ")
        for line in joined.splitlines():
            line = line.split("#")[0].strip()
            m = re.search(r"python bench\.py([^\"']*)", line)
            if m:
                cmds.append(shlex.split(m.group(1)))
    return cmds


def test_there_are_summaries():
    assert len(PROFILES) >= 10


@pytest.mark.parametrize("path", PROFILES, ids=[os.path.basename(p) for p in PROFILES])
def test_summary_commands_parse(path):
    text = open(path).read()
    cmds = _bench_commands(text)
    assert cmds, f"{os.path.basename(path)}: no bench.py command quoted"
    for argv in cmds:
        args = bench.build_parser().parse_args(argv)  # SystemExit on an unknown flag
        assert args.warmup >= 3
    assert re.search(r"kernel_source_hash: `[0-9a-f]{16}`", text), "no source hash"
