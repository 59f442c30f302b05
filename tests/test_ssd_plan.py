"""The SSD kernels' launch plan (csrc/ssd_plan.h, host only): which walk a
problem takes, how the ticket walk cuts the heads and how many CTAs it
launches, compiled with the host compiler and checked on the CPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "selective_state_space_113_b300", "csrc")


@pytest.fixture(scope="module")
def plan_exe(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path_factory.mktemp("plan") / "ssd_plan_check")
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-I", CSRC,
                    os.path.join(ROOT, "tests", "ssd_plan_check.cpp"), "-o", exe], check=True)
    return exe


def plans(exe, *cases):
    args = [str(v) for c in cases for v in c]
    out = subprocess.run([exe, *args], capture_output=True, text=True, check=True).stdout
    return [tuple(int(v) for v in line.split()) for line in out.splitlines()]


def test_wave_tail_takes_the_ticket_walk(plan_exe):
    # the Mamba-2 2.7B-shaped layer: 320 heads of 32 chunks on 148 SMs
    # (2.16 waves, run as 3): the ticket walk, three segments of 11/11/10
    # chunks, 960 units on 148 CTAs
    assert plans(plan_exe, (320, 32, 148, 0, 0)) == [(1, 11, 3, 960, 148)]


def test_full_waves_and_few_heads_keep_one_head_per_cta(plan_exe):
    got = plans(plan_exe, (296, 32, 148, 0, 0), (148, 32, 148, 0, 0), (24, 64, 148, 0, 0),
                (1, 1, 148, 0, 0))
    assert got == [(0, 32, 1, 296, 296), (0, 32, 1, 148, 148), (0, 64, 1, 24, 24),
                   (0, 1, 1, 1, 1)]


def test_the_15_percent_rule(plan_exe):
    # 160 heads: 2 waves for 1.08 of work (85% above) -> tickets; 290 heads:
    # 2 waves for 1.96 (2% above) -> one head per CTA; 250: 2 for 1.69 (18%)
    got = plans(plan_exe, (160, 32, 148, 0, 0), (290, 32, 148, 0, 0), (250, 32, 148, 0, 0))
    assert [g[0] for g in got] == [1, 0, 1]


def test_segments_are_equal_and_cover_the_head(plan_exe):
    for heads, nch in [(320, 32), (160, 32), (600, 7), (149, 1), (500, 100), (200, 3)]:
        dyn, seg, nseg, units, ctas = plans(plan_exe, (heads, nch, 148, 0, 0))[0]
        assert dyn == 1
        assert 1 <= seg <= nch and nseg == -(-nch // seg) and units == heads * nseg
        assert seg * nseg >= nch > seg * (nseg - 1)        # the segments cover the head once
        assert ctas == min(units, 148)


def test_forced_segments_and_ctas(plan_exe):
    got = plans(plan_exe, (8, 5, 148, 1, 0), (8, 5, 148, 2, 3), (8, 5, 148, 9, 0),
                (21, 3, 148, 0, 5), (1000, 7, 148, 0, 0))
    # forced: the ticket walk even with few heads; a segment longer than the
    # head is the whole head; at most want_ctas CTAs (segments by the rule,
    # here whole heads).  1000 heads of 7 chunks fill 7 waves to 3.6%: one
    # head per CTA
    assert got == [(1, 1, 5, 40, 40), (1, 2, 3, 24, 3), (1, 5, 1, 8, 8), (1, 3, 1, 21, 5),
                   (0, 7, 1, 1000, 1000)]
