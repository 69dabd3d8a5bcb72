"""The static tile schedule of the two-problem GEMM launch, on the CPU.

A linear's dgrad and wgrad GEMMs run as one persistent launch: the problem
with the costlier tiles is dealt round-robin over the CTA pairs, and the
other problem's tiles then go, in order, to whichever pair frees up first.
Each CTA evaluates its own share of that list schedule in closed form
(csrc/f8_sched.h).  tests/csrc/sched_check.cc compiles that header and
compares every worker's tile list with a direct simulation of the list
scheduler (a priority queue of free times), on the launch shapes of the
Llama-3.1 8B and 70B linears, exhaustively over small parameters, and on
random ones; identical lists also mean every tile is run exactly once.  The
planner's tile counts, costs and decisions to share a launch are pinned for
the backward passes of the Llama-3.1 8B and 70B linears (grouped: the
attention projections; not grouped: the FFN linears)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_closed_form_schedule_equals_list_scheduling(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "sched_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-Wall", "-Werror", "-o", str(exe),
                    os.path.join(HERE, "csrc", "sched_check.cc")], check=True)
    r = subprocess.run([str(exe), "20000"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert " 0 mismatches" in r.stdout
