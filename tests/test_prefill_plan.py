"""The prefill kernels' launch plan replayed on the host (no GPU): the
prefill source's own plan functions, compiled into a small host program
(tests/prefill_plan_replay.cu), for a sweep of token counts of every shape
the GPU tests run through the prefill kernels, checked for the K split
(one wave, at least two K blocks a chunk, exact cover), the scratch carve
against the handle's allocation, and K2's channel block."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152                                   # GB300

SHAPES = [(4, 2560, 320), (8, 4096, 512), (2, 256, 64), (1, 512, 128), (3, 192, 192),
          (8, 128, 256), (2, 2560, 320), (2, 8192, 320), (4, 8192, 320), (1, 40960, 320)]


@pytest.fixture(scope="module")
def replay(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("plan") / "prefill_plan_replay")
    res = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                          "--expt-relaxed-constexpr", os.path.join(ROOT, "tests", "prefill_plan_replay.cu"),
                          "-o", exe], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    return exe


@pytest.mark.parametrize("HC,HS,r", SHAPES, ids=[f"HC{s[0]}_HS{s[1]}_r{s[2]}" for s in SHAPES])
def test_prefill_plan_invariants(replay, HC, HS, r):
    res = subprocess.run([replay, str(HC), str(HS), str(r), str(SMS)],
                         capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-1000:]
    lines = res.stdout.splitlines()
    assert lines[-1] == "DONE fails=0"


def test_prefill_plan_at_the_default_shape(replay):
    # the plan the measurements rest on: K chunks only below 19 token tiles,
    # the halved K2 block only for a single tile
    res = subprocess.run([replay, "4", "2560", "320", str(SMS)], capture_output=True, text=True,
                         timeout=120)
    plan = {int(ln.split()[0][2:]): dict(kv.split("=") for kv in ln.split()[1:])
            for ln in res.stdout.splitlines() if ln.startswith("M=")}
    assert plan[1]["S"] == "20" and plan[128]["S"] == "20" and plan[512]["S"] == "9"
    assert plan[2048]["S"] == "2" and plan[4096]["S"] == "1" and plan[65536]["S"] == "1"
    assert plan[128]["ncu"] == "32" and plan[129]["ncu"] == "64" and plan[8192]["ncu"] == "64"
