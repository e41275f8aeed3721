"""The decode kernel's launch plan replayed on the host (no GPU): the
kernel's own plan functions, compiled from its source into a small host
program (tests/geom_replay.cu), for every M of every shape the GPU tests run,
checked for shared-memory bounds, exact channel coverage, exchange capacity
and tensor-memory / issuer limits."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS, SMEM_OPTIN = 152, 232448          # GB300: SMs, opt-in shared memory per block (bytes)

# (HC, HS, r, every M in 1..32 must have a decode plan; larger M up to the
# kernel's limit may fall back to the prefill kernels)
SHAPES = [(4, 2560, 320, True), (8, 4096, 512, True), (4, 256, 32, True), (8, 128, 24, True),
          (2, 2560, 320, True), (2, 8192, 320, True), (4, 8192, 320, True), (4, 256, 64, True),
          (1, 40960, 320, False)]


@pytest.fixture(scope="module")
def replay(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("geom") / "geom_replay")
    res = subprocess.run([nvcc, "-std=c++17", "-O1", "-gencode", "arch=compute_103a,code=sm_103a",
                          "--expt-relaxed-constexpr", os.path.join(ROOT, "tests", "geom_replay.cu"),
                          "-o", exe], capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-3000:]
    return exe


@pytest.mark.parametrize("HC,HS,r,all_planned", SHAPES,
                         ids=[f"HC{s[0]}_HS{s[1]}_r{s[2]}" for s in SHAPES])
def test_decode_plan_invariants(replay, HC, HS, r, all_planned):
    res = subprocess.run([replay, str(HC), str(HS), str(r), str(SMS), str(SMEM_OPTIN)],
                         capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-1000:]
    lines = res.stdout.splitlines()
    assert lines[-1] == "DONE fails=0"
    planned = [ln for ln in lines if " plan G=" in ln]
    if all_planned:
        missing = [ln for ln in lines if "plan=none" in ln and int(ln.split()[0][2:]) <= 32]
        assert not missing, missing
    else:
        # no decode plan: the dispatcher sends these calls to the prefill kernels
        assert not planned
