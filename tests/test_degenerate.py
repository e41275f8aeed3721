"""Degenerate inputs of the method on the GPU, on the decode and the prefill
path, against the fp64 oracle (aiter PR #5913, "Technical Details": the
(COMBINE), (N), (G2) and (MIX) bullets at their limits):

  * injection logits +inf / -inf / 0, so iw = 2 / 0 / 1;
  * an all-zero token (R = y = 0): R2 = 0, rrms = 1 / sqrt(eps), xn = 0, so
    lora, inj_next and x are exactly 0;
  * 1 + Wnorm = 0 (Wnorm = -1): xn = 0 on every channel;
  * Wu = 0: G = 1/2 exactly, x = (1/2) mean_s xn;
  * y = 0: R2 equals R bit for bit.

Values so large that the fp32 sum of squares overflows (|R2| beyond ~1e17 at
HS = 2560) are outside what an fp32 implementation of (N) can represent and
are not exercised.
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import PATH_DECODE, PATH_PREFILL, HcGatedResidual, inputs

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu

PATHS = [(PATH_DECODE, 6), (PATH_PREFILL, 200)]


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _run(case, path):
    d = tl.device_case(case)
    with HcGatedResidual(max_M=case["M"]) as op:
        return op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                          force_path=path, check=True)


@pytest.mark.parametrize("path,M", PATHS)
def test_infinite_and_zero_injection_logits(torch_cuda, path, M):
    case = tl.make_case(M, seed=51)
    inj = case["inj"].copy()
    inj[0, :] = np.inf
    inj[1, :] = -np.inf
    inj[2, :] = 0.0
    inj[3, 0], inj[3, 1] = np.inf, -np.inf
    case["inj"] = inj
    out = _run(case, path)
    ref = tl.oracle_ref(case)
    tl.assert_parity(out, ref, label=f"inj limits path={path}")
    # iw = 0 drops y: R2 = R exactly on that token
    np.testing.assert_array_equal(tl.to_f64(out["R2"])[1], tl.f64(case, "R")[1])


@pytest.mark.parametrize("path,M", PATHS)
def test_all_zero_token(torch_cuda, path, M):
    case = tl.make_case(M, seed=52)
    for k in ("R", "y"):
        a = case[k].copy()
        a[2] = 0
        case[k] = a
    out = _run(case, path)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"zero token path={path}")
    for k in ("R2", "x", "lora", "inj_next"):
        assert np.all(tl.to_f64(out[k])[2] == 0.0), k
    np.testing.assert_allclose(tl.to_f64(out["rrms"])[2], 1.0 / np.sqrt(inputs.DEFAULT.eps), rtol=2e-3)


@pytest.mark.parametrize("path,M", PATHS)
def test_norm_weight_minus_one_zeroes_xn(torch_cuda, path, M):
    case = tl.make_case(M, seed=53)
    case["Wnorm"] = inputs.to_bf16_bits(np.full(inputs.DEFAULT.HC * inputs.DEFAULT.HS, -1.0))
    out = _run(case, path)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"Wnorm=-1 path={path}")
    for k in ("x", "lora", "inj_next"):
        assert np.all(tl.to_f64(out[k]) == 0.0), k


@pytest.mark.parametrize("path,M", PATHS)
def test_zero_up_weight_gives_half_gates(torch_cuda, path, M):
    case = tl.make_case(M, seed=54)
    case["Wu"] = np.zeros_like(case["Wu"])
    out = _run(case, path)
    ref = tl.oracle_ref(case)
    np.testing.assert_array_equal(ref["G"], 0.5)
    tl.assert_parity(out, ref, label=f"Wu=0 path={path}")


@pytest.mark.parametrize("path,M", PATHS)
def test_zero_block_output_keeps_R(torch_cuda, path, M):
    case = tl.make_case(M, seed=55)
    case["y"] = np.zeros_like(case["y"])
    out = _run(case, path)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"y=0 path={path}")
    np.testing.assert_array_equal(tl.to_f64(out["R2"]), tl.f64(case, "R"))
