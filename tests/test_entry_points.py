"""The combine-only and mix-only entry points (aiter PR #5913, "Behavior and
intent": the combine and mix entry points beside combine_and_mix) against
the fp64 oracle, and against the fused call on the same inputs.

combine: R2 = bf16(R + y * 2 sigmoid(inj / HC)) alone, with a strided inj
(the previous call's inj_next view).  Its R2 must equal, bit for bit, the R2
the fused call stores (both paths form it with the same weight and rounding).
mix: every step after COMBINE on R taken as the combined residual; on the
decode path (M <= 32) and the prefill path, folded and unfolded weights.
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import (ERR_ALIAS, ERR_INVALID_ARG, ERR_UNSUPPORTED,
                                          PATH_DECODE, PATH_PREFILL, HcGatedResidual, HcGrError,
                                          inputs)

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu

SMALL = inputs.Shape(HC=4, HS=256, r=64)


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _bits(t):
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy()


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("M,shape", [(1, inputs.DEFAULT), (5, inputs.DEFAULT), (32, inputs.DEFAULT),
                                     (300, inputs.DEFAULT), (7, SMALL), (1000, SMALL),
                                     (3, inputs.WIDE)])
def test_combine_matches_oracle_and_fused_R2(torch_cuda, M, shape):
    torch = torch_cuda
    case = tl.make_case(M, shape, seed=21)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        R2 = op.combine(d["R"], d["y"], d["inj"])
        fused = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           check=True)
        torch.cuda.synchronize()
    ref, _ = tl.oracle.combine(tl.f64(case, "R"), tl.f64(case, "y"), tl.f64(case, "inj"))
    g = tl.to_f64(R2)
    assert np.max(np.abs(g - ref) / (tl.TOL_BF16 * (1.0 + np.abs(ref)))) <= 1.0
    np.testing.assert_array_equal(_bits(R2), _bits(fused["R2"]))


def test_combine_strided_inj_view(torch_cuda):
    # inj taken from a wider row (stride 8 floats), like the inj_next columns
    # of a packed [M, n_pad] projection output
    torch = torch_cuda
    M, shape = 37, SMALL
    case = tl.make_case(M, shape, seed=22)
    d = tl.device_case(case)
    wide = torch.zeros((M, 8), dtype=torch.float32, device="cuda")
    wide[:, 3:3 + shape.HC] = d["inj"]
    view = wide[:, 3:3 + shape.HC]
    assert view.stride(0) == 8
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        a = op.combine(d["R"], d["y"], view)
        b = op.combine(d["R"], d["y"], d["inj"])
        torch.cuda.synchronize()
    np.testing.assert_array_equal(_bits(a), _bits(b))


def test_combine_special_values(torch_cuda):
    # y = 0 gives R2 = R; inj = -inf gives iw = 0, so R2 = R with no NaN.
    torch = torch_cuda
    M, shape = 9, SMALL
    case = tl.make_case(M, shape, seed=23)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        a = op.combine(d["R"], torch.zeros_like(d["y"]), d["inj"])
        b = op.combine(d["R"], d["y"], torch.full_like(d["inj"], -float("inf")))
        torch.cuda.synchronize()
    r = tl.to_f64(d["R"])
    np.testing.assert_array_equal(tl.to_f64(a), r)
    np.testing.assert_array_equal(tl.to_f64(b), r)


@pytest.fixture(scope="module")
def pool():
    with tl.oracle_pool() as p:
        yield p


def test_combine_full_size_every_row(torch_cuda, pool):
    # the 65536-token workload: bit-identical to the fused prefill R2 on every
    # element, and within tolerance of the oracle on every row
    torch = torch_cuda
    M, seed = 65536, 24
    case = {"shape": inputs.DEFAULT, "M": M, **inputs.weights(inputs.DEFAULT, seed),
            **tl.pooled_activations(pool, M, inputs.DEFAULT, seed)}
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M) as op:
        R2 = op.combine(d["R"], d["y"], d["inj"])
        fused = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           check=True, want_lora=False)
        torch.cuda.synchronize()
        assert torch.equal(R2.view(torch.int16), fused["R2"].view(torch.int16))
    del fused
    tl.assert_pooled_parity(pool, tl.host_outputs({"R2": R2}), M, shape=inputs.DEFAULT, seed=seed,
                            kind="combine", label="combine M=65536")


def test_combine_rejects(torch_cuda):
    torch = torch_cuda
    M, shape = 4, SMALL
    case = tl.make_case(M, shape, seed=25)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        with pytest.raises(HcGrError) as e:
            op.combine(d["R"], d["y"], d["inj"], out=d["R"])          # in place
        assert e.value.status == ERR_ALIAS
        lib, h = op._lib, op._h
        s = torch.cuda.current_stream().cuda_stream
        out = torch.empty_like(d["R"])
        args = (d["R"].data_ptr(), d["y"].data_ptr(), d["inj"].data_ptr())
        assert lib.hc_gr_combine(h, 0, 4, 256, *args, 4, out.data_ptr(), s) == ERR_INVALID_ARG
        assert lib.hc_gr_combine(h, M, 4, 256, *args, 3, out.data_ptr(), s) == ERR_INVALID_ARG
        assert lib.hc_gr_combine(h, M, 4, 256, args[0] + 2, args[1], args[2], 4, out.data_ptr(),
                                 s) == ERR_INVALID_ARG
        assert lib.hc_gr_combine(h, M, 4, 252, *args, 4, out.data_ptr(), s) == ERR_UNSUPPORTED
        assert lib.hc_gr_combine(h, M, 4, 256, *args, 4, None, s) == ERR_INVALID_ARG


# ------------------------------------------------------------------ mix
def _mix(case, path, shape, Wdi=None, fold=False):
    d = tl.device_case(case)
    with HcGatedResidual(max_M=case["M"], HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        kw = dict(Wdi=tl.to_dev(Wdi), fold_w=fold) if Wdi is not None else dict(Wd=d["Wd"], Wi=d["Wi"])
        return op.mix(d["R"], d["Wnorm"], d["Wu"], force_path=path, check=True, **kw)


@pytest.mark.parametrize("M", [1, 5, 32])
def test_mix_decode_matches_oracle(torch_cuda, M):
    case = tl.make_case(M, inputs.DEFAULT, seed=26)
    out = _mix(case, PATH_DECODE, inputs.DEFAULT)
    assert "R2" not in out
    tl.assert_parity(out, tl.oracle_mix_ref(case), label=f"mix decode M={M}")


@pytest.mark.parametrize("M", [33, 129, 512])
def test_mix_prefill_matches_oracle(torch_cuda, M):
    case = tl.make_case(M, inputs.DEFAULT, seed=27)
    out = _mix(case, PATH_PREFILL, inputs.DEFAULT)
    tl.assert_parity(out, tl.oracle_mix_ref(case), label=f"mix prefill M={M}")


@pytest.mark.parametrize("path,M", [(PATH_DECODE, 8), (PATH_PREFILL, 1024)])
@pytest.mark.parametrize("fold", [False, True])
def test_mix_merged_weight(torch_cuda, path, M, fold):
    case = tl.make_case(M, inputs.DEFAULT, seed=28)
    Wdi = tl.merged_weight_bits(case, 336, fold)
    out = _mix(case, path, inputs.DEFAULT, Wdi=Wdi, fold=fold)
    tl.assert_parity(out, tl.oracle_mix_ref(case, Wdi_bits=Wdi, fold_w=fold),
                     label=f"mix merged fold={fold} M={M}")


@pytest.mark.parametrize("path,M", [(PATH_DECODE, 4), (PATH_PREFILL, 300)])
def test_mix_equals_fused_with_nothing_injected(torch_cuda, path, M):
    # y = 0 makes COMBINE the identity on bf16 R, so the fused call and the
    # mix compute from the same residual: x, rrms, lora and inj_next agree
    # bit for bit
    torch = torch_cuda
    case = tl.make_case(M, inputs.DEFAULT, seed=29)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M) as op:
        m = op.mix(d["R"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"], force_path=path, check=True)
        f = op.forward(d["R"], torch.zeros_like(d["y"]), d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"],
                       Wi=d["Wi"], force_path=path, check=True)
        torch.cuda.synchronize()
    for k in ("x", "rrms", "lora", "inj_next"):
        assert torch.equal(m[k], f[k]), k


def test_mix_wide_shape(torch_cuda):
    case = tl.make_case(8, inputs.WIDE, seed=30)
    out = _mix(case, PATH_DECODE, inputs.WIDE)
    tl.assert_parity(out, tl.oracle_mix_ref(case), label="mix wide decode")


def test_mix_full_size_every_row(torch_cuda, pool):
    torch = torch_cuda
    M, seed = 65536, 31
    case = {"shape": inputs.DEFAULT, "M": M, **inputs.weights(inputs.DEFAULT, seed),
            **tl.pooled_activations(pool, M, inputs.DEFAULT, seed)}
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M) as op:
        out = op.mix(d["R"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"], check=True)
        torch.cuda.synchronize()
    tl.assert_pooled_parity(pool, tl.host_outputs(out), M, shape=inputs.DEFAULT, seed=seed,
                            kind="mix", label="mix M=65536")


def test_mix_rejects_partial_null(torch_cuda):
    # y given without inj (or the reverse) is neither the fused call nor the mix
    torch = torch_cuda
    case = tl.make_case(4, SMALL, seed=32)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=4, HC=4, HS=256, r=64) as op:
        args, out = op.prepare(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"])
        args.inj = None
        with pytest.raises(HcGrError) as e:
            op.launch(args, torch.cuda.current_stream().cuda_stream)
        assert e.value.status == ERR_INVALID_ARG
        with pytest.raises(HcGrError):
            op.forward(d["R"], d["y"], None, d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"])
