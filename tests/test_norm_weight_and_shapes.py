"""The [HS] norm weight shared by every stream, and other HC / HS, against the
fp64 oracle (aiter PR #5913, "Validation and unverified scope": full-width
norm weights beside the default, an untuned hidden size with HC=2, and wide
streams with HS=8192 and 40960).

Each case runs on the decode path (M <= 32) and on the prefill path, for the
fused call, the mix alone and folded merged weights.
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import PATH_AUTO, PATH_DECODE, PATH_PREFILL, HcGatedResidual, inputs

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _broadcast_case(M, shape, seed):
    # the [HS] norm weight: the seeded weight's first stream slice
    case = tl.make_case(M, shape, seed=seed)
    case["Wnorm"] = np.ascontiguousarray(case["Wnorm"][:shape.HS])
    return case


def _fused(case, path, Wdi=None, fold=False, mix=False):
    sh = case["shape"]
    d = tl.device_case(case)
    with HcGatedResidual(max_M=case["M"], HC=sh.HC, HS=sh.HS, r=sh.r) as op:
        kw = dict(Wdi=tl.to_dev(Wdi), fold_w=fold) if Wdi is not None else dict(Wd=d["Wd"], Wi=d["Wi"])
        if mix:
            return op.mix(d["R"], d["Wnorm"], d["Wu"], force_path=path, check=True, **kw)
        return op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], force_path=path,
                          check=True, **kw)


@pytest.mark.parametrize("path,M", [(PATH_DECODE, 1), (PATH_DECODE, 6), (PATH_PREFILL, 300),
                                    (PATH_PREFILL, 1024)])
def test_broadcast_norm_weight(torch_cuda, path, M):
    case = _broadcast_case(M, inputs.DEFAULT, seed=41)
    out = _fused(case, path)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"[HS] Wnorm M={M}")


@pytest.mark.parametrize("path,M", [(PATH_DECODE, 8), (PATH_PREFILL, 512)])
def test_broadcast_norm_weight_folded_merged(torch_cuda, path, M):
    case = _broadcast_case(M, inputs.DEFAULT, seed=42)
    Wdi = tl.merged_weight_bits(case, 336, True)
    out = _fused(case, path, Wdi=Wdi, fold=True)
    tl.assert_parity(out, tl.oracle_ref(case, Wdi_bits=Wdi, fold_w=True),
                     label=f"[HS] Wnorm folded M={M}")


@pytest.mark.parametrize("path,M", [(PATH_DECODE, 4), (PATH_PREFILL, 200)])
def test_broadcast_norm_weight_mix_only(torch_cuda, path, M):
    case = _broadcast_case(M, inputs.DEFAULT, seed=43)
    out = _fused(case, path, mix=True)
    tl.assert_parity(out, tl.oracle_mix_ref(case), label=f"[HS] Wnorm mix M={M}")


def test_broadcast_equals_tiled_full_width(torch_cuda):
    # the [HS] weight and the K-entry weight that repeats it give the same
    # bits on both paths
    torch = torch_cuda
    for path, M in ((PATH_DECODE, 5), (PATH_PREFILL, 260)):
        case = _broadcast_case(M, inputs.DEFAULT, seed=44)
        a = _fused(case, path)
        full = dict(case, Wnorm=np.tile(case["Wnorm"], inputs.DEFAULT.HC))
        b = _fused(full, path)
        for k in ("R2", "x", "rrms", "lora", "inj_next"):
            assert torch.equal(a[k], b[k]), (path, k)


OTHER_SHAPES = [inputs.Shape(HC=2, HS=2560, r=320), inputs.Shape(HC=2, HS=8192, r=320),
                inputs.Shape(HC=4, HS=8192, r=320), inputs.Shape(HC=1, HS=40960, r=320)]


@pytest.mark.parametrize("shape", OTHER_SHAPES, ids=lambda s: f"HC{s.HC}_HS{s.HS}")
@pytest.mark.parametrize("M", [3, 32, 257])
def test_other_hc_hs(torch_cuda, shape, M):
    case = tl.make_case(M, shape, seed=45)
    out = _fused(case, PATH_AUTO)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"HC={shape.HC} HS={shape.HS} M={M}")
