"""Prefill path (tcgen05 tensor-core kernels) against the fp64 oracle.

Covers ragged token counts around the 128-row tile, the mid-batch workload
(M in {512, 1024, 2048} with the merged 336-row weight, folded and unfolded),
the large-M workload (M up to 65536) and the wide variant (HC=8, HS=4096,
r=512) -- both with every token row drawn from the seed and every row checked
against the oracle in a pool of worker processes --, agreement with the
decode path, and determinism.
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import PATH_DECODE, PATH_PREFILL, HcGatedResidual, inputs

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def case2k():
    return tl.make_case(2048)


def _sub(case, M):
    return dict(case, R=case["R"][:M], y=case["y"][:M], inj=case["inj"][:M], M=M)


def _run(case, max_M, path=PATH_PREFILL, Wdi=None, fold=False, shape=inputs.DEFAULT, rows=None):
    d = tl.device_case(case)
    with HcGatedResidual(max_M=max_M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        kw = dict(Wdi=tl.to_dev(Wdi), fold_w=fold) if Wdi is not None else dict(Wd=d["Wd"], Wi=d["Wi"])
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], force_path=path, check=True,
                         **kw)
    if rows is not None:
        import torch
        idx = torch.as_tensor(np.asarray(rows), device=out["x"].device)
        out = {k: v.index_select(0, idx) for k, v in out.items()}
    return out


@pytest.mark.parametrize("M", [1, 33, 100, 128, 129, 224, 257, 511])
def test_prefill_ragged_token_counts(torch_cuda, case2k, M):
    case = _sub(case2k, M)
    out = _run(case, M)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"prefill M={M}")


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("M", [512, 1024, 2048])
def test_prefill_mid_batch_merged_weight(torch_cuda, case2k, M, fold):
    case = _sub(case2k, M)
    Wdi = tl.merged_weight_bits(case, 336, fold)
    out = _run(case, M, Wdi=Wdi, fold=fold)
    tl.assert_parity(out, tl.oracle_ref(case, Wdi_bits=Wdi, fold_w=fold),
                     label=f"prefill merged fold={fold} M={M}")


@pytest.mark.parametrize("M", [512, 2048])
def test_prefill_separate_weights(torch_cuda, case2k, M):
    case = _sub(case2k, M)
    tl.assert_parity(_run(case, M), tl.oracle_ref(case), label=f"prefill M={M}")


@pytest.fixture(scope="module")
def pool():
    with tl.oracle_pool() as p:
        yield p


def _full_case(pool, M, shape, seed=inputs.SEED):
    acts = tl.pooled_activations(pool, M, shape, seed)
    return {"shape": shape, "M": M, **inputs.weights(shape, seed), **acts}


@pytest.mark.parametrize("M", [4096, 8192, 16384, 32768, 65536])
def test_prefill_large_M_every_row(torch_cuda, pool, M):
    case = _full_case(pool, M, inputs.DEFAULT)
    out = tl.host_outputs(_run(case, M))
    tl.assert_pooled_parity(pool, out, M, shape=inputs.DEFAULT, label=f"prefill M={M}")


@pytest.mark.parametrize("M", [64, 1024, 8192])
def test_prefill_wide_variant_every_row(torch_cuda, pool, M):
    case = _full_case(pool, M, inputs.WIDE)
    out = tl.host_outputs(_run(case, M, shape=inputs.WIDE))
    tl.assert_pooled_parity(pool, out, M, shape=inputs.WIDE, label=f"wide prefill M={M}")


def test_prefill_agrees_with_decode(torch_cuda, case2k):
    case = _sub(case2k, 32)
    a = _run(case, 32, path=PATH_PREFILL)
    b = _run(case, 32, path=PATH_DECODE)
    ref = tl.oracle_ref(case)
    tl.assert_parity(a, ref, label="prefill M=32")
    tl.assert_parity(b, ref, label="decode M=32")
    np.testing.assert_array_equal(tl.to_f64(a["R2"]), tl.to_f64(b["R2"]))


def test_prefill_deterministic(torch_cuda, case2k):
    torch = torch_cuda
    case = _sub(case2k, 300)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=300) as op:
        outs = [op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           force_path=PATH_PREFILL, check=True) for _ in range(3)]
    for k in outs[0]:
        for o in outs[1:]:
            assert torch.equal(o[k], outs[0][k]), k


def test_prefill_other_shapes(torch_cuda):
    for HC, HS, r, M in ((2, 256, 64, 200), (1, 512, 128, 130), (3, 192, 192, 77), (8, 128, 256, 300)):
        s = inputs.Shape(HC=HC, HS=HS, r=r)
        case = tl.make_case(M, s, seed=7)
        tl.assert_parity(_run(case, M, shape=s), tl.oracle_ref(case),
                         label=f"prefill HC={HC} HS={HS} r={r} M={M}")
