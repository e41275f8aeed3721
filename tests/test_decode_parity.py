"""Decode path (M <= 32) against the fp64 oracle, through the C ABI.

Shapes: the single-token case and the decode sweep (HC=4, HS=2560, r=320,
M in {1, 2, 4, 8, 16, 32}) plus ragged token counts, the merged 336-row
weight folded and unfolded, a strided inj, and the wide variant (HC=8,
HS=4096, r=512, heavy-tailed R, y x10).
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import PATH_DECODE, HcGatedResidual, inputs

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def case32():
    return tl.make_case(32)


@pytest.fixture(scope="module")
def ref32(case32):
    return tl.oracle_ref(case32)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 16, 17, 31, 32])
def test_decode_default_shape(torch_cuda, case32, ref32, M):
    case = dict(case32, R=case32["R"][:M], y=case32["y"][:M], inj=case32["inj"][:M], M=M)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=32) as op:
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                         force_path=PATH_DECODE, check=True)
    ref = {k: v[:M] for k, v in ref32.items()}
    tl.assert_parity(out, ref, label=f"decode M={M}")


@pytest.mark.parametrize("fold", [False, True])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_decode_merged_weight(torch_cuda, case32, M, fold):
    case = dict(case32, R=case32["R"][:M], y=case32["y"][:M], inj=case32["inj"][:M], M=M)
    Wdi = tl.merged_weight_bits(case, 336, fold)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=32) as op:
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wdi=tl.to_dev(Wdi),
                         fold_w=fold, force_path=PATH_DECODE, check=True)
    ref = tl.oracle_ref(case, Wdi_bits=Wdi, fold_w=fold)
    tl.assert_parity(out, ref, label=f"decode merged fold={fold} M={M}")


def test_decode_strided_inj(torch_cuda, case32):
    # inj given as a column slice of a wider buffer (row stride 336), the way a
    # previous layer's packed output would hand it over.
    torch = torch_cuda
    M = 8
    case = dict(case32, R=case32["R"][:M], y=case32["y"][:M], inj=case32["inj"][:M], M=M)
    d = tl.device_case(case)
    packed = torch.full((M, 336), float("nan"), device="cuda")
    packed[:, 320:324] = d["inj"]
    inj_view = packed[:, 320:324]
    assert inj_view.stride() == (336, 1)
    with HcGatedResidual(max_M=32) as op:
        out = op.forward(d["R"], d["y"], inj_view, d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                         force_path=PATH_DECODE, check=True)
    tl.assert_parity(out, tl.oracle_ref(case), label="strided inj")


@pytest.mark.parametrize("M", [1, 8, 24, 32])
def test_decode_wide_variant(torch_cuda, M):
    # M = 1, 8: the two-role plan with rings on both roles; from 24 tokens the
    # planner moves to more up CTAs (only a forced decode reaches those plans)
    case = tl.make_case(M, inputs.WIDE)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=32, HC=8, HS=4096, r=512) as op:
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                         force_path=PATH_DECODE, check=True)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"wide decode M={M}")


def test_decode_small_shapes(torch_cuda):
    # shapes far from the defaults: HC=2 and HC=3, narrow streams, slices that
    # leave some CTAs without channels
    for HC, HS, r, M in ((2, 64, 16, 3), (3, 1024, 64, 5), (1, 512, 8, 2), (8, 128, 32, 32)):
        s = inputs.Shape(HC=HC, HS=HS, r=r)
        case = tl.make_case(M, s, seed=5)
        d = tl.device_case(case)
        with HcGatedResidual(max_M=M, HC=HC, HS=HS, r=r) as op:
            out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"],
                             Wi=d["Wi"], force_path=PATH_DECODE, check=True)
        tl.assert_parity(out, tl.oracle_ref(case), label=f"HC={HC} HS={HS} r={r} M={M}")


def test_decode_deterministic_and_batch_invariant(torch_cuda, case32):
    torch = torch_cuda
    d = tl.device_case(case32)
    with HcGatedResidual(max_M=32) as op:
        outs = [op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           force_path=PATH_DECODE, check=True) for _ in range(3)]
        one = op.forward(d["R"][5:6], d["y"][5:6], d["inj"][5:6], d["Wnorm"], d["Wu"],
                         Wd=d["Wd"], Wi=d["Wi"], force_path=PATH_DECODE, check=True)
    for k in outs[0]:
        for o in outs[1:]:
            assert torch.equal(o[k], outs[0][k]), k
    # row 5 alone against row 5 inside M=32: the same up to the summation order
    rep = tl.parity_report({k: v for k, v in one.items()},
                           {k: tl.to_f64(v)[5:6] for k, v in outs[0].items()})
    assert max(rep.values()) <= 0.5, rep
    np.testing.assert_array_equal(tl.to_f64(one["R2"]), tl.to_f64(outs[0]["R2"])[5:6])


@pytest.fixture(scope="module")
def case64():
    return tl.make_case(64, seed=71)


@pytest.mark.parametrize("M", [33, 40, 56, 64])
def test_decode_beyond_32_tokens(torch_cuda, case64, M):
    # the decode kernel up to its 64-token limit (exchange blocks of one
    # token's whole output row from M = 40 on)
    case = dict(case64, R=case64["R"][:M], y=case64["y"][:M], inj=case64["inj"][:M], M=M)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=64) as op:
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                         force_path=PATH_DECODE, check=True)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"decode M={M}")


@pytest.mark.parametrize("M,wide", [(33, False), (64, False), (65, False), (511, False),
                                    (20, True), (21, True)])
def test_auto_dispatch_around_the_crossover(torch_cuda, M, wide):
    # PATH_AUTO takes the decode kernel up to the measured crossover (M * K up
    # to 64 tokens at K = 10240: 64 tokens at the default shape, 20 at the
    # wide one) and the prefill kernels above; both sides of it, at both
    # shapes, match the oracle
    from hyper_connection_gated_gb300 import PATH_AUTO

    shape = inputs.WIDE if wide else inputs.DEFAULT
    case = tl.make_case(M, seed=72, shape=shape)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                         force_path=PATH_AUTO, check=True)
    tl.assert_parity(out, tl.oracle_ref(case), label=f"auto M={M}")


def test_decode_token_counts_alternate_on_one_handle(torch_cuda, case32, ref32):
    # consecutive calls of one handle with different plans (block sizes,
    # role splits) and both launch modes: each call leaves the reduce-scatter
    # words empty and the all-gather copy of the next parity ready
    torch = torch_cuda
    d = tl.device_case(case32)
    seq = [(1, False), (2, True), (8, True), (1, True), (1, True), (32, False), (2, False),
           (2, True), (4, True), (1, False), (3, True), (2, True)]
    with HcGatedResidual(max_M=32) as op:
        outs = [op.forward(d["R"][:M], d["y"][:M], d["inj"][:M], d["Wnorm"], d["Wu"], Wd=d["Wd"],
                           Wi=d["Wi"], force_path=PATH_DECODE, pdl=pdl) for M, pdl in seq]
        op.check()
        torch.cuda.synchronize()
    for (M, pdl), out in zip(seq, outs):
        tl.assert_parity(out, {k: v[:M] for k, v in ref32.items()}, label=f"M={M} pdl={pdl}")
