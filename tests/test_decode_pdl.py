"""Decode kernel launched as a programmatic dependent of the previous kernel
(hc_gr_args.pdl = 1): back-to-back calls on one stream -- different token
counts, different inputs, eager and captured in a CUDA graph -- each match the
fp64 oracle, and match the same calls made with plain stream order bit for
bit (the arithmetic does not depend on how the launches overlap).
"""
import numpy as np
import pytest

from hyper_connection_gated_gb300 import PATH_DECODE, HcGatedResidual

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu

MS = (2, 32, 1, 8, 5, 16)


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def cases():
    # one weight set, a different activation seed for every call
    out = []
    for i, M in enumerate(MS):
        out.append(tl.make_case(M, seed=1000 + i))
    return out


def _run_sequence(op, devs, pdl, torch):
    outs = []
    for d in devs:
        outs.append(op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"],
                               Wi=d["Wi"], force_path=PATH_DECODE, pdl=pdl))
    op.check()
    torch.cuda.synchronize()
    return outs


def test_pdl_back_to_back_matches_oracle_and_plain_order(torch_cuda, cases):
    torch = torch_cuda
    devs = [tl.device_case(c) for c in cases]
    with HcGatedResidual(max_M=32) as op:
        plain = _run_sequence(op, devs, False, torch)
        for _ in range(2):   # twice: the exchange buffers' call parity alternates
            pdl = _run_sequence(op, devs, True, torch)
            for c, o, ref_o in zip(cases, pdl, plain):
                tl.assert_parity(o, tl.oracle_ref(c), label=f"pdl M={c['M']}")
                for k in o:
                    assert torch.equal(o[k], ref_o[k]), (c["M"], k)


def test_pdl_in_cuda_graph(torch_cuda, cases):
    torch = torch_cuda
    devs = [tl.device_case(c) for c in cases]
    with HcGatedResidual(max_M=32) as op:
        plain = _run_sequence(op, devs, False, torch)
        stream = torch.cuda.Stream()
        outs = [{k: torch.empty_like(v) for k, v in p.items()} for p in plain]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for d, o in zip(devs, outs):
                op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           force_path=PATH_DECODE, pdl=True, out=o)
        for rep in range(3):
            for o in outs:
                for v in o.values():
                    v.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            op.check()
            for c, o, ref_o in zip(cases, outs, plain):
                for k in o:
                    assert torch.equal(o[k], ref_o[k]), (rep, c["M"], k)
        np.testing.assert_array_equal(tl.to_f64(outs[0]["R2"]), tl.to_f64(plain[0]["R2"]))
