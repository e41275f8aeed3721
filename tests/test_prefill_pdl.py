"""Prefill kernels chained by programmatic dependent launch
(hc_gr_args.pdl = 1): K1 is a programmatic dependent of the previous kernel
in the stream, the reduce of K1 and K2 of the reduce, so each prologue may
overlap its predecessor's tail (aiter PR #5913, "Technical Details": Kernel 2
consumes what Kernel 1 writes).

A CUDA graph of two chained calls -- the second call's K1 a dependent of the
first call's K2 -- is replayed 1000 times; every replay's outputs must equal,
bit for bit, the same call made in plain stream order, which itself matches
the fp64 oracle.  Shapes: the split-K path (M = 512, K chunks per stream),
the one-chunk path (M = 4096) and the wide variant (HC = 8, HS = 4096,
r = 512), whose K1 weight ring holds two column blocks per K block.  The
same replays in plain stream order (pdl = 0) guard K2's R2 ring: its slots
are read with ordinary loads and refilled by TMA, a write-after-read across
memory proxies that once corrupted one warp's x in a few percent of calls at
the wide shape.
"""
import pytest

from hyper_connection_gated_gb300 import PATH_PREFILL, HcGatedResidual, inputs

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu

REPLAYS = 1000


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.mark.parametrize("pdl", [True, False], ids=["pdl", "plain"])
@pytest.mark.parametrize("M,shape", [(512, inputs.DEFAULT), (4096, inputs.DEFAULT), (1024, inputs.WIDE)],
                         ids=["M512", "M4096", "wide_M1024"])
def test_prefill_graph_replays_bit_identical(torch_cuda, M, shape, pdl):
    torch = torch_cuda
    case = tl.make_case(M, shape, seed=61)
    d = tl.device_case(case)
    with HcGatedResidual(max_M=M, HC=shape.HC, HS=shape.HS, r=shape.r) as op:
        def call(out=None, pdl=False):
            return op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                              force_path=PATH_PREFILL, pdl=pdl, out=out)
        plain = call()
        op.check()
        tl.assert_parity(plain, tl.oracle_ref(case), label=f"plain prefill M={M}")
        outs = [{k: torch.empty_like(v) for k, v in plain.items()} for _ in range(2)]
        stream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for o in outs:
                call(out=o, pdl=pdl)
        torch.cuda.synchronize()
        mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
        with torch.cuda.stream(stream):
            for _ in range(REPLAYS):
                for o in outs:
                    for v in o.values():
                        v.fill_(float("nan"))
                graph.replay()
                for o in outs:
                    for k, v in o.items():
                        mismatches += (v.view(torch.int16) != plain[k].view(torch.int16)).any().long() \
                            if v.dtype == torch.bfloat16 else (v != plain[k]).any().long()
        torch.cuda.synchronize()
        op.check()
        assert int(mismatches.item()) == 0, f"{int(mismatches.item())} output tensors differed over {REPLAYS} replays"
