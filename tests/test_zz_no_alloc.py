"""hc_gr_forward_noalloc, the entry point that allocates no device memory.

Some callers may not call cudaMalloc on their call path: an engine whose
memory manager owns all device memory, or code that must not risk an
allocation's implicit device synchronisation.  This entry point keeps its
scratch in a fixed device array inside the library instead.  The tests call
it through the C ABI twice in a row with two token counts, with a caller
lora buffer and with lora = NULL (lora then lives in the shared array), and
check each result against the fp64 oracle and against the handle-based
hc_gr_forward on the same inputs, with the tolerances the parity tests use;
the status query reports no device-side failure.  The file is collected
last, and passes both alone and after the other tests.
"""
import ctypes

import pytest

from hyper_connection_gated_gb300 import HcGatedResidual, _native

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu

HC, HS, R_LOW = 4, 2560, 320


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def _outputs(torch, M, lora=True):
    out = {"R2": torch.empty((M, HC, HS), dtype=torch.bfloat16, device="cuda"),
           "rrms": torch.empty((M, HC), device="cuda"),
           "inj_next": torch.empty((M, HC), device="cuda"),
           "x": torch.empty((M, HS), dtype=torch.bfloat16, device="cuda")}
    if lora:
        out["lora"] = torch.empty((M, R_LOW), device="cuda")
    return out


def _noalloc(lib, stream, M, a, out):
    lora = out["lora"].data_ptr() if "lora" in out else None
    return lib.hc_gr_forward_noalloc(
        M, HC, HS, R_LOW, ctypes.c_float(1e-6), a["R"].data_ptr(), a["y"].data_ptr(),
        a["inj"].data_ptr(), a["Wnorm"].data_ptr(), a["Wd"].data_ptr(), a["Wi"].data_ptr(),
        a["Wu"].data_ptr(), out["R2"].data_ptr(), out["rrms"].data_ptr(),
        out["inj_next"].data_ptr(), out["x"].data_ptr(), lora, ctypes.c_void_p(stream.cuda_stream))


def test_noalloc_matches_oracle_and_forward_on_two_calls(torch_cuda):
    torch = torch_cuda
    lib = _native.lib()
    case = tl.make_case(8)
    d = tl.device_case(case)
    stream = torch.cuda.current_stream()
    with HcGatedResidual(max_M=8) as op:
        # two calls in a row with a caller lora, then two with lora = NULL,
        # then the smallest token counts, all sharing the one scratch array
        for M, with_lora in ((4, True), (8, True), (8, False), (3, False), (1, True), (2, False)):
            a = {k: v[:M] if k in ("R", "y", "inj") else v for k, v in d.items()}
            sub = dict(case, R=case["R"][:M], y=case["y"][:M], inj=case["inj"][:M], M=M)
            fwd = op.forward(a["R"], a["y"], a["inj"], a["Wnorm"], a["Wu"], Wd=a["Wd"], Wi=a["Wi"],
                             want_lora=with_lora, check=True)
            out = _outputs(torch, M, lora=with_lora)
            st = _noalloc(lib, stream, M, a, out)
            assert st == _native.OK, _native.strerror(st)
            assert lib.hc_gr_noalloc_check(ctypes.c_void_p(stream.cuda_stream)) == _native.OK
            tl.assert_parity(out, tl.oracle_ref(sub), label=f"noalloc M={M} lora={with_lora}")
            rep = tl.parity_report(out, {k: tl.to_f64(v) for k, v in fwd.items()})
            assert all(v <= 1.0 for v in rep.values()), (M, with_lora, rep)


def test_noalloc_rejects_sizes_beyond_its_limit(torch_cuda):
    torch = torch_cuda
    lib = _native.lib()
    buf = torch.zeros(1 << 20, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    eps = ctypes.c_float(1e-6)
    # more than 8 tokens
    assert lib.hc_gr_forward_noalloc(9, 4, 2560, 320, eps, *([p] * 12), None) == _native.ERR_UNSUPPORTED
    # r + HC = 340 above the 336 merged rows the array is sized for
    assert lib.hc_gr_forward_noalloc(2, 4, 2560, 336, eps, *([p] * 12), None) == _native.ERR_UNSUPPORTED
    # argument errors come first and leave the status clean
    assert lib.hc_gr_forward_noalloc(0, 4, 2560, 320, eps, *([p] * 12), None) == _native.ERR_INVALID_ARG
    assert lib.hc_gr_noalloc_check(None) == _native.OK
