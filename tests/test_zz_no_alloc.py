"""hc_gr_forward_noalloc, the entry point that allocates no device memory.

Some callers may not call cudaMalloc on their call path (an engine whose
memory manager owns all device memory, or code that must not risk an
allocation's implicit device synchronisation); this entry point keeps its
scratch in a fixed device array inside the library instead.  The test calls
it through the C ABI twice in a row, with two different token counts, and
checks each result against the handle-based hc_gr_forward on the same inputs
with the tolerances the parity tests use.  It lives in its own file, collected
last, and passes both alone and after the other tests.
"""
import ctypes

import pytest

from hyper_connection_gated_gb300 import HcGatedResidual, _native

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu


def _outputs(torch, M, HC, HS, r):
    return {"R2": torch.empty((M, HC, HS), dtype=torch.bfloat16, device="cuda"),
            "rrms": torch.empty((M, HC), device="cuda"),
            "inj_next": torch.empty((M, HC), device="cuda"),
            "x": torch.empty((M, HS), dtype=torch.bfloat16, device="cuda"),
            "lora": torch.empty((M, r), device="cuda")}


def test_noalloc_matches_forward_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _native.lib()
    case = tl.make_case(8)
    d = tl.device_case(case)
    HC, HS, r = 4, 2560, 320
    stream = torch.cuda.current_stream()
    with HcGatedResidual(max_M=8) as op:
        for M in (4, 8):      # two calls in a row, sharing the one scratch array
            args = {k: v[:M] if k in ("R", "y", "inj") else v for k, v in d.items()}
            ref = op.forward(args["R"], args["y"], args["inj"], args["Wnorm"], args["Wu"],
                             Wd=args["Wd"], Wi=args["Wi"], check=True)
            out = _outputs(torch, M, HC, HS, r)
            st = lib.hc_gr_forward_noalloc(
                M, HC, HS, r, ctypes.c_float(1e-6), args["R"].data_ptr(), args["y"].data_ptr(),
                args["inj"].data_ptr(), args["Wnorm"].data_ptr(), args["Wd"].data_ptr(),
                args["Wi"].data_ptr(), args["Wu"].data_ptr(), out["R2"].data_ptr(),
                out["rrms"].data_ptr(), out["inj_next"].data_ptr(), out["x"].data_ptr(),
                out["lora"].data_ptr(), ctypes.c_void_p(stream.cuda_stream))
            assert st == _native.OK, _native.strerror(st)
            torch.cuda.synchronize()
            rep = tl.parity_report(out, {k: tl.to_f64(v) for k, v in ref.items()})
            assert all(v <= 1.0 for v in rep.values()), (M, rep)


def test_noalloc_rejects_sizes_beyond_its_limit():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _native.lib()
    buf = torch.zeros(1 << 20, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    st = lib.hc_gr_forward_noalloc(9, 4, 2560, 320, ctypes.c_float(1e-6), *([p] * 12), None)
    assert st == _native.ERR_UNSUPPORTED
