"""The C ABI's error contract on a GPU: rejected arguments, aliasing, bounded
waits that expire, and a handle that stays usable afterwards."""
import ctypes

import pytest

from hyper_connection_gated_gb300 import (ERR_ALIAS, ERR_CUDA, ERR_INVALID_ARG, ERR_TIMEOUT,
                                          ERR_UNSUPPORTED, OK, PATH_DECODE, HcGatedResidual,
                                          HcGrError, _native, inputs)

from . import hcgr_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    shape = inputs.Shape(HC=4, HS=256, r=32)
    case = tl.make_case(4, shape, seed=3)
    d = tl.device_case(case)
    op = HcGatedResidual(max_M=8, HC=4, HS=256, r=32)
    yield torch, case, d, op
    op.close()


def _args(torch, d, M=4, HC=4, HS=256, r=32):
    out = {"R2": torch.empty_like(d["R"]), "rrms": torch.empty((M, HC), device="cuda"),
           "inj_next": torch.empty((M, HC), device="cuda"),
           "x": torch.empty((M, HS), dtype=torch.bfloat16, device="cuda"),
           "lora": torch.empty((M, r), device="cuda")}
    a = _native.Args()
    a.M, a.HC, a.HS, a.r, a.eps = M, HC, HS, r, 1e-6
    a.R, a.y, a.inj = d["R"].data_ptr(), d["y"].data_ptr(), d["inj"].data_ptr()
    a.Wnorm, a.Wd, a.Wi, a.Wu = (d["Wnorm"].data_ptr(), d["Wd"].data_ptr(), d["Wi"].data_ptr(),
                                 d["Wu"].data_ptr())
    a.R2, a.rrms, a.inj_next = out["R2"].data_ptr(), out["rrms"].data_ptr(), out["inj_next"].data_ptr()
    a.x, a.lora = out["x"].data_ptr(), out["lora"].data_ptr()
    return a, out


def _run(op, torch, a):
    return op.forward_raw(a, torch.cuda.current_stream().cuda_stream)


def test_valid_call_passes(env):
    torch, case, d, op = env
    a, out = _args(torch, d)
    assert _run(op, torch, a) == OK
    assert op.check_status(torch.cuda.current_stream().cuda_stream) == OK
    tl.assert_parity(out, tl.oracle_ref(case))


@pytest.mark.parametrize("field,value,status", [
    ("M", 0, ERR_INVALID_ARG), ("M", 9, ERR_UNSUPPORTED), ("eps", 0.0, ERR_INVALID_ARG),
    ("eps", float("nan"), ERR_INVALID_ARG), ("HS", 250, ERR_UNSUPPORTED),
    ("HC", 5, ERR_UNSUPPORTED), ("r", 40, ERR_UNSUPPORTED), ("R", None, ERR_INVALID_ARG),
    ("Wu", None, ERR_INVALID_ARG), ("x", None, ERR_INVALID_ARG), ("ld_inj", 3, ERR_INVALID_ARG),
    ("force_path", 7, ERR_INVALID_ARG),
])
def test_rejected_arguments(env, field, value, status):
    torch, case, d, op = env
    a, out = _args(torch, d)
    setattr(a, field, value)
    before = out["x"].clone()
    assert _run(op, torch, a) == status
    torch.cuda.synchronize()
    assert torch.equal(out["x"], before)     # nothing was launched


def test_misaligned_pointer(env):
    torch, case, d, op = env
    a, _ = _args(torch, d)
    a.R = d["R"].data_ptr() + 2
    assert _run(op, torch, a) == ERR_INVALID_ARG


def test_merged_weight_too_few_rows(env):
    torch, case, d, op = env
    a, _ = _args(torch, d)
    a.Wdi, a.n_pad = d["Wd"].data_ptr(), 35
    assert _run(op, torch, a) == ERR_UNSUPPORTED


@pytest.mark.parametrize("pair", [("x", "R2"), ("rrms", "inj_next"), ("R2", "R"), ("x", "y"),
                                  ("lora", "Wu"), ("inj_next", "inj"), ("x", "Wnorm")])
def test_aliasing_rejected(env, pair):
    torch, case, d, op = env
    a, _ = _args(torch, d)
    setattr(a, pair[0], getattr(a, pair[1]))
    assert _run(op, torch, a) == ERR_ALIAS


def test_partial_overlap_rejected(env):
    torch, case, d, op = env
    a, out = _args(torch, d)
    a.x = out["R2"].data_ptr() + (out["R2"].numel() * 2 - 16)   # last 16 bytes of R2
    assert _run(op, torch, a) == ERR_ALIAS


def test_python_side_dtype_checks(env):
    torch, case, d, op = env
    with pytest.raises(HcGrError):
        op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"].float(), Wd=d["Wd"], Wi=d["Wi"])
    with pytest.raises(HcGrError):
        op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"].t().contiguous().t(),
                   Wd=d["Wd"], Wi=d["Wi"])


def test_barrier_timeout_reported_and_recovered(env):
    # One CTA of the decode kernel leaves before the first grid barrier; the
    # others' bounded wait expires, the kernel returns, hc_gr_check reports
    # TIMEOUT, and the next call on the same handle is correct again.
    torch, case, d, op = env
    a, _ = _args(torch, d)
    a.force_path, a.debug_fault = PATH_DECODE, 1
    assert _run(op, torch, a) == OK
    assert op.check_status(torch.cuda.current_stream().cuda_stream) == ERR_TIMEOUT
    assert op.check_status(torch.cuda.current_stream().cuda_stream) == OK
    a2, out = _args(torch, d)
    assert _run(op, torch, a2) == OK
    assert op.check_status(torch.cuda.current_stream().cuda_stream) == OK
    tl.assert_parity(out, tl.oracle_ref(case))


def test_handle_shape_change_between_calls(env):
    # One handle, calls with different HC (same K): the barrier phase and the
    # workspace cannot leak from one call into the next.
    torch, case, d, op = env
    s2 = inputs.Shape(HC=8, HS=128, r=24)
    c2 = tl.make_case(3, s2, seed=9)
    d2 = tl.device_case(c2)
    for _ in range(2):
        o1 = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                        check=True)
        tl.assert_parity(o1, tl.oracle_ref(case))
        o2 = op.forward(d2["R"], d2["y"], d2["inj"], d2["Wnorm"], d2["Wu"], Wd=d2["Wd"],
                        Wi=d2["Wi"], check=True)
        tl.assert_parity(o2, tl.oracle_ref(c2))


def test_lora_optional(env):
    torch, case, d, op = env
    out = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                     want_lora=False, check=True)
    assert "lora" not in out
    tl.assert_parity(out, tl.oracle_ref(case))


def test_prepared_call_repeats_bit_identically(env):
    # prepare() validates once; launch() reruns the same call on the same
    # buffers, and every run gives the result forward() gives
    torch, case, d, op = env
    ref = op.forward(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                     check=True)
    args, out = op.prepare(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"],
                           pdl=True)
    h = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        for t in out.values():
            t.fill_(float("nan"))
        op.launch(args, h)
        op.check()
        for k in ref:
            assert torch.equal(out[k].view(torch.uint8), ref[k].view(torch.uint8)), k
    tl.assert_parity(out, tl.oracle_ref(case))


def test_prepared_call_rejects_like_forward(env):
    torch, case, d, op = env
    args, _ = op.prepare(d["R"], d["y"], d["inj"], d["Wnorm"], d["Wu"], Wd=d["Wd"], Wi=d["Wi"])
    args.eps = 0.0
    with pytest.raises(HcGrError) as ei:
        op.launch(args, torch.cuda.current_stream().cuda_stream)
    assert ei.value.status == ERR_INVALID_ARG


def test_size_limits_and_allocation_failure(env):
    # Sizes above the limits are refused on the host; a handle within them
    # whose workspace cannot be allocated (max_M = 2^30 tokens needs several
    # TB) reports a CUDA error and returns no handle; nothing is launched and
    # the device stays usable.
    torch, case, d, op = env
    lib = _native.lib()
    h = ctypes.c_void_p()
    assert lib.hc_gr_create(ctypes.byref(h), 0, _native.MAX_TOKENS + 1, 4, 2560, 320) == ERR_UNSUPPORTED
    assert h.value is None
    assert lib.hc_gr_create(ctypes.byref(h), 0, 8, 2, (1 << 29) + 8, 320) == ERR_UNSUPPORTED
    assert h.value is None
    assert lib.hc_gr_create(ctypes.byref(h), 0, _native.MAX_TOKENS, 4, 2560, 320) == ERR_CUDA
    assert h.value is None
    a, out = _args(torch, d)
    a.M = _native.MAX_TOKENS + 1
    assert _run(op, torch, a) == ERR_UNSUPPORTED
    a, out = _args(torch, d)
    assert _run(op, torch, a) == OK
    assert op.check_status(torch.cuda.current_stream().cuda_stream) == OK
    tl.assert_parity(out, tl.oracle_ref(case))
    torch.zeros(4, device="cuda").sum().item()     # torch sees no stale CUDA error
