"""Hyper-Connection gated residual for one GB300 GPU.

The computation runs in the CUDA library libhc_gr.so (C ABI:
include/hc_gr.h).  This module only marshals torch tensors -- used for device
memory and streams -- into that ABI: it checks dtypes and devices, allocates
outputs when the caller does not pass them, and forwards raw pointers.

    op = HcGatedResidual(max_M=4096)           # HC=4, HS=2560, r=320
    out = op.forward(R, y, inj, Wnorm, Wu, Wd=Wd, Wi=Wi)
    out["x"], out["R2"], out["rrms"], out["inj_next"], out["lora"]

    # fixed buffers, many calls: validate once, then one C call per step
    args, out = op.prepare(R, y, inj, Wnorm, Wu, Wd=Wd, Wi=Wi, pdl=True)
    op.launch(args, torch.cuda.current_stream().cuda_stream)
"""
from __future__ import annotations

import ctypes

from . import _native
from ._native import (HcGrError, OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIAS,  # noqa: F401
                      ERR_CUDA, ERR_TIMEOUT, PATH_AUTO, PATH_DECODE, PATH_PREFILL)

__all__ = ["HcGatedResidual", "HcGrError"]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class HcGatedResidual:
    """Handle on one device with a workspace for M <= max_M tokens.

    HC, HS and r set the largest shape the handle serves (HC * HS and r + HC
    bound later calls).
    """

    def __init__(self, max_M: int, HC: int = 4, HS: int = 2560, r: int = 320, device: int = 0):
        self._lib = _native.lib()
        h = ctypes.c_void_p()
        st = self._lib.hc_gr_create(ctypes.byref(h), device, max_M, HC, HS, r)
        if st != OK:
            raise HcGrError(st, _native.strerror(st))
        self._h = h
        self.device = device
        self.max_M, self.HC, self.HS, self.r = max_M, HC, HS, r

    # ------------------------------------------------------------------ calls
    def prepare(self, R, y, inj, Wnorm, Wu, Wd=None, Wi=None, Wdi=None, fold_w=False,
                eps: float = 1e-6, out: dict | None = None, want_lora: bool = True,
                force_path: int = PATH_AUTO, debug_fault: int = 0,
                pdl: bool = False) -> tuple["_native.Args", dict]:
        """Validates one call's tensors once and returns (args, out).

        R [M, HC, HS] bf16, y [M, HS] bf16, inj [M, HC] fp32 (rows may be
        strided), Wnorm [K] bf16 (or [HS]: one norm weight per channel,
        shared by every stream), Wu [K, r] bf16, and either Wd [r, K] + Wi
        [HC, K] or a merged Wdi [n_pad, K] (fold_w: (1 + Wnorm) folded in).
        y = inj = None is the mix alone: R is the combined residual and no R2
        is produced.  out holds R2, rrms, inj_next, x (and lora); they are
        allocated here when not given.  `launch(args)` then runs the call on these buffers
        as often as needed (a serving loop with fixed buffers), with none of
        the per-call checks of `forward`; the caller keeps every tensor alive.
        pdl: let the decode kernel start its weight copies before the
        previous kernel on the stream has finished (that kernel must not
        write the weights).
        """
        import torch

        M, HC, HS = R.shape
        r = Wu.shape[1]
        dev = R.device
        mix_only = y is None and inj is None
        for name, t in (("R", R), ("y", y), ("Wnorm", Wnorm), ("Wu", Wu), ("Wd", Wd),
                        ("Wi", Wi), ("Wdi", Wdi)):
            if t is None:
                continue
            if t.dtype != torch.bfloat16 or t.device != dev or not t.is_contiguous():
                raise HcGrError(ERR_INVALID_ARG, f"{name} must be a contiguous bf16 tensor on {dev}")
        if not mix_only:
            if y is None or inj is None:
                raise HcGrError(ERR_INVALID_ARG, "y and inj are both given or both None (mix only)")
            if inj.dtype != torch.float32 or inj.device != dev or inj.stride(1) != 1:
                raise HcGrError(ERR_INVALID_ARG, "inj must be fp32 on the same device, unit column stride")
            if tuple(y.shape) != (M, HS) or tuple(inj.shape) != (M, HC):
                raise HcGrError(ERR_INVALID_ARG, "shape mismatch")
        if Wnorm.numel() not in (HC * HS, HS) or tuple(Wu.shape) != (HC * HS, r):
            raise HcGrError(ERR_INVALID_ARG, "shape mismatch")
        if out is None:
            out = {} if mix_only else {"R2": torch.empty_like(R)}
            out.update({
                "rrms": torch.empty((M, HC), dtype=torch.float32, device=dev),
                "inj_next": torch.empty((M, HC), dtype=torch.float32, device=dev),
                "x": torch.empty((M, HS), dtype=torch.bfloat16, device=dev),
            })
            if want_lora:
                out["lora"] = torch.empty((M, r), dtype=torch.float32, device=dev)
        a = _native.Args()
        a.M, a.HC, a.HS, a.r, a.eps = M, HC, HS, r, eps
        a.R = R.data_ptr()
        if not mix_only:
            a.y, a.inj = y.data_ptr(), inj.data_ptr()
            a.ld_inj = inj.stride(0) if M > 1 else HC
        a.Wnorm, a.Wu = Wnorm.data_ptr(), Wu.data_ptr()
        a.wnorm_hs = 1 if Wnorm.numel() != HC * HS else 0
        if Wdi is not None:
            a.Wdi, a.n_pad = Wdi.data_ptr(), Wdi.shape[0]
        else:
            a.Wd, a.Wi = Wd.data_ptr(), Wi.data_ptr()
        a.fold_w = 1 if fold_w else 0
        if not mix_only:
            a.R2 = out["R2"].data_ptr()
        a.rrms, a.inj_next, a.x = out["rrms"].data_ptr(), out["inj_next"].data_ptr(), out["x"].data_ptr()
        a.lora = out["lora"].data_ptr() if out.get("lora") is not None else None
        a.force_path, a.debug_fault, a.pdl = force_path, debug_fault, 1 if pdl else 0
        return a, out

    def launch(self, args: "_native.Args", stream_handle: int) -> None:
        """Runs a prepared call on a raw stream handle (`stream.cuda_stream`);
        raises on a rejected call."""
        st = self._lib.hc_gr_forward_ex(self._h, ctypes.byref(args), ctypes.c_void_p(stream_handle))
        if st != OK:
            raise HcGrError(st, self._error_text(st))

    def forward(self, R, y, inj, Wnorm, Wu, Wd=None, Wi=None, Wdi=None, fold_w=False,
                eps: float = 1e-6, out: dict | None = None, want_lora: bool = True,
                stream=None, force_path: int = PATH_AUTO, debug_fault: int = 0,
                pdl: bool = False, check: bool = False) -> dict:
        """Runs the whole forward pass; returns the output tensors (arguments
        as in `prepare`, on `stream` or the current stream)."""
        import torch

        a, out = self.prepare(R, y, inj, Wnorm, Wu, Wd=Wd, Wi=Wi, Wdi=Wdi, fold_w=fold_w, eps=eps,
                              out=out, want_lora=want_lora, force_path=force_path,
                              debug_fault=debug_fault, pdl=pdl)
        s = stream if stream is not None else torch.cuda.current_stream(R.device)
        self.launch(a, s.cuda_stream)
        if check:
            self.check(s)
        return out

    def mix(self, R, Wnorm, Wu, Wd=None, Wi=None, Wdi=None, fold_w=False, eps: float = 1e-6,
            out: dict | None = None, want_lora: bool = True, stream=None,
            force_path: int = PATH_AUTO, pdl: bool = False, check: bool = False) -> dict:
        """Every step after COMBINE on R taken as the combined residual
        (R2 = R): returns rrms, inj_next, x (and lora); no R2."""
        return self.forward(R, None, None, Wnorm, Wu, Wd=Wd, Wi=Wi, Wdi=Wdi, fold_w=fold_w,
                            eps=eps, out=out, want_lora=want_lora, stream=stream,
                            force_path=force_path, pdl=pdl, check=check)

    def combine(self, R, y, inj, out=None, stream=None):
        """COMBINE alone: returns R2 = bf16(R + y * 2 sigmoid(inj / HC)).
        inj may be a row-strided view (unit column stride)."""
        import torch

        M, HC, HS = R.shape
        dev = R.device
        for name, t in (("R", R), ("y", y)):
            if t.dtype != torch.bfloat16 or t.device != dev or not t.is_contiguous():
                raise HcGrError(ERR_INVALID_ARG, f"{name} must be a contiguous bf16 tensor on {dev}")
        if inj.dtype != torch.float32 or inj.device != dev or inj.stride(1) != 1:
            raise HcGrError(ERR_INVALID_ARG, "inj must be fp32 on the same device, unit column stride")
        if tuple(y.shape) != (M, HS) or tuple(inj.shape) != (M, HC):
            raise HcGrError(ERR_INVALID_ARG, "shape mismatch")
        if out is None:
            out = torch.empty_like(R)
        elif out.dtype != torch.bfloat16 or out.shape != R.shape or not out.is_contiguous():
            raise HcGrError(ERR_INVALID_ARG, "out must be a contiguous bf16 tensor shaped like R")
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        st = self._lib.hc_gr_combine(self._h, M, HC, HS, R.data_ptr(), y.data_ptr(), inj.data_ptr(),
                                     inj.stride(0) if M > 1 else HC, out.data_ptr(),
                                     ctypes.c_void_p(s.cuda_stream))
        if st != OK:
            raise HcGrError(st, self._error_text(st))
        return out

    def forward_raw(self, args: "_native.Args", stream_handle: int) -> int:
        """hc_gr_forward_ex on a prepared argument struct; returns the status."""
        return self._lib.hc_gr_forward_ex(self._h, ctypes.byref(args), ctypes.c_void_p(stream_handle))

    def check(self, stream=None) -> None:
        """Waits for the stream and raises if a device-side wait expired."""
        import torch

        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        st = self._lib.hc_gr_check(self._h, ctypes.c_void_p(s.cuda_stream))
        if st != OK:
            raise HcGrError(st, self._error_text(st))

    def check_status(self, stream_handle: int = 0) -> int:
        return self._lib.hc_gr_check(self._h, ctypes.c_void_p(stream_handle))

    def _error_text(self, st: int) -> str:
        msg = _native.strerror(st)
        if st == ERR_CUDA:
            msg += ": " + self._lib.hc_gr_last_cuda_error(self._h).decode()
        return msg

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.hc_gr_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
