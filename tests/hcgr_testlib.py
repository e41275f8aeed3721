"""Shared test helpers: seeded cases, device upload, oracle reference, tolerances.

Tolerances (the GPU result against the fp64 oracle on the same inputs):
  * bf16 outputs R2 and x:       |g - o| <= 1e-2 * (1 + |o|), element-wise;
  * fp32 rrms:                   |g - o| <= 2e-3 * |o|, element-wise;
  * fp32 lora and inj_next:      |g - o| <= 2e-3 * max(|o|, rms of o over the
    token's row) -- "2e-3 relative" taken relative to the row's scale, since
    single elements of a dot product can sit arbitrarily close to zero.
"""
from __future__ import annotations

import numpy as np

import oracle
from hyper_connection_gated_gb300 import inputs

TOL_BF16 = 1e-2
TOL_F32 = 2e-3


def make_case(M: int, shape: inputs.Shape = inputs.DEFAULT, seed: int = inputs.SEED,
              distinct_rows: int | None = None) -> dict:
    w = inputs.weights(shape, seed)
    a = inputs.activations(M, shape, seed, distinct_rows)
    return {"shape": shape, "M": M, **w, **a}


def f64(case: dict, name: str) -> np.ndarray:
    v = case[name]
    if v.dtype == np.uint16:
        return inputs.bf16_bits_to_f64(v)
    return v.astype(np.float64)


def merged_weight_bits(case: dict, n_pad: int, fold: bool) -> np.ndarray:
    """The caller-side merged [n_pad, K] bf16 weight (optionally folded)."""
    W = oracle.merge_weight(f64(case, "Wd"), f64(case, "Wi"), f64(case, "Wnorm"), n_pad, fold)
    return inputs.to_bf16_bits(W)


def to_dev(bits_or_f32: np.ndarray, device="cuda"):
    import torch

    if bits_or_f32.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(bits_or_f32).view(np.int16))
        return t.to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(bits_or_f32)).to(device)


def device_case(case: dict, device="cuda") -> dict:
    return {k: to_dev(case[k], device) for k in ("R", "y", "inj", "Wnorm", "Wd", "Wi", "Wu")}


def oracle_ref(case: dict, rows=None, Wdi_bits=None, fold_w=False) -> dict:
    """fp64 oracle outputs for the given rows (all rows by default)."""
    sel = slice(None) if rows is None else np.asarray(rows)
    kw = dict(R=f64(case, "R")[sel], y=f64(case, "y")[sel], inj=f64(case, "inj")[sel],
              Wnorm=f64(case, "Wnorm"), Wu=f64(case, "Wu"), eps=case["shape"].eps)
    if Wdi_bits is not None:
        kw["Wdi"] = inputs.bf16_bits_to_f64(Wdi_bits)
        kw["fold_w"] = fold_w
    else:
        kw["Wd"], kw["Wi"] = f64(case, "Wd"), f64(case, "Wi")
    return oracle.forward(**kw)


def oracle_mix_ref(case: dict, rows=None, Wdi_bits=None, fold_w=False) -> dict:
    """fp64 oracle of the mix alone, with the case's R as the combined residual."""
    sel = slice(None) if rows is None else np.asarray(rows)
    kw = dict(Wnorm=f64(case, "Wnorm"), Wu=f64(case, "Wu"), eps=case["shape"].eps)
    if Wdi_bits is not None:
        kw["Wdi"] = inputs.bf16_bits_to_f64(Wdi_bits)
        kw["fold_w"] = fold_w
    else:
        kw["Wd"], kw["Wi"] = f64(case, "Wd"), f64(case, "Wi")
    return oracle.mix(inputs.bf16_bits_to_f64(case["R"][sel]), **kw)


def to_f64(t) -> np.ndarray:
    import torch

    return t.detach().to(torch.float64).cpu().numpy()


def parity_report(got: dict, ref: dict, rows=None) -> dict:
    """Worst error / bound ratio per output (<= 1 passes)."""
    sel = slice(None) if rows is None else np.asarray(rows)
    rep = {}
    M = ref["x"].shape[0]
    for k in ("R2", "x"):
        if k not in got or k not in ref:      # the mix alone produces no R2
            continue
        g = to_f64(got[k])[sel].reshape(M, -1)
        o = ref[k].reshape(M, -1)
        rep[k] = float(np.max(np.abs(g - o) / (TOL_BF16 * (1.0 + np.abs(o)))))
    g = to_f64(got["rrms"])[sel]
    rep["rrms"] = float(np.max(np.abs(g - ref["rrms"]) / (TOL_F32 * np.abs(ref["rrms"]))))
    for k in ("lora", "inj_next"):
        if got.get(k) is None:
            continue
        g = to_f64(got[k])[sel]
        o = ref[k]
        scale = np.maximum(np.abs(o), np.sqrt(np.mean(o * o, axis=1, keepdims=True)))
        # an all-zero reference row (a zero token) leaves no scale: only an
        # exact zero passes there
        scale = np.maximum(scale, np.finfo(np.float64).tiny)
        rep[k] = float(np.max(np.abs(g - o) / (TOL_F32 * scale)))
    for k in got:
        if got[k] is not None and not np.all(np.isfinite(to_f64(got[k])[sel])):
            rep[k + "_finite"] = float("inf")
    return rep


def assert_parity(got: dict, ref: dict, rows=None, label: str = "") -> dict:
    rep = parity_report(got, ref, rows)
    bad = {k: v for k, v in rep.items() if not v <= 1.0}
    assert not bad, f"{label}: outputs outside tolerance (error/bound): {rep}"
    return rep
