"""Shared test helpers: seeded cases, device upload, oracle reference, tolerances.

Tolerances (the GPU result against the fp64 oracle on the same inputs):
  * bf16 outputs R2 and x:       |g - o| <= 1e-2 * (1 + |o|), element-wise;
  * fp32 rrms:                   |g - o| <= 2e-3 * |o|, element-wise;
  * fp32 lora and inj_next:      |g - o| <= 2e-3 * max(|o|, rms of o over the
    token's row) -- "2e-3 relative" taken relative to the row's scale, since
    single elements of a dot product can sit arbitrarily close to zero.
"""
from __future__ import annotations

import contextlib
import multiprocessing
import os

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


def _ratios(g: dict, ref: dict) -> dict:
    """Worst error / bound ratio per output; g holds float64 arrays whose first
    axis matches ref's rows."""
    rep = {}
    M = ref["rrms"].shape[0] if "rrms" in ref else ref["R2"].shape[0]
    for k in ("R2", "x"):
        if k not in g or k not in ref:      # the mix alone produces no R2
            continue
        gk = g[k].reshape(M, -1)
        o = ref[k].reshape(M, -1)
        rep[k] = float(np.max(np.abs(gk - o) / (TOL_BF16 * (1.0 + np.abs(o)))))
    if "rrms" in g and "rrms" in ref:
        rep["rrms"] = float(np.max(np.abs(g["rrms"] - ref["rrms"]) / (TOL_F32 * np.abs(ref["rrms"]))))
    for k in ("lora", "inj_next"):
        if g.get(k) is None or k not in ref:
            continue
        o = ref[k]
        scale = np.maximum(np.abs(o), np.sqrt(np.mean(o * o, axis=1, keepdims=True)))
        # an all-zero reference row (a zero token) leaves no scale: only an
        # exact zero passes there
        scale = np.maximum(scale, np.finfo(np.float64).tiny)
        rep[k] = float(np.max(np.abs(g[k] - o) / (TOL_F32 * scale)))
    for k, v in g.items():
        if v is not None and not np.all(np.isfinite(v)):
            rep[k + "_finite"] = float("inf")
    return rep


def parity_report(got: dict, ref: dict, rows=None) -> dict:
    """Worst error / bound ratio per output (<= 1 passes)."""
    sel = slice(None) if rows is None else np.asarray(rows)
    g = {k: to_f64(v)[sel] for k, v in got.items() if v is not None}
    return _ratios(g, ref)


def assert_parity(got: dict, ref: dict, rows=None, label: str = "") -> dict:
    rep = parity_report(got, ref, rows)
    bad = {k: v for k, v in rep.items() if not v <= 1.0}
    assert not bad, f"{label}: outputs outside tolerance (error/bound): {rep}"
    return rep


# ------------------------------------------------------------ every row, pooled
# Large cases are checked on every row.  The rows are cut into chunks; a pool
# of single-threaded worker processes, started with "spawn" (so no CUDA state
# is inherited), draws each chunk's inputs from the seed again, runs the
# oracle on those rows and compares them with the GPU's rows.

_WORKER_CACHE: dict = {}


def _worker_weights(shape, seed, merged):
    """Weights (float64) of one case, kept per worker; merged = (n_pad, fold)
    adds the merged weight the caller would build."""
    key = (shape, seed, merged)
    if key not in _WORKER_CACHE:
        _WORKER_CACHE.clear()
        w = {k: inputs.bf16_bits_to_f64(v) for k, v in inputs.weights(shape, seed).items()}
        if merged is not None:
            n_pad, fold = merged
            w["Wdi"] = inputs.bf16_bits_to_f64(inputs.to_bf16_bits(
                oracle.merge_weight(w["Wd"], w["Wi"], w["Wnorm"], n_pad, fold)))
        _WORKER_CACHE[key] = w
    return _WORKER_CACHE[key]


def _gen_task(args):
    start, stop, shape, seed = args
    return start, inputs.activation_rows(start, stop, shape, seed)


def _check_task(args):
    """One chunk: the oracle on rows start..stop-1 against the GPU's rows."""
    start, stop, shape, seed, kind, merged, got = args
    w = _worker_weights(shape, seed, merged)
    a = inputs.activation_rows(start, stop, shape, seed)
    R = inputs.bf16_bits_to_f64(a["R"])
    if kind == "combine":
        ref = {"R2": oracle.combine(R, inputs.bf16_bits_to_f64(a["y"]),
                                    a["inj"].astype(np.float64))[0]}
    else:
        kw = dict(Wnorm=w["Wnorm"], Wu=w["Wu"], eps=shape.eps)
        if merged is not None:
            kw.update(Wdi=w["Wdi"], fold_w=merged[1])
        else:
            kw.update(Wd=w["Wd"], Wi=w["Wi"])
        if kind == "mix":
            ref = oracle.mix(R, **kw)
        else:
            ref = oracle.forward(R=R, y=inputs.bf16_bits_to_f64(a["y"]),
                                 inj=a["inj"].astype(np.float64), **kw)
    g = {k: (inputs.bf16_bits_to_f64(v) if v.dtype == np.uint16 else v.astype(np.float64))
         for k, v in got.items()}
    return start, _ratios(g, ref)


def chunk_rows(M: int, shape) -> int:
    """Rows per pooled task: about four million elements of R."""
    return max(16, (1 << 22) // shape.K)


@contextlib.contextmanager
def oracle_pool(workers: int | None = None):
    """A spawn-started pool of single-threaded (one BLAS thread) workers."""
    n = workers or (len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                    else os.cpu_count())
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        pool = multiprocessing.get_context("spawn").Pool(max(1, n))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield pool
    finally:
        pool.terminate()
        pool.join()


def pooled_activations(pool, M: int, shape=inputs.DEFAULT, seed: int = inputs.SEED,
                       step: int | None = None) -> dict:
    """activations(M) drawn chunk by chunk in the pool (identical values)."""
    step = step or chunk_rows(M, shape)
    tasks = [(s, min(M, s + step), shape, seed) for s in range(0, M, step)]
    out = {"R": np.empty((M, shape.HC, shape.HS), np.uint16),
           "y": np.empty((M, shape.HS), np.uint16), "inj": np.empty((M, shape.HC), np.float32)}
    for start, a in pool.imap_unordered(_gen_task, tasks):
        for k, v in a.items():
            out[k][start:start + v.shape[0]] = v
    return out


def host_outputs(got: dict) -> dict:
    """GPU outputs as numpy: bf16 tensors as uint16 bits, fp32 as float32."""
    import torch

    out = {}
    for k, v in got.items():
        if v is None:
            continue
        v = v.detach().contiguous()
        out[k] = (v.view(torch.int16).cpu().numpy().view(np.uint16) if v.dtype == torch.bfloat16
                  else v.cpu().numpy())
    return out


def pooled_parity(pool, got: dict, M: int, shape=inputs.DEFAULT, seed: int = inputs.SEED,
                  kind: str = "forward", merged=None, step: int | None = None) -> dict:
    """Every row of a GPU result (host_outputs form) against the oracle, in
    the pool.  kind: "forward", "mix" or "combine"; merged = (n_pad, fold)
    for a merged weight.  Returns the worst ratio per output over all rows
    and, per output, the start row of the chunk where it is worst."""
    step = step or chunk_rows(M, shape)
    tasks = [(s, min(M, s + step), shape, seed, kind, merged,
              {k: v[s:min(M, s + step)] for k, v in got.items()}) for s in range(0, M, step)]
    worst, where = {}, {}
    for start, rep in pool.imap_unordered(_check_task, tasks):
        for k, v in rep.items():
            if k not in worst or not v <= worst[k]:
                worst[k], where[k] = v, start
    return {"worst": worst, "chunk_start": where, "rows": M}


def assert_pooled_parity(pool, got: dict, M: int, label: str = "", **kw) -> dict:
    rep = pooled_parity(pool, got, M, **kw)
    bad = {k: v for k, v in rep["worst"].items() if not v <= 1.0}
    assert not bad, f"{label}: outputs outside tolerance (error/bound) over all {M} rows: {rep}"
    return rep
