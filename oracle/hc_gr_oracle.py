"""fp64 CPU oracle for the Hyper-Connection gated residual (test infrastructure).

This is test infrastructure, not part of the library: only the tests, the
smoke check and the benchmark's CPU-baseline leg may import it.  The CUDA
path never calls it and shares no code with it.

Source of every formula: aiter PR #5913, "Two-stage Hyper-Connection Gated
Residual kernel", section "Technical Details" (the bullets (COMBINE), (N),
(G1), (G2), (MIX) and (INJ)), and the two-stage split described right after
them (Kernel 1 stores R2, rrms, lora before SiLU and inj_next; Kernel 2
rebuilds xn = R2 * rrms * (1 + Wnorm)).  The merged, folded down/inject
weight is the one in that page's "Performance" setup ("Merged down/inject
weight: 336 rows with (1+w) folded in").

Readings taken where the page leaves a step open:
  * R2 is stored in bf16 and every later step (rrms, xn, the projections and
    the mix) uses the stored, rounded R2, because Kernel 2 rebuilds xn from
    the stored R2.
  * lora is the un-scaled product xn . Wd^T; the 1/HC belongs to the SiLU
    argument (the page writes both "h = SiLU(lora / HC)" and "lora
    (pre-SiLU)").
  * eps sits inside the square root, added to the mean of squares.
  * Wnorm has K entries, one per (stream, channel), or HS entries shared by
    every stream (norm_weight).
  * With a folded weight W' = bf16(W * (1 + Wnorm)), the projections read
    R2 * rrms against W'; the mix still uses the full xn with (1 + Wnorm).

Everything is computed in float64; inputs are the exact values of the bf16 /
fp32 arrays the GPU receives.  Shapes (M tokens):
  R [M, HC, HS], y [M, HS], inj [M, HC], Wnorm [K], Wd [r, K], Wi [HC, K],
  Wu [K, r], K = HC * HS.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16, ties to even.

    bfloat16 keeps 8 significant bits and float32's exponent range; values
    below 2**-126 are quantised to multiples of 2**-133 (subnormals) and
    values that round past the largest finite bfloat16 become infinite.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                          # x = m * 2**e, 0.5 <= |m| < 1
    with np.errstate(invalid="ignore", over="ignore"):
        out = np.ldexp(np.rint(m * 256.0) / 256.0, e)
        small = np.abs(x) < 2.0 ** -126
        if np.any(small):
            out = np.where(small, np.rint(x * 2.0 ** 133) * 2.0 ** -133, out)
        big = np.isfinite(x) & (np.abs(out) > BF16_MAX)
        if np.any(big):
            out = np.where(big, np.copysign(np.inf, x), out)
    return out


def sigmoid(x) -> np.ndarray:
    """Logistic function 1 / (1 + exp(-x)), exact limits at +-inf."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def combine(R, y, inj):
    """(COMBINE) depth re-injection.

    iw = 2 * sigmoid(inj / HC) per stream, R2[s, c] = R[s, c] + y[c] * iw[s].
    Returns (R2 rounded to bf16 -- the stored next residual --, R2 unrounded).
    """
    HC = R.shape[1]
    iw = 2.0 * sigmoid(np.asarray(inj, np.float64) / HC)        # [M, HC]
    r2 = R + y[:, None, :] * iw[:, :, None]                      # [M, HC, HS]
    return bf16_round(r2), r2


def grouped_rrms(R2, eps):
    """(N) reciprocal RMS per stream: rsqrt(mean_c R2[s, c]^2 + eps)."""
    ms = np.mean(R2 * R2, axis=2)                                # [M, HC]
    return 1.0 / np.sqrt(ms + eps)


def norm_weight(Wnorm, HC, HS):
    """The norm weight as [HC, HS]: a full-width weight has K = HC * HS
    entries, one per (stream, channel); an [HS] weight is one per channel,
    shared by every stream (the page's default next to its "full-width norm
    weights" variant)."""
    w = np.asarray(Wnorm, np.float64).reshape(-1)
    if w.size == HC * HS:
        return w.reshape(HC, HS)
    if w.size == HS:
        return np.broadcast_to(w[None, :], (HC, HS))
    raise ValueError("Wnorm must have HC * HS or HS entries")


def normalise(R2, rrms, Wnorm):
    """(N) xn[s, c] = R2[s, c] * rrms_s * (1 + Wnorm[s, c]), flattened to K."""
    M, HC, HS = R2.shape
    w = norm_weight(Wnorm, HC, HS)
    xn = R2 * rrms[:, :, None] * (1.0 + w)[None]
    return xn.reshape(M, HC * HS)


def project(xrow, W):
    """Row-vector times transposed weight: out[m, n] = sum_k x[m, k] W[n, k]."""
    return xrow @ np.asarray(W, np.float64).T


def silu_h(lora, HC):
    """(G1) h = SiLU(lora / HC) with SiLU(u) = u * sigmoid(u)."""
    u = lora / HC
    return u * sigmoid(u)


def up_gate(h, Wu):
    """(G2) G = sigmoid(h . Wu^T); Wu is [K, r] so G is [M, K]."""
    return sigmoid(project(h, Wu))


def gated_mean(G, xn, HC):
    """(MIX) x[c] = (1/HC) * sum_s G[s, c] * xn[s, c]."""
    M, K = xn.shape
    HS = K // HC
    return (G * xn).reshape(M, HC, HS).sum(axis=1) / HC


def split_merged(Wdi, r, HC):
    """Rows 0..r-1 of a merged [n_pad, K] weight are Wd, rows r..r+HC-1 Wi.

    Rows r+HC..n_pad-1 are padding and never read.
    """
    Wdi = np.asarray(Wdi, np.float64)
    return Wdi[:r], Wdi[r:r + HC]


def merge_weight(Wd, Wi, Wnorm, n_pad, fold):
    """Merged down/inject weight [n_pad, K] in float64 (not yet rounded).

    With fold=True each column k carries the factor (1 + Wnorm[k]), the
    "(1+w) folded in" layout of the page's benchmark setup.  Padding rows
    are zero.
    """
    Wd = np.asarray(Wd, np.float64)
    Wi = np.asarray(Wi, np.float64)
    r, K = Wd.shape
    HC = Wi.shape[0]
    if n_pad < r + HC:
        raise ValueError("n_pad must hold r + HC rows")
    W = np.zeros((n_pad, K), dtype=np.float64)
    W[:r] = Wd
    W[r:r + HC] = Wi
    if fold:
        W[:r + HC] *= (1.0 + norm_weight(Wnorm, HC, K // HC).reshape(K))[None, :]
    return W


def forward(R, y, inj, Wnorm, Wu, eps, Wd=None, Wi=None, Wdi=None,
            fold_w=False):
    """The whole per-token path, in the page's order: (COMBINE), then the
    mix of the combined residual.

    Either (Wd, Wi) or a merged Wdi is given.  With fold_w the given
    projection weights already carry (1 + Wnorm) in their columns.
    Returns a dict with R2 (bf16-rounded), rrms, xn, lora, inj_next, h, G, x.
    """
    R = np.asarray(R, np.float64)
    y = np.asarray(y, np.float64)
    R2, _ = combine(R, y, inj)
    out = mix(R2, Wnorm, Wu, eps, Wd=Wd, Wi=Wi, Wdi=Wdi, fold_w=fold_w)
    out["R2"] = R2
    return out


def mix(R2, Wnorm, Wu, eps, Wd=None, Wi=None, Wdi=None, fold_w=False):
    """Every step after (COMBINE) -- (N), (G1), (INJ), (G2), (MIX) -- on an
    already-combined residual R2 [M, HC, HS] (the page's mix entry point).

    Weights as in forward.  Returns rrms, xn, lora, inj_next, h, G, x.
    """
    R2 = np.asarray(R2, np.float64)
    M, HC, HS = R2.shape
    r = np.asarray(Wu).shape[1]
    if Wdi is not None:
        Wd, Wi = split_merged(Wdi, r, HC)
    rrms = grouped_rrms(R2, eps)
    xn = normalise(R2, rrms, Wnorm)
    if fold_w:
        xp = (R2 * rrms[:, :, None]).reshape(M, HC * HS)
    else:
        xp = xn
    lora = project(xp, Wd)
    inj_next = project(xp, Wi)
    h = silu_h(lora, HC)
    G = up_gate(h, Wu)
    x = gated_mean(G, xn, HC)
    return {"rrms": rrms, "xn": xn, "lora": lora,
            "inj_next": inj_next, "h": h, "G": G, "x": x}
