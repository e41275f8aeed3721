"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes one step of the method (aiter PR #5913, "Technical Details":
(COMBINE), (N), (G1), (INJ), (G2), (MIX)) by a closed form, a library routine
that computes the same textbook function, an invariant of the definition, or
pure-Python brute force on tiny shapes.  The set is chosen so that a dropped
term, a wrong sign or scale, a transposed operand or a stream-index mix-up in
the oracle fails at least one test.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from hyper_connection_gated_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(rng, *shape, scale=1.0):
    return oracle.bf16_round(scale * rng.standard_normal(shape))


def _case(rng, M, HC, HS, r, wn_scale=0.1):
    K = HC * HS
    return dict(
        R=_rand(rng, M, HC, HS), y=_rand(rng, M, HS),
        inj=(2.0 * rng.standard_normal((M, HC))).astype(np.float32).astype(np.float64),
        Wnorm=_rand(rng, K, scale=wn_scale), Wd=_rand(rng, r, K, scale=K ** -0.5),
        Wi=_rand(rng, HC, K, scale=K ** -0.5), Wu=_rand(rng, K, r, scale=r ** -0.5),
        eps=1e-6)


# ----------------------------------------------------------------- bf16 rounding
def test_bf16_round_hand_values():
    u = 2.0 ** -7                      # bf16 spacing just above 1.0
    cases = {
        1.0 + u / 2: 1.0,              # tie -> even (mantissa 0)
        1.0 + 3 * u / 2: 1.0 + 2 * u,  # tie -> even (mantissa 2)
        1.0 + u / 2 + 2.0 ** -30: 1.0 + u,   # just above the tie -> up
        -(1.0 + u / 2): -1.0,
        3.0: 3.0,
        1.5 * 2.0 ** -133: 2.0 * 2.0 ** -133,  # subnormal tie -> even
        2.0 ** 128: math.inf,
        -(2.0 - 2.0 ** -9) * 2.0 ** 127: -math.inf,   # above the overflow midpoint
        0.0: 0.0,
    }
    got = oracle.bf16_round(np.array(list(cases)))
    np.testing.assert_array_equal(got, np.array(list(cases.values())))


def test_bf16_round_matches_torch_on_float32_values():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even; float32
    # inputs are exact in float64, so one rounding happens on both sides.
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(200000) * np.exp2(rng.integers(-130, 120, 200000))).astype(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(f.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_bf16_round_matches_input_packer():
    rng = np.random.default_rng(2)
    f = rng.standard_normal(10000).astype(np.float32).astype(np.float64)
    np.testing.assert_array_equal(
        oracle.bf16_round(f), inputs.bf16_bits_to_f64(inputs.to_bf16_bits(f)))


# ----------------------------------------------------------------------- sigmoid
def test_sigmoid_closed_forms_and_library():
    s = oracle.sigmoid(np.array([0.0, math.log(3.0), -math.inf, math.inf, -1e30]))
    np.testing.assert_allclose(s, [0.5, 0.75, 0.0, 1.0, 0.0], rtol=1e-15, atol=0)
    x = np.linspace(-40, 40, 4001)
    np.testing.assert_allclose(oracle.sigmoid(x), scipy.special.expit(x), rtol=1e-13, atol=0)
    np.testing.assert_allclose(oracle.sigmoid(x) + oracle.sigmoid(-x), 1.0, rtol=1e-15)


# ----------------------------------------------------------------------- COMBINE
def test_combine_y_zero_gives_R():
    rng = np.random.default_rng(3)
    c = _case(rng, 3, 4, 16, 8)
    R2, _ = oracle.combine(c["R"], np.zeros_like(c["y"]), c["inj"])
    np.testing.assert_array_equal(R2, c["R"])


def test_combine_inj_zero_gives_R_plus_y():
    rng = np.random.default_rng(4)
    c = _case(rng, 3, 4, 16, 8)
    R2, _ = oracle.combine(c["R"], c["y"], np.zeros((3, 4)))
    np.testing.assert_array_equal(R2, oracle.bf16_round(c["R"] + c["y"][:, None, :]))


@pytest.mark.parametrize("neg", [-math.inf, -1e30])
def test_combine_inj_to_minus_infinity_drops_y(neg):
    rng = np.random.default_rng(5)
    c = _case(rng, 2, 4, 16, 8)
    R2, _ = oracle.combine(c["R"], c["y"], np.full((2, 4), neg))
    assert np.all(np.isfinite(R2))
    np.testing.assert_array_equal(R2, c["R"])


def test_combine_scale_closed_form():
    # inj = HC ln 3 -> sigmoid(ln 3) = 3/4 -> iw = 3/2; inj = +inf -> iw = 2.
    # Dyadic R and y make R + y iw exact in bf16, so the result is exact.
    HC, HS = 4, 8
    R = np.arange(HC * HS, dtype=np.float64).reshape(1, HC, HS) / 8.0
    y = np.arange(HS, dtype=np.float64).reshape(1, HS) / 4.0
    inj = np.array([[HC * math.log(3.0), math.inf, 0.0, -math.inf]])
    R2, r2 = oracle.combine(R, y, inj)
    iw = np.array([1.5, 2.0, 1.0, 0.0])
    want = R + y[:, None, :] * iw[None, :, None]
    np.testing.assert_allclose(r2, want, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(R2, want)


# ------------------------------------------------------------ N: grouped RMSNorm
def test_rrms_constant_rows_closed_form():
    a = np.array([0.5, 3.0, -2.0, 0.0])
    R2 = np.broadcast_to(a[None, :, None], (1, 4, 64)).copy()
    eps = 1e-6
    np.testing.assert_allclose(oracle.grouped_rrms(R2, eps)[0], 1.0 / np.sqrt(a * a + eps),
                               rtol=1e-15)


def test_rrms_plain_rmsnorm_matches_torch():
    # HC = 1 and Wnorm = 0 reduce the grouped norm to the textbook RMSNorm.
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, 1, 96))
    eps = 1e-3
    rrms = oracle.grouped_rrms(x, eps)
    xn = oracle.normalise(x, rrms, np.zeros(96))
    want = torch.nn.functional.rms_norm(torch.from_numpy(x[:, 0]), (96,), eps=eps).numpy()
    np.testing.assert_allclose(xn, want, rtol=1e-13, atol=1e-15)


def test_rrms_per_stream_matches_torch_groups():
    # The norm is taken per stream: a [HC, HS] row is HC independent RMSNorms,
    # each with its own slice of the K-wide Wnorm.
    rng = np.random.default_rng(7)
    HC, HS = 3, 40
    x = rng.standard_normal((4, HC, HS))
    w = rng.standard_normal(HC * HS) * 0.1
    xn = oracle.normalise(x, oracle.grouped_rrms(x, 1e-6), w).reshape(4, HC, HS)
    for s in range(HC):
        want = torch.nn.functional.rms_norm(
            torch.from_numpy(x[:, s]), (HS,), weight=torch.from_numpy(1.0 + w[s * HS:(s + 1) * HS]),
            eps=1e-6).numpy()
        np.testing.assert_allclose(xn[:, s], want, rtol=1e-13, atol=1e-15)


def test_rrms_scale_invariance():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 4, 32))
    a = oracle.grouped_rrms(x, 0.0)
    b = oracle.grouped_rrms(x * 2.0 ** 5, 0.0)
    np.testing.assert_allclose(b * 2.0 ** 5, a, rtol=1e-14)
    w = np.zeros(128)
    np.testing.assert_allclose(oracle.normalise(x * 32, b, w), oracle.normalise(x, a, w), rtol=1e-14)


def test_rrms_zero_row_is_eps_only():
    eps = 1e-6
    r = oracle.grouped_rrms(np.zeros((1, 2, 8)), eps)
    np.testing.assert_allclose(r, 1.0 / math.sqrt(eps), rtol=1e-15)


# ------------------------------------------------------------------ G1 and INJ
def test_projection_one_hot_rows_pick_entries():
    rng = np.random.default_rng(9)
    M, K, n = 3, 24, 5
    xn = rng.standard_normal((M, K))
    ks = [3, 0, 23, 11, 7]
    W = np.zeros((n, K))
    W[np.arange(n), ks] = 1.0
    np.testing.assert_array_equal(oracle.project(xn, W), xn[:, ks])


def test_projection_is_x_times_W_transposed():
    # A non-square, non-symmetric case: out[m, n] = sum_k x[m, k] W[n, k].
    x = np.array([[1.0, 2.0, 3.0]])
    W = np.array([[1.0, 0.0, 0.0], [0.0, 10.0, 100.0]])
    np.testing.assert_array_equal(oracle.project(x, W), [[1.0, 320.0]])


def test_silu_h_matches_torch_with_hc_scaling():
    HC = 4
    lora = np.linspace(-60, 60, 241).reshape(1, -1)
    want = torch.nn.functional.silu(torch.from_numpy(lora / HC)).numpy()
    np.testing.assert_allclose(oracle.silu_h(lora, HC), want, rtol=1e-13, atol=1e-300)
    # closed form: lora = HC ln 3 -> u = ln 3 -> h = (3/4) ln 3
    np.testing.assert_allclose(oracle.silu_h(np.array([HC * math.log(3.0)]), HC),
                               0.75 * math.log(3.0), rtol=1e-15)


# ------------------------------------------------------------------- G2 and MIX
def test_up_gate_zero_weight_is_half():
    h = np.random.default_rng(10).standard_normal((2, 6))
    np.testing.assert_array_equal(oracle.up_gate(h, np.zeros((20, 6))), 0.5)


def test_up_gate_one_hot_rows():
    h = np.array([[0.0, math.log(3.0), -math.log(3.0)]])
    Wu = np.array([[0, 1, 0], [0, 0, 1], [1, 0, 0], [0, 2, 0]], dtype=np.float64)
    np.testing.assert_allclose(oracle.up_gate(h, Wu), [[0.75, 0.25, 0.5, 0.9]], rtol=1e-14)


def test_gated_mean_closed_form():
    # G = 1/2 everywhere: x = (1/2) * mean over streams of xn.
    rng = np.random.default_rng(11)
    HC, HS = 4, 6
    xn = rng.standard_normal((2, HC * HS))
    x = oracle.gated_mean(np.full_like(xn, 0.5), xn, HC)
    np.testing.assert_allclose(x, 0.5 * xn.reshape(2, HC, HS).mean(axis=1), rtol=1e-15)
    # stream-dependent gate picks out a weighted mean with weights G[s]/HC
    G = np.repeat(np.array([[1.0, 0.0, 0.25, 0.5]]), HS, axis=1).reshape(1, HC * HS)
    xs = np.repeat(np.array([[8.0, 100.0, 4.0, 2.0]]), HS, axis=1).reshape(1, HC * HS)
    np.testing.assert_allclose(oracle.gated_mean(G, xs, HC), (8.0 + 0 + 1.0 + 1.0) / 4.0)


def test_whole_op_zero_up_weight():
    # Wu = 0 gives G = 1/2 and x = (1/2) mean_s xn, whatever the other inputs.
    rng = np.random.default_rng(12)
    c = _case(rng, 3, 4, 16, 8)
    c["Wu"] = np.zeros_like(c["Wu"])
    out = oracle.forward(**c)
    np.testing.assert_array_equal(out["G"], 0.5)
    np.testing.assert_allclose(out["x"], 0.5 * out["xn"].reshape(3, 4, 16).mean(axis=1),
                               rtol=1e-15)


def test_whole_op_constant_rows_closed_form():
    # R2 constant per stream, Wnorm = 0, Wu = 0: xn[s, c] = a_s / sqrt(a_s^2 + eps)
    # and x[c] = (1/2) mean_s xn[s].
    HC, HS, r, eps = 4, 8, 4, 1e-6
    a = np.array([0.5, -2.0, 3.0, 1.0])
    R = np.broadcast_to(a[None, :, None], (1, HC, HS)).copy()
    out = oracle.forward(R=R, y=np.zeros((1, HS)), inj=np.zeros((1, HC)), Wnorm=np.zeros(HC * HS),
                         Wd=np.ones((r, HC * HS)), Wi=np.ones((HC, HC * HS)),
                         Wu=np.zeros((HC * HS, r)), eps=eps)
    xs = a / np.sqrt(a * a + eps)
    np.testing.assert_allclose(out["x"][0], np.full(HS, 0.5 * xs.mean()), rtol=1e-14)
    np.testing.assert_allclose(out["lora"][0], np.full(r, HS * xs.sum()), rtol=1e-14)
    np.testing.assert_allclose(out["inj_next"][0], np.full(HC, HS * xs.sum()), rtol=1e-14)


# ----------------------------------------------------------------- invariants
def test_stream_permutation_invariance():
    rng = np.random.default_rng(13)
    M, HC, HS, r = 3, 4, 16, 8
    c = _case(rng, M, HC, HS, r)
    p = np.array([2, 0, 3, 1])
    kperm = (p[:, None] * HS + np.arange(HS)[None, :]).reshape(-1)
    q = dict(c, R=c["R"][:, p], inj=c["inj"][:, p], Wnorm=c["Wnorm"][kperm],
             Wd=c["Wd"][:, kperm], Wi=c["Wi"][:, kperm], Wu=c["Wu"][kperm])
    a, b = oracle.forward(**c), oracle.forward(**q)
    for k in ("lora", "inj_next", "x"):
        np.testing.assert_allclose(b[k], a[k], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(b["R2"], a["R2"][:, p])
    np.testing.assert_allclose(b["rrms"], a["rrms"][:, p], rtol=1e-15)


def test_batch_invariance():
    rng = np.random.default_rng(14)
    c = _case(rng, 5, 2, 8, 4)
    full = oracle.forward(**c)
    one = oracle.forward(**dict(c, R=c["R"][3:4], y=c["y"][3:4], inj=c["inj"][3:4]))
    for k in ("R2", "rrms", "lora", "inj_next", "x"):
        np.testing.assert_allclose(one[k][0], full[k][3], rtol=1e-14, atol=1e-15)


def test_mix_is_the_path_with_nothing_injected():
    # The mix entry point runs (N) onwards on R as the combined residual.
    # With y = 0, COMBINE leaves every bf16 R unchanged whatever inj is
    # (R + 0 * iw = R), so the whole path must give the same outputs.
    rng = np.random.default_rng(16)
    c = _case(rng, 4, 4, 16, 8)
    m = oracle.mix(c["R"], c["Wnorm"], c["Wu"], c["eps"], Wd=c["Wd"], Wi=c["Wi"])
    f = oracle.forward(**dict(c, y=np.zeros_like(c["y"])))
    np.testing.assert_array_equal(f["R2"], c["R"])
    for k in ("rrms", "lora", "inj_next", "h", "G", "x"):
        np.testing.assert_array_equal(m[k], f[k])
    assert "R2" not in m


def test_mix_constant_rows_closed_form():
    # Mix alone on constant streams a_s with Wnorm = 0 and Wu = 0:
    # x[c] = (1/2) mean_s a_s / sqrt(a_s^2 + eps), lora[n] = HS sum_s xn_s for
    # all-ones Wd rows -- the closed form of (N), (G1), (G2) and (MIX).
    HC, HS, r, eps = 4, 8, 4, 1e-6
    a = np.array([1.5, -0.25, 2.0, -4.0])
    R = np.broadcast_to(a[None, :, None], (2, HC, HS)).copy()
    out = oracle.mix(R, np.zeros(HC * HS), np.zeros((HC * HS, r)), eps,
                     Wd=np.ones((r, HC * HS)), Wi=np.ones((HC, HC * HS)))
    xs = a / np.sqrt(a * a + eps)
    np.testing.assert_allclose(out["rrms"], np.broadcast_to(1.0 / np.sqrt(a * a + eps), (2, HC)),
                               rtol=1e-15)
    np.testing.assert_allclose(out["x"], np.full((2, HS), 0.5 * xs.mean()), rtol=1e-14)
    np.testing.assert_allclose(out["lora"], np.full((2, r), HS * xs.sum()), rtol=1e-14)


def test_broadcast_norm_weight_is_the_tiled_full_width_one():
    # An [HS] norm weight acts on every stream alike: the same outputs as the
    # K-entry weight that repeats it HC times, and a stream permutation of
    # R no longer needs a matching permutation of Wnorm.
    rng = np.random.default_rng(17)
    M, HC, HS, r = 3, 4, 16, 8
    c = _case(rng, M, HC, HS, r)
    w_hs = _rand(rng, HS, scale=0.1)
    a = oracle.forward(**dict(c, Wnorm=w_hs))
    b = oracle.forward(**dict(c, Wnorm=np.tile(w_hs, HC)))
    for k in ("R2", "rrms", "xn", "lora", "inj_next", "x"):
        np.testing.assert_array_equal(a[k], b[k])
    xn = a["xn"].reshape(M, HC, HS)
    R2 = a["R2"]
    for s_ in range(HC):
        np.testing.assert_allclose(xn[:, s_], R2[:, s_] * a["rrms"][:, s_, None] * (1.0 + w_hs),
                                   rtol=1e-15)
    Wf = oracle.merge_weight(c["Wd"], c["Wi"], w_hs, n_pad=12, fold=True)
    np.testing.assert_array_equal(Wf, oracle.merge_weight(c["Wd"], c["Wi"], np.tile(w_hs, HC), 12,
                                                          fold=True))
    with pytest.raises(ValueError):
        oracle.forward(**dict(c, Wnorm=np.zeros(HS + 1)))


def test_fold_equivalence_exact_weights():
    # Folding (1 + Wnorm) into the weight columns is the same product when the
    # fold is kept in float64; the mix still sees (1 + Wnorm).
    rng = np.random.default_rng(15)
    c = _case(rng, 3, 4, 16, 8)
    base = oracle.forward(**c)
    Wdi = oracle.merge_weight(c["Wd"], c["Wi"], c["Wnorm"], n_pad=16, fold=True)
    f = oracle.forward(**dict(c, Wd=None, Wi=None), Wdi=Wdi, fold_w=True)
    for k in ("lora", "inj_next", "x", "R2", "rrms"):
        np.testing.assert_allclose(f[k], base[k], rtol=1e-12, atol=1e-14)
    g = oracle.forward(**dict(c, Wd=None, Wi=None),
                       Wdi=oracle.merge_weight(c["Wd"], c["Wi"], c["Wnorm"], 12, fold=False))
    for k in ("lora", "inj_next", "x"):
        np.testing.assert_allclose(g[k], base[k], rtol=1e-13, atol=1e-15)


def test_merge_weight_layout():
    Wd = np.arange(6, dtype=np.float64).reshape(2, 3) + 1
    Wi = -np.arange(3, dtype=np.float64).reshape(1, 3) - 1
    wn = np.array([1.0, 0.0, -0.5])
    W = oracle.merge_weight(Wd, Wi, wn, n_pad=4, fold=True)
    np.testing.assert_array_equal(W, [[2, 2, 1.5], [8, 5, 3], [-2, -2, -1.5], [0, 0, 0]])


# ------------------------------------------------------------------ brute force
def _brute(R, y, inj, Wnorm, Wd, Wi, Wu, eps):
    """Direct per-element evaluation with Python scalars and math.exp."""
    M, HC, HS = len(R), len(R[0]), len(R[0][0])
    r = len(Wd)
    K = HC * HS
    sig = lambda v: 1.0 / (1.0 + math.exp(-v)) if v > -700 else 0.0
    res = {k: [] for k in ("R2", "rrms", "lora", "inj_next", "x")}
    for m in range(M):
        R2 = [[0.0] * HS for _ in range(HC)]
        for s in range(HC):
            iw = 2.0 * sig(inj[m][s] / HC)
            for c in range(HS):
                R2[s][c] = float(oracle.bf16_round(R[m][s][c] + y[m][c] * iw))
        rr = []
        for s in range(HC):
            acc = 0.0
            for c in range(HS):
                acc += R2[s][c] * R2[s][c]
            rr.append(1.0 / math.sqrt(acc / HS + eps))
        xn = [0.0] * K
        for s in range(HC):
            for c in range(HS):
                xn[s * HS + c] = R2[s][c] * rr[s] * (1.0 + Wnorm[s * HS + c])
        lora = [sum(xn[k] * Wd[n][k] for k in range(K)) for n in range(r)]
        injn = [sum(xn[k] * Wi[j][k] for k in range(K)) for j in range(HC)]
        h = [(l / HC) * sig(l / HC) for l in lora]
        G = [sig(sum(h[n] * Wu[k][n] for n in range(r))) for k in range(K)]
        x = [sum(G[s * HS + c] * xn[s * HS + c] for s in range(HC)) / HC for c in range(HS)]
        res["R2"].append(R2)
        res["rrms"].append(rr)
        res["lora"].append(lora)
        res["inj_next"].append(injn)
        res["x"].append(x)
    return {k: np.array(v) for k, v in res.items()}


@pytest.mark.parametrize("M,HC,HS,r", [(2, 2, 4, 2), (3, 3, 8, 4), (1, 4, 5, 3)])
def test_brute_force_tiny(M, HC, HS, r):
    rng = np.random.default_rng(100 + HC)
    c = _case(rng, M, HC, HS, r, wn_scale=0.3)
    got = oracle.forward(**c)
    want = _brute(c["R"].tolist(), c["y"].tolist(), c["inj"].tolist(), c["Wnorm"].tolist(),
                  c["Wd"].tolist(), c["Wi"].tolist(), c["Wu"].tolist(), c["eps"])
    for k, v in want.items():
        np.testing.assert_allclose(got[k], v, rtol=1e-12, atol=1e-14, err_msg=k)
