"""The seeded input generator: determinism, prefix rows, distributions."""
import numpy as np

from hyper_connection_gated_gb300 import inputs


def test_uniforms_deterministic_and_counter_based():
    a = inputs.uniforms(7, 3, 0, 5000)
    b = inputs.uniforms(7, 3, 1000, 1000)
    np.testing.assert_array_equal(a[1000:2000], b)
    assert np.all((a > 0) & (a <= 1))
    assert not np.array_equal(a, inputs.uniforms(8, 3, 0, 5000))
    assert not np.array_equal(a, inputs.uniforms(7, 4, 0, 5000))


def test_normals_any_window():
    z = inputs.normals(1, 1, 0, 101)
    np.testing.assert_array_equal(inputs.normals(1, 1, 37, 20), z[37:57])
    np.testing.assert_array_equal(inputs.normals(1, 1, 38, 21), z[38:59])


def test_distributions():
    z = inputs.normals(inputs.SEED, 9, 0, 400000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    t = inputs.student_t3(inputs.SEED, 9, 0, 200000)
    # Student-t(3): median 0, interquartile range 2 * 0.7649
    q1, q3 = np.quantile(t, [0.25, 0.75])
    assert abs(np.median(t)) < 0.02 and abs((q3 - q1) - 1.5297) < 0.03


def test_bf16_bits_roundtrip():
    v = np.array([1.0, -2.5, 0.0, 3.0e38, 1e-40, np.inf])
    b = inputs.to_bf16_bits(v)
    assert b.dtype == np.uint16
    np.testing.assert_array_equal(inputs.bf16_bits_to_f64(b)[[0, 1, 2, 5]], v[[0, 1, 2, 5]])


def test_activation_prefix_rows_and_shapes():
    s = inputs.Shape(HC=2, HS=64, r=16)
    a = inputs.activations(5, s)
    b = inputs.activations(2, s)
    assert a["R"].shape == (5, 2, 64) and a["y"].shape == (5, 64) and a["inj"].shape == (5, 2)
    for k in ("R", "y", "inj"):
        np.testing.assert_array_equal(a[k][:2], b[k])
    c = inputs.activations(7, s, distinct_rows=3)
    np.testing.assert_array_equal(c["R"][5], a["R"][2])


def test_weight_scales():
    s = inputs.Shape(HC=4, HS=256, r=64)
    w = {k: inputs.bf16_bits_to_f64(v) for k, v in inputs.weights(s).items()}
    assert w["Wd"].shape == (64, 1024) and w["Wi"].shape == (4, 1024) and w["Wu"].shape == (1024, 64)
    assert abs(w["Wd"].std() * np.sqrt(1024) - 1) < 0.05
    assert abs(w["Wu"].std() * np.sqrt(64) - 1) < 0.05
    assert abs(w["Wnorm"].std() / 0.1 - 1) < 0.1
