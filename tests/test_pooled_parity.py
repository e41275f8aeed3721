"""The every-row parity checker used by the full-size GPU tests, on the CPU.

The full-size tests cut a large case into row chunks and check each chunk in
a spawn-started worker pool that draws the chunk's inputs from the seed again
and runs the oracle.  Here the checker is pinned without a GPU: the pooled
inputs equal the serial generator's, the oracle's own outputs (stored in the
GPU's output types) pass, and one planted wrong value in any single row --
first row, a chunk boundary, the last row, each output -- fails with the
right chunk reported.
"""
import numpy as np
import pytest

import oracle
from hyper_connection_gated_gb300 import inputs

from . import hcgr_testlib as tl

SHAPE = inputs.Shape(HC=2, HS=64, r=16)
M, STEP = 300, 64


@pytest.fixture(scope="module")
def pool():
    with tl.oracle_pool(workers=3) as p:
        yield p


def _as_gpu_types(ref):
    """The oracle's outputs stored the way the GPU returns them."""
    return {"R2": inputs.to_bf16_bits(ref["R2"]), "x": inputs.to_bf16_bits(ref["x"]),
            "rrms": ref["rrms"].astype(np.float32), "inj_next": ref["inj_next"].astype(np.float32),
            "lora": ref["lora"].astype(np.float32)}


@pytest.fixture(scope="module")
def case_and_ref():
    case = tl.make_case(M, SHAPE, seed=11)
    return case, _as_gpu_types(tl.oracle_ref(case))


def test_pooled_inputs_equal_serial_generator(pool):
    a = tl.pooled_activations(pool, M, SHAPE, seed=11, step=STEP)
    b = inputs.activations(M, SHAPE, seed=11)
    for k in b:
        np.testing.assert_array_equal(a[k], b[k])


def test_oracle_outputs_pass(pool, case_and_ref):
    _, got = case_and_ref
    rep = tl.pooled_parity(pool, got, M, SHAPE, seed=11, step=STEP)
    assert set(rep["worst"]) == {"R2", "x", "rrms", "inj_next", "lora"}
    # bf16 storage alone costs up to 2**-9 |o|, a fifth of the bound
    assert max(rep["worst"].values()) <= 0.25, rep


@pytest.mark.parametrize("key,row", [("x", 0), ("R2", 63), ("rrms", 64), ("lora", 191),
                                     ("inj_next", M - 1)])
def test_one_planted_row_is_caught(pool, case_and_ref, key, row):
    _, good = case_and_ref
    got = {k: v.copy() for k, v in good.items()}
    v = got[key].reshape(M, -1)
    if v.dtype == np.uint16:      # a bf16 value moved by three times its bound 1e-2 (1 + |o|)
        j = int(np.argmax(np.abs(inputs.bf16_bits_to_f64(v[row]))))
        o = inputs.bf16_bits_to_f64(v[row, j:j + 1])[0]
        v[row, j] = inputs.to_bf16_bits(np.array([o + 0.03 * (1.0 + abs(o))]))[0]
    else:                         # an fp32 value moved by 1 %
        j = int(np.argmax(np.abs(v[row])))
        v[row, j] *= 1.01
    rep = tl.pooled_parity(pool, got, M, SHAPE, seed=11, step=STEP)
    assert rep["worst"][key] > 1.0, rep
    assert rep["chunk_start"][key] == row // STEP * STEP
    others = {k: w for k, w in rep["worst"].items() if k != key}
    assert max(others.values()) <= 0.25


def test_mix_and_combine_kinds(pool):
    case = tl.make_case(M, SHAPE, seed=11)
    R = tl.f64(case, "R")
    mixed = oracle.mix(R, Wnorm=tl.f64(case, "Wnorm"), Wu=tl.f64(case, "Wu"), eps=SHAPE.eps,
                       Wd=tl.f64(case, "Wd"), Wi=tl.f64(case, "Wi"))
    got = {"x": inputs.to_bf16_bits(mixed["x"]), "rrms": mixed["rrms"].astype(np.float32),
           "inj_next": mixed["inj_next"].astype(np.float32), "lora": mixed["lora"].astype(np.float32)}
    rep = tl.pooled_parity(pool, got, M, SHAPE, seed=11, kind="mix", step=STEP)
    assert max(rep["worst"].values()) <= 0.25 and "R2" not in rep["worst"]
    R2 = oracle.combine(R, tl.f64(case, "y"), tl.f64(case, "inj"))[0]
    rep = tl.pooled_parity(pool, {"R2": inputs.to_bf16_bits(R2)}, M, SHAPE, seed=11,
                           kind="combine", step=STEP)
    assert rep["worst"] == {"R2": 0.0}
    # the mix checked as the fused call fails: R is not R2
    rep = tl.pooled_parity(pool, got, M, SHAPE, seed=11, kind="forward", step=STEP)
    assert max(rep["worst"].values()) > 1.0


def test_merged_weight_kind(pool):
    case = tl.make_case(M, SHAPE, seed=11)
    Wdi = tl.merged_weight_bits(case, 24, True)
    ref = tl.oracle_ref(case, Wdi_bits=Wdi, fold_w=True)
    rep = tl.pooled_parity(pool, _as_gpu_types(ref), M, SHAPE, seed=11, merged=(24, True),
                           step=STEP)
    assert max(rep["worst"].values()) <= 0.25, rep
