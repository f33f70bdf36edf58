"""Pins of the oracle's second and third workloads (CPU only).

* Row inverse RMS, FreeToken PR #101 ("The problem": rsqrt(mean(x^2) + eps)
  per row; "Accuracy": judged against float64).
* com.microsoft.EngramGate, its kernel README ("Description", "Inputs",
  "Attributes"): RMS-normalised key and query with per-stream scales, a
  scaled dot product, a signed-square-root sigmoid gate with a fixed 1e-6
  floor, the gate times the value row shared by the streams.

Each pin is a fact the oracle does not compute itself: worked examples with
hand-derived values, library routines (numpy's norm, scipy's expit), exact
invariants (power-of-two scaling, sign symmetry, permutations), closed forms
(a zero dot product gives exactly 1/2; key == query gives dot = sqrt(D)).
A dropped or misplaced term (epsilon, the 1/D of the mean, the 1/sqrt(D),
the floor, the scale row of a stream, the value row of a batch index) fails
at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from _util import DT_CODE, to_codes
from hyper_connection_rank_gb300 import inputs as I

scipy_special = pytest.importorskip("scipy.special")


@pytest.fixture(autouse=True, params=["cpu", pytest.param("gpu-session", marks=pytest.mark.gpu)])
def session(request):
    """Every pin runs twice: in the CPU test session and again, marked gpu, in
    the session that runs beside the GPU tests on the host processor of the
    machine that holds the GPU. The checker that judges the GPU results is
    then pinned on that host's architecture (aarch64 there, x86-64 here) and
    compiler, not only on the one it was written on."""
    return request.param


@pytest.fixture(scope="module")
def oracle():
    import oracle as O
    O.build()
    return O


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------- inverse RMS --

def test_inv_rms_worked_examples(oracle):
    # [3, 4]: mean of squares 12.5, 1/sqrt(12.5) = sqrt(2)/5
    got = oracle.inv_rms(f32([[3, 4], [1, 1], [0, 0]]), dtype=0, epsilon=0.0)
    assert got[0] == pytest.approx(0.28284271247461900976, rel=1e-15)
    assert got[1] == 1.0
    assert math.isinf(got[2])
    # epsilon sits under the square root: a zero row gives 1/sqrt(eps)
    z = oracle.inv_rms(f32([[0, 0, 0, 0]]), dtype=0, epsilon=0.25)
    assert z[0] == 2.0
    # and adds to the mean, not the sum: [2, 2, 2, 2] with eps 5 -> 1/sqrt(4 + 5) = 1/3
    assert oracle.inv_rms(f32([[2, 2, 2, 2]]), dtype=0, epsilon=5.0)[0] == pytest.approx(1 / 3, rel=1e-15)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_inv_rms_matches_library_norm(oracle, dt):
    x = I.make_inv_rms_input(64, 1024, dt, seed=3)
    got = oracle.inv_rms(to_codes(x), dtype=DT_CODE[dt], epsilon=0.0)
    x64 = x.to(torch.float64).numpy()
    ref = math.sqrt(x64.shape[1]) / np.linalg.norm(x64, axis=1)
    np.testing.assert_allclose(got, ref, rtol=1e-13)


def test_inv_rms_power_of_two_scaling_is_exact(oracle):
    x = I.make_inv_rms_input(16, 512, "f32", seed=4)
    a = oracle.inv_rms(to_codes(x), dtype=0, epsilon=0.0)
    b = oracle.inv_rms(to_codes(x * 8.0), dtype=0, epsilon=0.0)
    np.testing.assert_array_equal(b * 8.0, a)


def test_inv_rms_mean_not_sum(oracle):
    # a row repeated twice has the same mean of squares, hence the same result
    x = I.make_inv_rms_input(8, 256, "f32", seed=5)
    a = oracle.inv_rms(to_codes(x), dtype=0, epsilon=1e-3)
    b = oracle.inv_rms(to_codes(torch.cat([x, x], dim=1)), dtype=0, epsilon=1e-3)
    np.testing.assert_allclose(a, b, rtol=1e-14)


def test_inv_rms_dtype_codes_agree(oracle):
    # the same values given as bf16 codes and as float32 give the same result
    x = I.make_inv_rms_input(8, 384, "bf16", seed=6)
    a = oracle.inv_rms(to_codes(x), dtype=DT_CODE["bf16"], epsilon=1e-6)
    b = oracle.inv_rms(to_codes(x.float()), dtype=0, epsilon=1e-6)
    np.testing.assert_array_equal(a, b)


# ------------------------------------------------------------- Engram gate --

def engram(oracle, d, dt="f32", eps=1e-5):
    return oracle.engram_gate(*[to_codes(d[k]) for k in ("key", "query", "value", "key_scale", "query_scale")],
                              dtype=DT_CODE[dt], epsilon=eps)


def ones_scales(M, D):
    return torch.ones(M, D), torch.ones(M, D)


def test_engram_zero_dot_gives_half(oracle):
    # orthogonal key and query: dot = 0, sign(0) = 0, gate = sigmoid(0) = 1/2 exactly
    key = torch.tensor([[[1.0, 0.0, 1.0, 0.0]]])
    query = torch.tensor([[[0.0, 3.0, 0.0, -2.0]]])
    value = torch.tensor([[5.0, -1.5, 0.25, 7.0]])
    ks, qs = ones_scales(1, 4)
    out, gate = engram(oracle, dict(key=key, query=query, value=value, key_scale=ks, query_scale=qs))
    assert gate[0, 0] == 0.5
    np.testing.assert_array_equal(out[0, 0], f32([2.5, -0.75, 0.125, 3.5]))


@pytest.mark.parametrize("D", [16, 81, 256])
def test_engram_key_equals_query(oracle, D):
    # eps = 0, unit scales: k^ = q^, sum k^^2 = D, dot = D / sqrt(D) = sqrt(D),
    # gate = sigmoid(D ** 0.25)
    k = I.make_engram_inputs(2, 1, D, "f32", seed=7)["key"]
    ks, qs = ones_scales(1, D)
    out, gate = engram(oracle, dict(key=k, query=k.clone(), value=torch.ones(2, D), key_scale=ks, query_scale=qs),
                       eps=0.0)
    np.testing.assert_allclose(gate, scipy_special.expit(D ** 0.25), rtol=1e-14)


def test_engram_epsilon_inside_the_norms(oracle):
    # key == query, unit scales: sum k^^2 = D * m / (m + eps) with m = mean(k^2)
    D, eps = 32, 0.75
    k = I.make_engram_inputs(3, 1, D, "f32", seed=8)["key"]
    ks, qs = ones_scales(1, D)
    _, gate = engram(oracle, dict(key=k, query=k.clone(), value=torch.ones(3, D), key_scale=ks, query_scale=qs),
                     eps=eps)
    m = (k.double() ** 2).mean(dim=-1).numpy()[:, 0]
    dot = D * m / (m + eps) / math.sqrt(D)
    np.testing.assert_allclose(gate[:, 0], scipy_special.expit(np.sqrt(dot)), rtol=1e-14)


def test_engram_sign_symmetry(oracle):
    d = I.make_engram_inputs(4, 3, 64, "f32", seed=9)
    _, g1 = engram(oracle, d)
    d2 = dict(d, query=-d["query"])
    _, g2 = engram(oracle, d2)
    np.testing.assert_allclose(g1 + g2, 1.0, rtol=0, atol=1e-15)
    assert np.all((g1 > 0.5) == (g2 < 0.5))


def test_engram_floor(oracle):
    # dot = t / (rms(q) sqrt 2) ~ 6.7e-7 < 1e-6: the gate is sigmoid(sqrt(1e-6)) = sigmoid(1e-3)
    t = 2.0 ** -20
    key = torch.tensor([[[1.0, 1.0]]])
    query = torch.tensor([[[1.0, -1.0 + t]]])
    ks, qs = ones_scales(1, 2)
    _, gate = engram(oracle, dict(key=key, query=query, value=torch.ones(1, 2), key_scale=ks, query_scale=qs), eps=0.0)
    assert gate[0, 0] == pytest.approx(scipy_special.expit(1e-3), rel=1e-15)
    # above the floor the square root of |dot| is used: t = 2**-10 -> dot = 2**-10 / (rms(q) sqrt(2))
    t = 2.0 ** -10
    query = torch.tensor([[[1.0, -1.0 + t]]])
    _, gate = engram(oracle, dict(key=key, query=query, value=torch.ones(1, 2), key_scale=ks, query_scale=qs), eps=0.0)
    rq = math.sqrt((1.0 + (1.0 - t) ** 2) / 2.0)
    assert gate[0, 0] == pytest.approx(scipy_special.expit(math.sqrt(t / rq / math.sqrt(2.0))), rel=1e-14)


def test_engram_power_of_two_scaling(oracle):
    d = I.make_engram_inputs(3, 2, 48, "f32", seed=10)
    _, g1 = engram(oracle, d, eps=0.0)
    _, g2 = engram(oracle, dict(d, key=d["key"] * 4.0, query=d["query"] * 0.5), eps=0.0)
    np.testing.assert_array_equal(g1, g2)


def test_engram_stream_selects_scale_row(oracle):
    d = I.make_engram_inputs(5, 2, 40, "f32", seed=11)
    out1, g1 = engram(oracle, d)
    # swapping the two streams of key, query and both scale tables swaps the outputs
    sw = lambda t: t.flip(1) if t.dim() == 3 else t.flip(0)
    out2, g2 = engram(oracle, dict(d, key=sw(d["key"]), query=sw(d["query"]), key_scale=sw(d["key_scale"]),
                                   query_scale=sw(d["query_scale"])))
    np.testing.assert_array_equal(g2, g1[:, ::-1])
    np.testing.assert_array_equal(out2, out1[:, ::-1])
    # swapping only the scale rows changes the gates
    _, g3 = engram(oracle, dict(d, key_scale=sw(d["key_scale"]), query_scale=sw(d["query_scale"])))
    assert np.abs(g3 - g1).max() > 1e-4


def test_engram_value_row_is_shared_by_the_streams(oracle):
    d = I.make_engram_inputs(4, 3, 32, "f32", seed=12)
    out, gate = engram(oracle, d)
    v = d["value"].numpy()
    for b in range(4):
        for m in range(3):
            np.testing.assert_allclose(out[b, m], gate[b, m] * v[b], rtol=1e-7, atol=1e-30)


def test_engram_one_stream_row_independence(oracle):
    # a row's result does not depend on the other rows of the call
    d = I.make_engram_inputs(6, 2, 24, "f32", seed=13)
    out, gate = engram(oracle, d)
    sub = {k: (v[2:3] if k in ("key", "query", "value") else v) for k, v in d.items()}
    out1, gate1 = engram(oracle, sub)
    np.testing.assert_array_equal(out1[0], out[2])
    np.testing.assert_array_equal(gate1[0], gate[2])
