"""CPU pins of the oracle's RMS-style normalization and of its use as the
projection input (page "Qwen3 CPU Inference Critical Path": the exact
kernel inventory's SimplifiedLayerNormalization, FP32 RMS-style
normalization over the last axis with epsilon 1e-6; the fusion list's
"RMSNorm into packed projection input" and "final RMSNorm, LM-head GEMV,
and greedy ArgMax").

Pins: hand-worked fixtures (tests/golden/rmsnorm_hand_worked.json); the
closed form of a constant row; the mean of the squared output, which must
be S / (S + eps) for S = mean(x^2) (summed here with math.fsum, an
independent exact summation); invariance under scaling the row when
eps = 0; gamma acting elementwise; the normalized projection equal to the
plain projection of x times sqrt(K) / ||x||; and a copy of the oracle with
each of several planted mistakes failing at least one of these.
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.packing import pack_codes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_hand_worked.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _norm(x, gamma, eps, lib=None):
    g = None if gamma is None else np.asarray(gamma, dtype=np.float32)
    return oracle.rms_normalize(np.asarray(x, dtype=np.float64)[None, :], g, eps=eps,
                                lib=lib)[0]


def test_hand_worked_fixtures(oracle_lib):
    for c in _cases():
        got = _norm(c["x"], c["gamma"], c["eps"], oracle_lib)
        np.testing.assert_allclose(got, c["expected"], rtol=1e-15, atol=0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_constant_row_closed_form(oracle_lib, dtype):
    """x[k] = c: out[k] = c gamma[k] / sqrt(c^2 + eps)."""
    K = 37
    gamma = np.linspace(0.5, 2.0, K).astype(np.float32)
    for c in (-3.0, 0.25, 7.5):
        x = torch.full((1, K), c, dtype=dtype)
        got = oracle.rms_normalize(x, gamma, eps=1e-6, lib=oracle_lib)[0]
        want = c * gamma.astype(np.float64) / math.sqrt(c * c + 1e-6)
        np.testing.assert_allclose(got, want, rtol=1e-14)


def test_mean_square_invariant(oracle_lib):
    rng = np.random.default_rng(3)
    for K in (1, 2, 63, 1000):
        x = rng.standard_normal((4, K)) * rng.uniform(0.01, 10.0, size=(4, 1))
        eps = 1e-6 if K > 1 else 0.5
        y = oracle.rms_normalize(x, None, eps=eps, lib=oracle_lib)
        for m in range(4):
            S = math.fsum(v * v for v in x[m]) / K
            got = math.fsum(v * v for v in y[m]) / K
            assert math.isclose(got, S / (S + eps), rel_tol=1e-12), (K, m)


def test_scale_invariance_without_eps(oracle_lib):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 129))
    y = oracle.rms_normalize(x, None, eps=0.0, lib=oracle_lib)
    for alpha in (3.5, -0.125, 1024.0):
        ya = oracle.rms_normalize(alpha * x, None, eps=0.0, lib=oracle_lib)
        np.testing.assert_allclose(ya, np.sign(alpha) * y, rtol=1e-13)


def test_gamma_is_elementwise(oracle_lib):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 50))
    gamma = rng.uniform(-2, 2, 50).astype(np.float32)
    y1 = oracle.rms_normalize(x, None, eps=1e-6, lib=oracle_lib)
    yg = oracle.rms_normalize(x, gamma, eps=1e-6, lib=oracle_lib)
    np.testing.assert_allclose(yg, y1 * gamma.astype(np.float64)[None, :], rtol=1e-15)


def test_normalized_projection_is_scaled_plain_projection(oracle_lib):
    """eps = 0, gamma = 1: Y(norm(x)) = Y(x) * sqrt(K) / ||x|| with the
    separately pinned matmulnbits oracle on the fp32 row."""
    rng = np.random.default_rng(6)
    M, N, K, bs = 3, 11, 96, 32
    nb = K // bs
    Q = rng.integers(0, 16, size=(N, K))
    S = rng.uniform(0.005, 0.02, size=(N, nb)).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    Yn, _ = oracle.rmsnorm_matmul(x, None, 0.0, pack_codes(Q, bs), S, None, None, N=N, K=K,
                                  block_size=bs, lib=oracle_lib)
    Yp, _ = oracle.matmulnbits(x, pack_codes(Q, bs), S, None, None, N=N, K=K, block_size=bs,
                               lib=oracle_lib)
    norms = np.array([math.sqrt(math.fsum(float(v) ** 2 for v in row)) for row in x])
    np.testing.assert_allclose(Yn, Yp * (math.sqrt(K) / norms)[:, None], rtol=1e-12)


def test_double_activations_match_fp32_activations(oracle_lib):
    """The double input path widens exactly: fp32 values passed as fp32 or
    as double give bitwise the same projection."""
    rng = np.random.default_rng(7)
    N, K, bs = 5, 70, 16
    nb = -(-K // bs)
    Q = rng.integers(0, 16, size=(N, K))
    S = rng.uniform(0.005, 0.02, size=(N, nb)).astype(np.float32)
    x = rng.standard_normal((2, K)).astype(np.float32)
    a, _ = oracle.matmulnbits(x, pack_codes(Q, bs), S, None, None, N=N, K=K, block_size=bs,
                              lib=oracle_lib)
    b, _ = oracle.matmulnbits(x.astype(np.float64), pack_codes(Q, bs), S, None, None, N=N,
                              K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(a, b)


def test_argmax_takes_the_first_of_equal_logits():
    Y = np.array([[1.0, 3.0, 3.0, -1.0], [-2.0, -2.0, -5.0, -2.0]])
    assert oracle.lm_head_argmax(Y).tolist() == [1, 0]


# --- planted mistakes in a copy of the oracle's normalization ------------------

MUTATIONS = {
    "sum instead of mean": ("double r = 1.0 / sqrt(sumsq / (double)K + eps);",
                            "double r = 1.0 / sqrt(sumsq + eps);"),
    "eps outside the square root": ("double r = 1.0 / sqrt(sumsq / (double)K + eps);",
                                    "double r = 1.0 / (sqrt(sumsq / (double)K) + eps);"),
    "square root dropped": ("double r = 1.0 / sqrt(sumsq / (double)K + eps);",
                            "double r = 1.0 / (sumsq / (double)K + eps);"),
    "gamma dropped": ("double g = gamma ? (double)gamma[k] : 1.0;", "double g = 1.0;"),
    "absolute value instead of square": ("      sumsq += x * x;", "      sumsq += fabs(x);"),
    "gamma indexed by row": ("double g = gamma ? (double)gamma[k] : 1.0;",
                             "double g = gamma ? (double)gamma[m % K] : 1.0;"),
}


def _pins_pass(lib):
    for c in _cases():
        if not np.allclose(_norm(c["x"], c["gamma"], c["eps"], lib), c["expected"],
                           rtol=1e-12, atol=0):
            return False
    rng = np.random.default_rng(8)
    x = rng.standard_normal((3, 40))
    gamma = rng.uniform(0.5, 2.0, 40).astype(np.float32)
    y1 = oracle.rms_normalize(x, None, eps=1e-6, lib=lib)
    yg = oracle.rms_normalize(x, gamma, eps=1e-6, lib=lib)
    if not np.allclose(yg, y1 * gamma.astype(np.float64)[None, :], rtol=1e-14):
        return False
    for m in range(3):
        S = math.fsum(v * v for v in x[m]) / 40
        if not math.isclose(math.fsum(v * v for v in y1[m]) / 40, S / (S + 1e-6),
                            rel_tol=1e-12):
            return False
    return True


def test_pins_pass_on_the_real_oracle(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_each_planted_normalization_mistake_fails_a_pin(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(before) == 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", str(path), "-o", str(so),
                    "-lm"], check=True)
    assert not _pins_pass(oracle.load(str(so))), f"mutation '{name}' survived every pin"
