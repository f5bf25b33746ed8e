"""CPU pins of the oracle's gated-MLP pair, Y = g * sigmoid(g) * u with g, u
two MatMulNBits projections of the same activations (page "Qwen3 CPU
Inference Critical Path": the graph-level fusion "gate projection, SiLU, and
gate/up multiplication"; SiLU as x * Sigmoid(x))."""
import math

import numpy as np
import torch

import oracle
from tests.packing import dense_weights, pack_codes, pack_zero_points


def _weight(rng, N, K, bs):
    nb = -(-K // bs)
    Q = rng.integers(0, 16, size=(N, K))
    Z = rng.integers(0, 16, size=(N, nb))
    S = rng.uniform(0.01, 0.05, size=(N, nb)).astype(np.float32)
    bias = rng.normal(0, 0.1, size=N).astype(np.float32)
    packed = (pack_codes(Q, bs), S, pack_zero_points(Z), bias)
    return packed, dense_weights(Q, Z, S, bs), bias.astype(np.float64)


def test_gate_up_brute_force_with_python_math(oracle_lib):
    """Tiny case in plain Python: dense weights from the logical codes, the
    dot products by hand, SiLU by math.exp."""
    rng = np.random.default_rng(3)
    M, N, K, bs = 2, 5, 40, 16
    gw, Wg, bg = _weight(rng, N, K, bs)
    uw, Wu, bu = _weight(rng, N, K, bs)
    A = rng.normal(0, 1, size=(M, K)).astype(np.float32)
    Y, g, u, _, _ = oracle.gate_up(A, gw, uw, N=N, K=K, block_size=bs, lib=oracle_lib)
    for m in range(M):
        for n in range(N):
            gv = sum(float(A[m, k]) * Wg[n, k] for k in range(K)) + bg[n]
            uv = sum(float(A[m, k]) * Wu[n, k] for k in range(K)) + bu[n]
            ref = gv / (1.0 + math.exp(-gv)) * uv
            assert math.isclose(Y[m, n], ref, rel_tol=1e-12, abs_tol=1e-12)
            assert math.isclose(g[m, n], gv, rel_tol=1e-12, abs_tol=1e-12)


def test_gate_up_special_values(oracle_lib):
    """A = 0 leaves only the biases: g = bias_g, u = bias_u; a zero gate bias
    gives Y = 0 (SiLU(0) = 0); a large gate gives Y close to g * u."""
    rng = np.random.default_rng(4)
    N, K, bs = 6, 32, 32
    gw, _, bg = _weight(rng, N, K, bs)
    uw, _, bu = _weight(rng, N, K, bs)
    A = np.zeros((1, K), dtype=np.float32)
    Y, g, u, _, _ = oracle.gate_up(A, gw, uw, N=N, K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(g[0], bg) and np.array_equal(u[0], bu)
    gw0 = gw[:3] + (np.zeros(N, dtype=np.float32),)
    Y0, _, _, _, _ = oracle.gate_up(A, gw0, uw, N=N, K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(Y0, np.zeros_like(Y0))
    big = gw[:3] + (np.full(N, 40.0, dtype=np.float32),)
    Yb, gb, ub, _, _ = oracle.gate_up(A, big, uw, N=N, K=K, block_size=bs, lib=oracle_lib)
    assert np.allclose(Yb, gb * ub, rtol=1e-15, atol=0)


def test_gate_up_sampling_matches_full(oracle_lib):
    rng = np.random.default_rng(5)
    M, N, K, bs = 4, 9, 70, 16
    gw, _, _ = _weight(rng, N, K, bs)
    uw, _, _ = _weight(rng, N, K, bs)
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    full = oracle.gate_up(A, gw, uw, N=N, K=K, block_size=bs, lib=oracle_lib)[0]
    rows, cols = np.array([3, 0]), np.array([8, 1, 4])
    part = oracle.gate_up(A, gw, uw, N=N, K=K, block_size=bs, rows=rows, cols=cols,
                          lib=oracle_lib)[0]
    assert np.array_equal(part, full[np.ix_(rows, cols)])
