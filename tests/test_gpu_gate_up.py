"""GPU parity of the fused gated-MLP pair (mnb_matmul_gate_up) against the
oracle: Y = g * sigmoid(g) * u with g, u two MatMulNBits projections of A.

Bound, element by element: the kernel forms g and u within the matmul bound
e = 2e-3 * sum|a w| + 1e-5 each, then the product in fp32 and one rounding
to the output dtype. Since |d silu / dx| <= 1.1,
|Y - Y_ref| <= 1.1 e_g (|u| + e_u) + (|silu(g)| + 1.1 e_g) e_u
              + 2^-8 |Y_ref| (bf16 output; 2^-24 for fp32) + 1e-6 (|Y_ref| + 1)."""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import make_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def pair(M, N, K, bs, dtype, with_zp, bias, seed):
    g = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp, bias=bias, seed=seed)
    u = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp, bias=bias, seed=seed + 1)
    u.A = g.A
    return g, u


def run(dev, g, u):
    f = lambda t: None if t is None else t.to(dev)
    wg = mnb.mnb_prepack(f(g.B), f(g.scales), f(g.zero_points), g.N, g.K, g.block_size)
    wu = mnb.mnb_prepack(f(u.B), f(u.scales), f(u.zero_points), u.N, u.K, u.block_size)
    Y = mnb.mnb_matmul_gate_up(f(g.A), wg, wu, f(g.bias), f(u.bias))
    torch.cuda.synchronize()
    return Y


def check_pair(Y, g, u, what, rows=None, cols=None):
    R, gv, uv, mg, mu = oracle.gate_up(
        g.A, (g.B, g.scales, g.zero_points, g.bias), (u.B, u.scales, u.zero_points, u.bias),
        N=g.N, K=g.K, block_size=g.block_size, rows=rows, cols=cols)
    Yh = Y.float().cpu().double().numpy()
    if rows is not None:
        Yh = Yh[np.ix_(rows, cols)]
    eg, eu = 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5
    silu = gv / (1 + np.exp(-gv))
    out = 2.0 ** -8 if Y.dtype == torch.bfloat16 else 2.0 ** -24
    bound = (1.1 * eg * (np.abs(uv) + eu) + (np.abs(silu) + 1.1 * eg) * eu
             + out * np.abs(R) + 1e-6 * (np.abs(R) + 1))
    err = np.abs(Yh - R)
    assert np.all(err <= bound), (what, float(np.max(err / bound)))


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
def test_gate_up_tails(dev, bs, dtype, with_zp):
    """Ragged N and K, partial last block, M across the 16-row slices."""
    i = 0
    for (N, K) in ((7, bs + 1), (129, 257), (1000, 700)):
        for M in (1, 3, 16, 17):
            i += 1
            g, u = pair(M, N, K, bs, dtype, with_zp, bias=(i % 2 == 0), seed=50 * bs + i)
            check_pair(run(dev, g, u), g, u, f"M{M} N{N} K{K} bs{bs}")


def test_gate_up_qwen3_4b_decode_shape(dev):
    """Qwen3-4B gate/up, 2560 -> 9728, M = 1, bf16, bs 128: seeded sample of
    256 output columns."""
    g, u = pair(1, 9728, 2560, 128, torch.bfloat16, False, bias=False, seed=7)
    Y = run(dev, g, u)
    cols = np.sort(np.random.default_rng(1).choice(9728, 256, replace=False))
    check_pair(Y, g, u, "qwen3-4b gate/up", rows=np.array([0]), cols=cols)


def test_gate_up_matches_two_projections(dev):
    """The fused call agrees with two separate projections combined on the
    GPU in fp32 (within the bf16 output rounding of each path)."""
    g, u = pair(4, 3000, 1024, 32, torch.bfloat16, True, bias=True, seed=11)
    Y = run(dev, g, u).float()
    f = lambda t: None if t is None else t.to(dev)
    wg = mnb.mnb_prepack(f(g.B), f(g.scales), f(g.zero_points), g.N, g.K, 32)
    wu = mnb.mnb_prepack(f(u.B), f(u.scales), f(u.zero_points), u.N, u.K, 32)
    G = mnb.mnb_matmul(f(g.A), wg, f(g.bias)).float()
    U = mnb.mnb_matmul(f(g.A), wu, f(u.bias)).float()
    ref = G * torch.sigmoid(G) * U
    torch.cuda.synchronize()
    assert torch.allclose(Y, ref, rtol=2e-2, atol=1e-3)


def test_gate_up_bitwise_reproducible(dev):
    g, u = pair(2, 2560, 9728, 128, torch.bfloat16, False, bias=True, seed=13)
    assert torch.equal(run(dev, g, u), run(dev, g, u))


@pytest.mark.parametrize("bs", [32, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
def test_gate_up_tensor_core_path(dev, bs, with_zp):
    """M > 16 with bf16 activations: the tensor-core kernel's paired mode
    (64 output columns per CTA; ragged M and N; the split-K variant for the
    small shapes). The per-weight bf16 rounding of this path averages out at
    K >= 256, where the stated bound applies."""
    i = 0
    for (M, N, K) in ((40, 1000, 512), (300, 777, 1024), (129, 2560, 256), (2048, 130, 768)):
        i += 1
        g, u = pair(M, N, K, bs, torch.bfloat16, with_zp, bias=(i % 2 == 1), seed=90 * bs + i)
        Y = run(dev, g, u)
        rng = np.random.default_rng(i)
        rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, 7, replace=False)]))
        cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 40, replace=False)]))
        check_pair(Y, g, u, f"tensor-core M{M} N{N} K{K} bs{bs}", rows=rows, cols=cols)


def test_gate_up_qwen3_4b_prefill_sampled(dev):
    """Qwen3-4B gate/up at M = 2048 (bf16, bs 128, zero points, bias):
    8 rows x 64 columns sampled."""
    g, u = pair(2048, 9728, 2560, 128, torch.bfloat16, True, bias=True, seed=21)
    Y = run(dev, g, u)
    rng = np.random.default_rng(2)
    rows = np.sort(rng.choice(2048, 8, replace=False))
    cols = np.sort(rng.choice(9728, 64, replace=False))
    check_pair(Y, g, u, "qwen3-4b prefill gate/up", rows=rows, cols=cols)
