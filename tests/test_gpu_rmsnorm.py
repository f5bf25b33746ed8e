"""GPU parity of the fused RMSNorm prologue and greedy-ArgMax epilogue
(mnb_matmul_rmsnorm) against the oracle (oracle.rmsnorm_matmul,
oracle.lm_head_argmax), through the C ABI.

Bound, element by element, with mag = sum_k |a'[m,k] w[n,k]| over the
normalized activations a':

  |Y - R| <= (2e-3 + u_stage + 1e-5) * mag + 1e-5 + u_out * |R|

2e-3 * mag + 1e-5 is the matmul tolerance. u_stage is the one rounding of
the staged normalized row: 2^-8 for bf16 activations (the row is rounded to
bf16, as the unfused graph rounds the normalization's output) and 2^-16 for
fp32 ones (hi + lo pair). 1e-5 * mag covers the fp32 sum of squares and
scale. u_out is the output's rounding (tests/tolerance.py).

ArgMax: the kernel compares fp32 values, so several indices can be correct
when logits are within the bound of each other. The check is that the
chosen index is a valid maximum: R[idx] + b[idx] >= max_n (R[n] - b[n]);
and, when the logits are also stored, that no stored logit exceeds the
chosen one and no earlier index equals it when the values are fp32.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.tolerance import U_OUT

pytestmark = pytest.mark.gpu

U_STAGE = {torch.float32: 2.0 ** -16, torch.bfloat16: 2.0 ** -8}


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def run(prob, dev, gamma, normalize=True, logits=True, argmax=False, eps=1e-6):
    f = lambda t: None if t is None else t.to(dev)
    w = mnb.mnb_prepack(f(prob.B), f(prob.scales), f(prob.zero_points), prob.N, prob.K,
                        prob.block_size)
    Y, idx = mnb.mnb_matmul_rmsnorm(f(prob.A), w, f(prob.bias), gamma=f(gamma), eps=eps,
                                    normalize=normalize, logits=logits, argmax=argmax)
    torch.cuda.synchronize()
    return Y, idx


def reference(prob, gamma, normalize=True, eps=1e-6, rows=None, cols=None):
    if normalize:
        return oracle.rmsnorm_matmul(prob.A, gamma, eps, prob.B, prob.scales, prob.zero_points,
                                     prob.bias, N=prob.N, K=prob.K, block_size=prob.block_size,
                                     rows=rows, cols=cols)
    return oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, prob.bias,
                              N=prob.N, K=prob.K, block_size=prob.block_size, rows=rows,
                              cols=cols)


def bound(R, mag, dtype):
    return (2e-3 + U_STAGE[dtype] + 1e-5) * mag + 1e-5 + U_OUT[dtype] * np.abs(R)


def check_logits(Y, R, mag, what):
    y = Y.float().cpu().double().numpy()
    assert np.all(np.isfinite(y)), what
    b = bound(R, mag, Y.dtype)
    err = np.abs(y - R)
    assert np.all(err <= b), (what, float(np.max(err / b)))


def check_argmax(idx, R, b, Y, what):
    idx = idx.cpu().numpy()
    for m in range(R.shape[0]):
        i = int(idx[m])
        assert 0 <= i < R.shape[1], (what, m, i)
        assert R[m, i] + b[m, i] >= np.max(R[m] - b[m]), (what, m, i)
        if Y is not None:
            y = Y[m].float().cpu().numpy()
            assert y[i] == y.max(), (what, m)
            if Y.dtype == torch.float32:
                assert i == int(np.argmax(y)), (what, m)


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
def test_rmsnorm_projection_tails(dev, bs, dtype, with_zp):
    """Ragged N and K, partial last block, M across 1..16, with and without
    gamma and bias; the ArgMax of every case too."""
    i = 0
    for (N, K) in ((7, bs + 1), (129, 257), (1000, 700)):
        for M in (1, 3, 16):
            i += 1
            prob = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp,
                                bias=(i % 2 == 0), seed=70 * bs + i)
            gamma = None if i % 3 == 0 else (
                torch.rand(K, generator=torch.Generator().manual_seed(i)) * 1.5 + 0.25)
            Y, idx = run(prob, dev, gamma, argmax=True)
            R, mag = reference(prob, gamma)
            check_logits(Y, R, mag, f"M{M} N{N} K{K} bs{bs}")
            check_argmax(idx, R, bound(R, mag, dtype), Y, f"M{M} N{N} K{K} bs{bs}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_plain_projection_with_argmax_only(dev, dtype):
    """normalize = 0 is the plain product; with the logits not stored the
    ArgMax alone comes back."""
    prob = make_problem(4, 3000, 640, 64, dtype=dtype, zero_points=True, bias=True, seed=17)
    Y, idx = run(prob, dev, None, normalize=False, logits=True, argmax=True)
    R, mag = reference(prob, None, normalize=False)
    b = 2e-3 * mag + 1e-5 + U_OUT[dtype] * np.abs(R)
    y = Y.float().cpu().double().numpy()
    assert np.all(np.abs(y - R) <= b)
    check_argmax(idx, R, b, Y, "plain")
    Y2, idx2 = run(prob, dev, None, normalize=False, logits=False, argmax=True)
    assert Y2 is None
    assert torch.equal(idx, idx2)


def test_argmax_ties_take_the_first_index(dev):
    """Rows whose weights repeat every 16 output rows give exactly equal
    logits in several places: the smallest index wins."""
    M, N, K, bs = 2, 64, 128, 32
    prob = make_problem(M, N, K, bs, dtype=torch.float32, seed=23)
    prob.B[16:] = prob.B[:16].repeat(3, 1, 1)
    prob.scales[16:] = prob.scales[:16].repeat(3, 1)
    Y, idx = run(prob, dev, None, normalize=True, argmax=True)
    y = Y.cpu().numpy()
    for m in range(M):
        i = int(idx[m])
        assert i < 16 and y[m, i] == y[m].max() and i == int(np.argmax(y[m]))


def test_qwen3_4b_final_norm_lm_head_argmax(dev):
    """Final RMSNorm + LM head (151936 x 2560, bf16, bs 128) + ArgMax, M = 1:
    logits on 512 seeded columns, the ArgMax against every column."""
    prob = make_problem(1, 151936, 2560, 128, dtype=torch.bfloat16, seed=29,
                        scale_range=(0.002, 0.01))
    gamma = torch.rand(2560, generator=torch.Generator().manual_seed(30)) + 0.5
    Y, idx = run(prob, dev, gamma, argmax=True)
    R, mag = reference(prob, gamma)
    check_argmax(idx, R, bound(R, mag, torch.bfloat16), Y, "lm_head")
    cols = np.sort(np.random.default_rng(2).choice(151936, 512, replace=False))
    check_logits(Y[:, cols], R[:, cols], mag[:, cols], "lm_head logits")


@pytest.mark.parametrize("M", [17, 512, 2048])
def test_prefill_rows_on_the_tensor_core_kernel(dev, M):
    """M > 16 with bf16 rows TMA can stage: the tensor-core kernel normalizes
    each staged A tile (A * gamma, rounded to bf16 once) and scales each
    output row by r[m] over the whole K. Qwen3-4B-like K (2560, bs 128, zero
    points, bias); seeded rows beyond 64 rows, every column."""
    N, K = 1536, 2560
    prob = make_problem(M, N, K, 128, dtype=torch.bfloat16, zero_points=True, bias=True,
                        seed=M, scale_range=(0.002, 0.01))
    gamma = torch.rand(K, generator=torch.Generator().manual_seed(M)) * 1.5 + 0.25
    Y, _ = run(prob, dev, gamma)
    rows = None if M <= 64 else np.sort(np.random.default_rng(M).choice(M, 48, replace=False))
    R, mag = reference(prob, gamma, rows=rows)
    check_logits(Y if rows is None else Y[rows], R, mag, f"prefill M{M}")


@pytest.mark.parametrize("case", ["tails", "fp32", "argmax", "no_gamma", "plain"])
def test_prefill_rows_other_forms(dev, case):
    """Ragged tiles on the tensor-core kernel (M 300, N 1000, K 704); and the
    forms served by 16-row decode slices: fp32 rows, rows TMA cannot stage
    (K % 8 != 0) with the ArgMax; gamma absent; normalize = 0."""
    M, N, K, dt = 300, 1000, 704, torch.bfloat16
    if case == "fp32":
        dt = torch.float32
    if case == "argmax":
        K = 700
    prob = make_problem(M, N, K, 64, dtype=dt, zero_points=True, bias=True, seed=len(case))
    gamma = None if case == "no_gamma" else (
        torch.rand(K, generator=torch.Generator().manual_seed(5)) * 1.5 + 0.25)
    normalize = case != "plain"
    Y, idx = run(prob, dev, gamma, normalize=normalize, argmax=case == "argmax")
    rows = np.sort(np.random.default_rng(3).choice(M, 40, replace=False))
    R, mag = reference(prob, gamma, normalize=normalize, rows=rows)
    check_logits(Y[rows], R, mag, f"prefill {case}")
    if case == "argmax":
        check_argmax(idx[rows], R, bound(R, mag, dt), Y[rows], "prefill argmax")
