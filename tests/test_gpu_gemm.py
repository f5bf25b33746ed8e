"""GPU parity of the tensor-core (tcgen05/TMEM) prefill path and of the
M > 16 dispatch against the oracle, through the C ABI.

The bf16 path feeds each dequantised weight w = (q - z) * s to the tensor
core as two bf16 values, hi = w rounded and lo = the remainder, multiplied
into one fp32 accumulator: exact for bf16 scales, within 2^-16 for fp32
scales. So the stated bound 2e-3 * sum|a w| + 1e-5 holds for every input,
including tiny K and inputs built so that every weight's single bf16
rounding would err in the same direction (tests/adversarial.py); these
tests apply that bound everywhere.

fp32 activations take the tf32 kernel: the dequantised weight is rounded
to tf32 (2^-11) and the tensor core reads A with a tf32 significand
(2^-10), so each product is within 1.5e-3 of exact and the stated bound
holds rigorously for any K.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B, make_problem
from tests.adversarial import aligned_rounding_problem
from tests.tolerance import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def run(prob, dev, path="auto"):
    f = lambda t: None if t is None else t.to(dev)
    w = mnb.mnb_prepack(f(prob.B), f(prob.scales), f(prob.zero_points), prob.N, prob.K,
                        prob.block_size)
    Y = mnb.mnb_matmul(f(prob.A), w, f(prob.bias), path=path)
    torch.cuda.synchronize()
    return Y


def ref(prob, rows=None, cols=None):
    return oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, prob.bias,
                              N=prob.N, K=prob.K, block_size=prob.block_size,
                              rows=rows, cols=cols)


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("scale_f32", [False, True])
def test_gemm_tiles_and_tails(dev, bs, with_zp, scale_f32):
    """M, N and K tails around the 128 x 128 x 64 tile (ragged M and N, a
    partial last block), bf16 activations, with and without bias."""
    i = 0
    for (M, N, K) in ((128, 128, 256), (129, 257, 520), (300, 1000, 1024), (17, 16, 264),
                      (200, 130, 2560)):
        i += 1
        prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=with_zp,
                            bias=(i % 2 == 0), seed=10 * bs + i)
        if scale_f32:
            prob.scales = prob.scales.float()
        Y = run(prob, dev, path="gemm")
        R, mag = ref(prob)
        check(Y, R, mag, f"gemm M{M} N{N} K{K} bs{bs}")


@pytest.mark.parametrize("K", [8, 16, 40, 64, 136])
def test_gemm_small_k_within_stated_bound(dev, K):
    """Tiny K, where nothing averages out: the stated bound still holds."""
    prob = make_problem(130, 70, K, 16, dtype=torch.bfloat16, zero_points=True, bias=True,
                        seed=K)
    Y = run(prob, dev, path="gemm")
    R, mag = ref(prob)
    check(Y, R, mag, f"gemm small K{K}")


@pytest.mark.parametrize("scale_dtype", [torch.bfloat16, torch.float32], ids=["sbf16", "sf32"])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_gemm_adversarial_rounding_within_stated_bound(dev, bs, with_zp, scale_dtype):
    """Weights whose single bf16 rounding all err the same way (about 1.9x
    the stated bound if rounded once): 128-row tiles with a K split."""
    prob = aligned_rounding_problem(130, 70, bs, 4, scale_dtype=scale_dtype,
                                    zero_points=with_zp, seed=bs)
    Y = run(prob, dev, path="gemm")
    R, mag = ref(prob)
    check(Y, R, mag, f"adversarial bs{bs}")


def test_gemm_adversarial_rounding_256_row_tiles(dev):
    """The same inputs on a shape whose plan takes 256-row tiles (more
    output tiles than SMs), sampled rows and columns."""
    prob = aligned_rounding_problem(2048, 2560, 128, 3, scale_dtype=torch.bfloat16,
                                    zero_points=True, seed=5)
    assert mnb.mnb_matmul_plan(2048, 2560, prob.K, 128, zero_points=True)["tile_rows"] == 256
    Y = run(prob, dev)
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(2048, 16, replace=False))
    cols = np.sort(rng.choice(2560, 64, replace=False))
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, "adversarial 256-row tiles")


def test_gemm_matches_gemv_path_at_crossover(dev):
    """M = 16 through both kernels agree within the bound (same inputs)."""
    prob = make_problem(16, 2560, 2560, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=77)
    R, mag = ref(prob)
    check(run(prob, dev, path="gemm"), R, mag, "gemm M16")
    check(run(prob, dev, path="gemv"), R, mag, "gemv M16")


@pytest.mark.parametrize("M", [17, 64, 100])
def test_fp32_activations_above_16_rows(dev, M):
    """fp32 activations with M > 16 (and 16-byte rows) run the tf32 kernel."""
    prob = make_problem(M, 700, 1000, 32, dtype=torch.float32, zero_points=True, bias=True,
                        seed=M)
    Y = run(prob, dev)
    R, mag = ref(prob)
    check(Y, R, mag, f"fp32 M{M}")


@pytest.mark.parametrize("M", [512, 2048])
@pytest.mark.parametrize("proj", QWEN3_4B["projections"], ids=lambda p: p.name)
def test_qwen3_4b_prefill_sampled(dev, M, proj):
    """Qwen3-4B prefill shapes (bf16 A, bs 128, zero points, fp32 bias):
    seeded sample of 8 rows x 64 columns checked element by element."""
    prob = make_problem(M, proj.N, proj.K, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=M + proj.N, scale_range=(0.002, 0.01))
    Y = run(prob, dev)
    rng = np.random.default_rng(M * 7 + proj.K)
    rows = np.sort(rng.choice(M, 8, replace=False))
    cols = np.sort(rng.choice(proj.N, 64, replace=False))
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, f"prefill {proj.name} M{M}")


def test_gemm_bitwise_reproducible(dev):
    prob = make_problem(300, 1000, 2560, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=3)
    assert torch.equal(run(prob, dev, "gemm"), run(prob, dev, "gemm"))


@pytest.mark.parametrize("N", [12300, 12352])
@pytest.mark.parametrize("bs,with_zp", [(32, True), (64, False), (256, True)])
def test_gemm_256_row_tiles_with_tails(dev, bs, with_zp, N):
    """Enough output tiles for the 256-row tile variant (two A halves per B
    tile): ragged M (777 = 3*256 + 9) and N, a partial last block; seeded
    rows (incl. the first and the last) x columns (incl. the ragged N tail)
    checked element by element. N = 12300 (rows of Y not a multiple of 16
    bytes) takes the direct stores; N = 12352 = 96.5 * 128 the TMA stores
    of the staged tile, whose last tile has one 64-column box inside N and
    one wholly past it."""
    M, K = 777, 520
    prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=with_zp, bias=True,
                        seed=bs + 5)
    Y = run(prob, dev, path="gemm")
    rng = np.random.default_rng(bs)
    rows = np.unique(np.concatenate([[0, 255, 256, 511, 767, 768, M - 1],
                                     rng.choice(M, 9, replace=False)]))
    cols = np.unique(np.concatenate([np.arange(N - 12, N), np.arange(0, 16),
                                     rng.choice(N, 48, replace=False)]))
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, f"gemm256 bs{bs}")


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("scale_f32", [False, True])
def test_tf32_gemm_tiles_and_tails(dev, bs, with_zp, scale_f32):
    """fp32 activations on the tf32 kernel: ragged M and N around the
    128 x 128 tile, a partial last block, K from 4 to 2560."""
    i = 0
    for (M, N, K) in ((128, 128, 256), (129, 257, 520), (300, 1000, 1024), (17, 16, 264),
                      (200, 130, 2560), (33, 70, 4), (150, 40, 100)):
        i += 1
        prob = make_problem(M, N, K, bs, dtype=torch.float32, zero_points=with_zp,
                            bias=(i % 2 == 0), seed=20 * bs + i)
        if not scale_f32:
            prob.scales = prob.scales.to(torch.bfloat16)
        Y = run(prob, dev, path="gemm")
        assert Y.dtype == torch.float32
        R, mag = ref(prob)
        check(Y, R, mag, f"tf32 M{M} N{N} K{K} bs{bs}")


def test_fp32_rows_the_tma_cannot_address(dev):
    """K = 1001 fp32 rows are not 16-byte strided: the dispatch keeps them on
    the decode kernel's 16-row slices; forcing the tensor-core path is
    refused."""
    prob = make_problem(40, 300, 1001, 64, dtype=torch.float32, zero_points=True, bias=True,
                        seed=9)
    R, mag = ref(prob)
    check(run(prob, dev), R, mag, "fp32 K1001 auto")
    with pytest.raises(mnb.MnbError) as e:
        run(prob, dev, path="gemm")
    assert e.value.status == -8


@pytest.mark.parametrize("proj", ["q", "o", "gate", "down"])
def test_qwen3_0p6b_fp32_prefill_sampled(dev, proj):
    """Qwen3-0.6B prefill shapes as the artifact stores them (fp32 A and
    scales, bs 32, zero points), M = 512: seeded 8 rows x 64 columns."""
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_0P6B
    p = {q.name: q for q in QWEN3_0P6B["projections"]}[proj]
    prob = make_problem(512, p.N, p.K, 32, dtype=torch.float32, zero_points=True, bias=False,
                        seed=p.N + p.K)
    Y = run(prob, dev)
    rng = np.random.default_rng(p.N)
    rows = np.sort(rng.choice(512, 8, replace=False))
    cols = np.sort(rng.choice(p.N, 64, replace=False))
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, f"0.6B {proj}")
