"""GPU parity of the persistent CTA-pair tensor-core kernel (path
"gemm_pair": tcgen05.mma.cta_group::2, 256-row tiles over two SMs, two TMEM
accumulators) against the oracle, through the C ABI.

Each dequantised weight reaches the tensor core as the exact bf16 pair hi +
lo (bf16 scales) or within 2^-16 of w (fp32 scales), so the stated bound
2e-3 * sum|a w| + 1e-5 applies everywhere, including tiny K and inputs whose
single bf16 rounding would all err the same way (tests/adversarial.py).
Shapes cover ragged M, N and K, every block size, zero points, both scale
dtypes, tile widths of 4 to 8 weight tiles per CTA and pairs that take
several tiles in turn (both accumulators, reused).
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


def run(prob, dev, path="gemm_pair"):
    f = lambda t: None if t is None else t.to(dev)
    w = mnb.mnb_prepack(f(prob.B), f(prob.scales), f(prob.zero_points), prob.N, prob.K,
                        prob.block_size)
    Y = mnb.mnb_matmul(f(prob.A), w, f(prob.bias), path=path, workspace=None)
    torch.cuda.synchronize()
    return Y


def ref(prob, rows=None, cols=None):
    return oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, prob.bias,
                              N=prob.N, K=prob.K, block_size=prob.block_size,
                              rows=rows, cols=cols)


def sample(n, k, seed, edges=()):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.asarray(edges, dtype=np.int64),
                                     rng.choice(n, min(n, k), replace=False)]))


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("scale_f32", [False, True])
def test_pair_tiles_and_tails(dev, bs, with_zp, scale_f32):
    """One tile and a few: ragged M (inside and past the 128 rows of a CTA)
    and N (inside one CTA's weight tiles and past them), a partial last
    block, with and without bias; every element checked."""
    i = 0
    for (M, N, K) in ((256, 256, 256), (257, 300, 520), (17, 16, 264), (600, 1000, 1024),
                      (130, 2560, 640)):
        i += 1
        prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=with_zp,
                            bias=(i % 2 == 0), seed=20 * bs + i)
        if scale_f32:
            prob.scales = prob.scales.float()
        Y = run(prob, dev)
        R, mag = ref(prob)
        check(Y, R, mag, f"pair M{M} N{N} K{K} bs{bs}")
    assert mnb.mnb_fault_status() == 0


@pytest.mark.parametrize("N", [1024, 2560, 4096, 9728, 4100])
def test_pair_several_tiles_per_pair(dev, N):
    """More tiles than CTA pairs (each pair runs several tiles through both
    accumulators); the tile width the plan picks for N (4 to 8 weight tiles
    per CTA); seeded rows (the first and last of each CTA's half) x columns
    (both CTAs' halves of a tile, the ragged N tail)."""
    M, K, bs = 4096, 192, 64
    plan = mnb.mnb_matmul_plan(M, N, K, bs, zero_points=True, path="gemm_pair")
    assert plan["pair_cols"] in (128, 160, 192, 224, 256)
    prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=True, bias=True,
                        seed=N)
    Y = run(prob, dev)
    rows = sample(M, 24, N, edges=[0, 127, 128, 255, 256, 3839, 3840, M - 1])
    cols = sample(N, 96, N + 1, edges=list(range(0, 8)) + list(range(N - 8, N)) +
                  [plan["pair_cols"] // 2 - 1, plan["pair_cols"] // 2])
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, f"pair several tiles N{N}")
    assert mnb.mnb_fault_status() == 0


@pytest.mark.parametrize("K", [8, 16, 40, 64, 136])
def test_pair_small_k_within_stated_bound(dev, K):
    prob = make_problem(300, 70, K, 16, dtype=torch.bfloat16, zero_points=True, bias=True,
                        seed=K)
    Y = run(prob, dev)
    R, mag = ref(prob)
    check(Y, R, mag, f"pair small K{K}")


@pytest.mark.parametrize("scale_dtype", [torch.bfloat16, torch.float32], ids=["sbf16", "sf32"])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("bs", [16, 64, 128])
def test_pair_adversarial_rounding_within_stated_bound(dev, bs, with_zp, scale_dtype):
    prob = aligned_rounding_problem(300, 70, bs, 4, scale_dtype=scale_dtype,
                                    zero_points=with_zp, seed=bs)
    Y = run(prob, dev)
    R, mag = ref(prob)
    check(Y, R, mag, f"pair adversarial bs{bs}")


def test_pair_adversarial_rounding_many_tiles(dev):
    prob = aligned_rounding_problem(2048, 9728, 128, 2, scale_dtype=torch.bfloat16,
                                    zero_points=True, seed=6)
    Y = run(prob, dev)
    rows = sample(2048, 12, 1, edges=[0, 2047])
    cols = sample(9728, 64, 2, edges=[0, 9727])
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, "pair adversarial many tiles")


@pytest.mark.parametrize("proj", QWEN3_4B["projections"], ids=lambda p: p.name)
def test_pair_qwen3_4b_prefill_sampled(dev, proj):
    """Qwen3-4B prefill shapes at M = 2048 (bf16 A, bs 128, zero points,
    fp32 bias): 8 seeded rows x 64 seeded columns."""
    M = 2048
    prob = make_problem(M, proj.N, proj.K, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=M + proj.N + 1, scale_range=(0.002, 0.01))
    Y = run(prob, dev)
    rows = sample(M, 8, proj.K)
    cols = sample(proj.N, 64, proj.N)
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y[rows][:, cols], R, mag, f"pair prefill {proj.name}")


def test_pair_bitwise_reproducible(dev):
    """Two runs agree bitwise (each output is summed in k order by one
    accumulator); the tile-per-CTA kernel, which splits K over a cluster on
    this shape, agrees within the bound."""
    prob = make_problem(600, 1000, 2560, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=3)
    a = run(prob, dev)
    assert torch.equal(a, run(prob, dev))
    R, mag = ref(prob)
    check(run(prob, dev, path="gemm"), R, mag, "tile kernel")
    check(a, R, mag, "pair kernel")


def test_pair_refusals(dev):
    """fp32 activations, and a plan query for them, are refused."""
    prob = make_problem(64, 128, 256, 64, dtype=torch.float32, seed=1)
    with pytest.raises(mnb.MnbError) as e:
        run(prob, dev)
    assert e.value.status == -8
    with pytest.raises(mnb.MnbError):
        mnb.mnb_matmul_plan(64, 128, 256, 64, a_dtype=torch.float32, path="gemm_pair")


@pytest.mark.parametrize("path", ["gemm", "gemm_pair"])
def test_codes_equal_to_zero_point_give_bias_exactly(dev, path):
    """Every code equal to its block's zero point makes every weight exactly
    zero (hi = lo = 0 in both tensor-core kernels, no offset to cancel), so
    Y is the bias rounded to bf16, bit for bit, on a ragged shape with
    several tiles."""
    M, N, K, bs = 300, 1000, 512, 32
    prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=True, bias=True,
                        seed=4)
    nb = K // bs
    Z = torch.randint(0, 16, (N, nb), generator=torch.Generator().manual_seed(2))
    prob.zero_points = (Z[:, 0::2] | (Z[:, 1::2] << 4)).to(torch.uint8)
    codes = Z.repeat_interleave(bs, dim=1)
    prob.B = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8).view(N, nb, bs // 2)
    Y = run(prob, dev, path=path)
    R, mag = ref(prob)
    assert not mag.any()
    want = prob.bias.to(torch.bfloat16).expand(M, N)
    assert torch.equal(Y.cpu(), want)
