"""GPU parity of the prepack and the small-M (decode) kernel against the
oracle, called through the C ABI.

Every case draws seeded inputs on the CPU (workloads.make_problem), runs the
CUDA path on them and compares element by element with the double-precision
oracle on the same host tensors, within tests/tolerance.py's bound.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import (QWEN3_0P6B, QWEN3_4B,
                                                          make_problem)
from tests.tolerance import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def to_dev(prob, dev):
    f = lambda t: None if t is None else t.to(dev)
    return f(prob.A), f(prob.B), f(prob.scales), f(prob.zero_points), f(prob.bias)


def run_gpu(prob, dev, path="auto", stream=None):
    A, B, S, Z, bias = to_dev(prob, dev)
    w = mnb.mnb_prepack(B, S, Z, prob.N, prob.K, prob.block_size, stream=stream)
    Y = mnb.mnb_matmul(A, w, bias, path=path, stream=stream)
    torch.cuda.synchronize()
    return Y, w


def ref(prob, rows=None, cols=None):
    return oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, prob.bias,
                              N=prob.N, K=prob.K, block_size=prob.block_size,
                              rows=rows, cols=cols)


def parity(prob, dev, what, path="auto"):
    Y, _ = run_gpu(prob, dev, path)
    R, mag = ref(prob)
    return check(Y, R, mag, what)


# --- prepack -----------------------------------------------------------------

@pytest.mark.parametrize("N,K,bs", [(16, 64, 16), (7, 33, 16), (129, 257, 32),
                                    (33, 1000, 64), (5, 130, 128), (17, 300, 256),
                                    (3072, 1024, 32), (1, 1, 16)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
def test_prepack_round_trip_is_lossless(dev, N, K, bs, dtype, with_zp):
    prob = make_problem(1, N, K, bs, dtype=dtype, zero_points=with_zp, seed=N + K)
    _, B, S, Z, _ = to_dev(prob, dev)
    w = mnb.mnb_prepack(B, S, Z, N, K, bs)
    B2, S2, Z2 = mnb.mnb_unprepack(w)
    torch.cuda.synchronize()
    # storage padding past K is not kept: compare with it cleared
    Bexp = prob.B.clone().view(N, -1)
    nb = -(-K // bs)
    for k in range(K, nb * bs):
        byte = k // 2
        Bexp[:, byte] &= 0xF0 if k % 2 == 0 else 0x0F
    assert torch.equal(B2.cpu().view(N, -1), Bexp)
    assert torch.equal(S2.cpu().view(torch.uint8), prob.scales.view(torch.uint8))
    if with_zp:
        Zexp = prob.zero_points.clone()
        if nb % 2 == 1:
            Zexp[:, -1] &= 0x0F
        assert torch.equal(Z2.cpu(), Zexp)
    else:
        assert Z2 is None


# --- tails and edge cases ------------------------------------------------------

@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
def test_gemv_tail_matrix(dev, bs, dtype, with_zp):
    """K in {bs-1, bs+1, 3bs+7}, N in {1, 7, 129}, M in {1, 3, 8, 9, 16},
    with and without bias: partial blocks, odd N, packed-byte tails (page
    "Qwen3 CPU Inference Critical Path", section "Export contract": partial K
    blocks, odd N and packed-byte tails are mandatory synthetic tests)."""
    worst = 0.0
    seed = 0
    for K in (bs - 1, bs + 1, 3 * bs + 7):
        for N in (1, 7, 129):
            for M in (1, 3, 8, 9, 16):
                for bias in (False, True):
                    seed += 1
                    prob = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp,
                                        bias=bias, seed=1000 * bs + seed)
                    worst = max(worst, parity(prob, dev, f"M{M} N{N} K{K} bs{bs}"))
    assert worst <= 1.0


@pytest.mark.parametrize("M", [1, 2, 4, 8, 12, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gemv_many_tiles_and_cluster_splits(dev, M, dtype):
    """Shapes that take every split-K arrangement: a few tiles with long K
    (cluster split), many tiles with short K, a ragged N tail."""
    for (N, K, bs) in ((2560, 9728, 128), (1024, 2560, 128), (4099, 1024, 32),
                       (40, 4096, 64)):
        prob = make_problem(M, N, K, bs, dtype=dtype, zero_points=True, bias=True,
                            seed=N + M)
        parity(prob, dev, f"M{M} N{N} K{K}")


def test_codes_equal_to_zero_point_give_bias(dev):
    """Every code equal to its block's zero point makes every weight zero:
    Y = bias, within the bound at sum|a*w| = 0 (the kernel's offset
    cancellation is exact only up to fp32 rounding)."""
    M, N, K, bs = 3, 100, 256, 32
    prob = make_problem(M, N, K, bs, dtype=torch.float32, zero_points=True,
                        bias=True, seed=3)
    nb = K // bs
    Z = torch.randint(0, 16, (N, nb), generator=torch.Generator().manual_seed(1))
    prob.zero_points = (Z[:, 0::2] | (Z[:, 1::2] << 4)).to(torch.uint8)
    codes = Z.repeat_interleave(bs, dim=1)
    prob.B = (codes[:, 0::2] | (codes[:, 1::2] << 4)).to(torch.uint8).view(N, nb, bs // 2)
    Y, _ = run_gpu(prob, dev)
    R, mag = ref(prob)
    assert not mag.any()
    assert np.array_equal(R, np.broadcast_to(prob.bias.double().numpy(), (M, N)))
    check(Y, R, mag, "codes equal to zero point")


# --- the workloads' shapes -----------------------------------------------------

def test_single_gemv_config(dev):
    """A fp32 [1,1024] ~ N(0,1); codes uniform; bs 32; fp32 scales
    U[0.005, 0.02]; no zero points; no bias; seed 0."""
    prob = make_problem(1, 3072, 1024, 32, dtype=torch.float32, seed=0)
    parity(prob, dev, "single GEMV")


@pytest.mark.parametrize("proj", QWEN3_0P6B["projections"] + [QWEN3_0P6B["lm_head"]],
                         ids=lambda p: p.name)
def test_qwen3_0p6b_decode_shapes(dev, proj):
    prob = make_problem(1, proj.N, proj.K, 32, dtype=torch.float32, zero_points=True,
                        seed=11, scale_range=(0.005, 0.02))
    parity(prob, dev, proj.name)


@pytest.mark.parametrize("proj", QWEN3_4B["projections"] + [QWEN3_4B["lm_head"]],
                         ids=lambda p: p.name)
def test_qwen3_4b_decode_shapes(dev, proj):
    prob = make_problem(1, proj.N, proj.K, 128, dtype=torch.bfloat16, seed=12,
                        scale_range=(0.002, 0.01))
    parity(prob, dev, proj.name)


# --- reproducibility, streams, host entry point --------------------------------

def test_bitwise_reproducible_with_and_without_programmatic_launch(dev):
    prob = make_problem(4, 2560, 9728, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=5)
    Y1, w = run_gpu(prob, dev)
    A = prob.A.to(dev)
    bias = prob.bias.to(dev)
    Y2 = mnb.mnb_matmul(A, w, bias)
    mnb.mnb_set_programmatic_launch(False)
    try:
        Y3 = mnb.mnb_matmul(A, w, bias)
    finally:
        mnb.mnb_set_programmatic_launch(True)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2) and torch.equal(Y1, Y3)


def test_side_stream(dev):
    prob = make_problem(2, 1000, 700, 64, dtype=torch.float32, zero_points=True, seed=6)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        Y, _ = run_gpu(prob, dev, stream=s)
    R, mag = ref(prob)
    check(Y, R, mag, "side stream")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_matmul_from_host(dev, dtype):
    prob = make_problem(1, 2048, 1024, 32, dtype=dtype, zero_points=True, seed=7)
    _, B, S, Z, _ = to_dev(prob, dev)
    w = mnb.mnb_prepack(B, S, Z, prob.N, prob.K, 32)
    A_host = prob.A.pin_memory()
    Y_host = torch.empty(1, prob.N, dtype=dtype).pin_memory()
    A_dev = torch.empty_like(A_host, device=dev)
    Y_dev = torch.empty(1, prob.N, dtype=dtype, device=dev)
    mnb.mnb_matmul_from_host(A_host, A_dev, w, Y_dev, Y_host)
    torch.cuda.synchronize()
    R, mag = ref(prob)
    check(Y_host, R, mag, "from host")


def test_invalid_arguments_raise_and_launch_nothing(dev):
    prob = make_problem(1, 64, 128, 32, seed=8)
    A, B, S, Z, _ = to_dev(prob, dev)
    w = mnb.mnb_prepack(B, S, Z, 64, 128, 32)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul(torch.zeros(17, 128, device=dev), w, path="gemv")
    assert e.value.status == -8
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul(A, w, out=A[:, :64])  # output overlaps the input
    assert e.value.status == -6
    torch.cuda.synchronize()


# --- fused-N projections (one launch, shared activations) ---------------------

@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
def test_grouped_projections_match_oracle(dev, M, dtype, with_zp):
    """q/k/v-like group (N 4096/1024/1023, shared A) and a 4-weight group
    with a ragged K: each output against the oracle on the shared A."""
    for K, bs, Ns in ((2560, 128, (4096, 1024, 1023)), (1000, 32, (96, 7, 300, 129))):
        probs = [make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp,
                              bias=(i % 2 == 0), seed=100 * i + M) for i, N in enumerate(Ns)]
        A = probs[0].A
        ws, biases = [], []
        for pr in probs:
            _, B, S, Z, b = to_dev(pr, dev)
            ws.append(mnb.mnb_prepack(B, S, Z, pr.N, K, bs))
            biases.append(b)
        outs = mnb.mnb_matmul_grouped(A.to(dev), ws, biases)
        torch.cuda.synchronize()
        for pr, Y in zip(probs, outs):
            R, mag = oracle.matmulnbits(A, pr.B, pr.scales, pr.zero_points, pr.bias,
                                        N=pr.N, K=K, block_size=bs)
            check(Y, R, mag, f"grouped N{pr.N} K{K}")
