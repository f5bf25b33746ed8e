"""GPU parity of the QDQ INT4 re-layout (mnb_prepack_qdq) through both
kernels against the oracle's QDQ statement (page "Qwen3 CPU Inference
Critical Path", section "qwen3-int4-qdq": logical UINT4 [K, N] with
DequantizeLinear along axis 0 for projections, [N, K] along axis 1 for the
tied LM head; zero points default to 0)."""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from tests.packing import pack_flat
from tests.tolerance import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def qdq_problem(M, N, K, bs, *, axis, sdtype, adtype, with_zp, seed):
    """Seeded logical weight and its QDQ storage (host tensors)."""
    g = torch.Generator().manual_seed(seed)
    nb = -(-K // bs)
    Q = torch.randint(0, 16, (N, K), generator=g).numpy()
    Z = torch.randint(0, 16, (N, nb), generator=g).numpy()
    S = (torch.rand(N, nb, generator=g) * 0.015 + 0.005).to(sdtype)
    A = torch.randn(M, K, generator=g).to(adtype)
    bias = torch.randn(N, generator=g) * 0.02
    if axis == 0:
        Bq, Sq, Zq = pack_flat(Q.T), S.t().contiguous(), pack_flat(Z.T)
    else:
        Bq, Sq, Zq = pack_flat(Q), S.contiguous(), pack_flat(Z)
    return A, torch.from_numpy(Bq), Sq, (torch.from_numpy(Zq) if with_zp else None), bias


def run_and_check(dev, M, N, K, bs, *, axis, sdtype, adtype, with_zp, seed, path="auto"):
    A, Bq, Sq, Zq, bias = qdq_problem(M, N, K, bs, axis=axis, sdtype=sdtype, adtype=adtype,
                                      with_zp=with_zp, seed=seed)
    f = lambda t: None if t is None else t.to(dev)
    w = mnb.mnb_prepack_qdq(f(Bq), f(Sq), f(Zq), N, K, bs, axis=axis)
    Y = mnb.mnb_matmul(A.to(dev), w, bias.to(dev), path=path)
    torch.cuda.synchronize()
    R, mag = oracle.qdq_matmul(A, Bq, Sq, Zq, bias, N=N, K=K, block_size=bs, axis=axis)
    return check(Y, R, mag, f"qdq axis{axis} M{M} N{N} K{K} bs{bs}")


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
def test_qdq_tails_through_the_decode_kernel(dev, axis, bs, with_zp):
    """Odd N, K and N*K (flattened nibbles straddling rows), partial last
    block, M in {1, 3, 16}."""
    i = 0
    for (N, K) in ((7, 33), (129, 257), (33, 1000), (5, bs + 1)):
        for M in (1, 3, 16):
            i += 1
            run_and_check(dev, M, N, K, bs, axis=axis, sdtype=torch.bfloat16,
                          adtype=torch.bfloat16, with_zp=with_zp, seed=100 * bs + i)


@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("sdtype", [torch.float32, torch.bfloat16])
def test_qdq_through_the_tensor_core_kernel(dev, axis, sdtype):
    for (M, N, K) in ((200, 1000, 1024), (129, 257, 520)):
        run_and_check(dev, M, N, K, 32, axis=axis, sdtype=sdtype, adtype=torch.bfloat16,
                      with_zp=True, seed=M + N, path="gemm")


@pytest.mark.parametrize("adtype", [torch.float32, torch.bfloat16])
def test_qdq_contract_shapes(dev, adtype):
    """The QDQ contract's encoding (bs 32, bf16 scales, explicit UINT4 zero
    points) on Qwen3-0.6B projection shapes, K x N = 1024 x 2048 and
    3072 x 1024, and the tied LM-head access (axis 1), sampled columns."""
    run_and_check(dev, 1, 2048, 1024, 32, axis=0, sdtype=torch.bfloat16, adtype=adtype,
                  with_zp=True, seed=1)
    run_and_check(dev, 1, 1024, 3072, 32, axis=0, sdtype=torch.bfloat16, adtype=adtype,
                  with_zp=True, seed=2)
    run_and_check(dev, 1, 4096, 1024, 32, axis=1, sdtype=torch.bfloat16, adtype=adtype,
                  with_zp=True, seed=3)


def test_qdq_and_matmulnbits_layouts_pack_identically(dev):
    """The same logical weight prepacked from QDQ storage (axis 1, explicit
    zero points) and from MatMulNBits storage gives identical packed bytes."""
    from tests.packing import pack_codes, pack_zero_points
    N, K, bs = 70, 300, 32
    g = torch.Generator().manual_seed(9)
    nb = -(-K // bs)
    Q = torch.randint(0, 16, (N, K), generator=g).numpy()
    Z = torch.randint(0, 16, (N, nb), generator=g).numpy()
    S = (torch.rand(N, nb, generator=g) * 0.01).to(torch.bfloat16).to(dev)
    w1 = mnb.mnb_prepack(torch.from_numpy(pack_codes(Q, bs)).to(dev), S,
                         torch.from_numpy(pack_zero_points(Z)).to(dev), N, K, bs)
    w2 = mnb.mnb_prepack_qdq(torch.from_numpy(pack_flat(Q)).to(dev), S,
                             torch.from_numpy(pack_flat(Z)).to(dev), N, K, bs, axis=1)
    torch.cuda.synchronize()
    assert torch.equal(w1.packed_b, w2.packed_b)
    assert torch.equal(w1.packed_scales, w2.packed_scales)
    assert torch.equal(w1.packed_zp, w2.packed_zp)
