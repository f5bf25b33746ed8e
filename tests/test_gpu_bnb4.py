"""GPU parity of the bitsandbytes-style 4-bit adapter (mnb_prepack_bnb4,
mnb_matmul_bnb4) against the oracle's statement (oracle.bnb4_matmul), through
the C ABI.

The code book is arbitrary (16 sorted values that are not bf16 numbers); the
kernel splits each code-book value c into bf16 hi = round(c) and lo =
round(c - hi), multiplied by the activations in two MMAs, so each weight is
within 2^-16 |w| of c * absmax (a single rounding could be 2^-8 |w| off,
twice the stated 2e-3 factor). The stated bound is applied throughout,
also on a code book and activations built so that a single rounding of each
value would err the same way (tests/adversarial.py). The re-layout itself is
checked bitwise: unpacking the plan gives the MatMulNBits storage of the
same logical codes and the absmax as per-row scales.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from tests.adversarial import aligned_rounding_codebook
from tests.packing import pack_bnb4_flat, pack_codes
from tests.tolerance import check

pytestmark = pytest.mark.gpu

CODE = (np.linspace(-1.0, 1.0, 16) + np.sin(np.arange(16)) * 0.013).astype(np.float32)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def problem(M, N, K, bs, a_dtype, s_dtype, bias, seed):
    rng = np.random.default_rng(seed)
    Q = rng.integers(0, 16, size=(N, K))
    absmax = torch.tensor(rng.uniform(0.01, 0.05, size=(N * K) // bs).astype(np.float32))
    absmax = absmax.to(s_dtype)
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(seed)).to(a_dtype)
    b = torch.tensor(rng.normal(0, 0.02, size=N).astype(np.float32)) if bias else None
    return Q, absmax, A, b


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("a_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("s_dtype", [torch.float32, torch.bfloat16])
def test_bnb4_matches_oracle(dev, bs, a_dtype, s_dtype):
    """Ragged N, K from one block to many, M across the 8-row slices."""
    i = 0
    for (N, K) in ((7, bs), (129, 4 * bs), (1000, 2560 // bs * bs or bs)):
        for M in (1, 5, 8, 17):
            i += 1
            Q, absmax, A, b = problem(M, N, K, bs, a_dtype, s_dtype, i % 2 == 0, 40 * bs + i)
            w = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(Q)).to(dev), absmax.to(dev),
                                     N, K, bs)
            Y = mnb.mnb_matmul_bnb4(A.to(dev), w, torch.tensor(CODE).to(dev),
                                    None if b is None else b.to(dev))
            torch.cuda.synchronize()
            R, mag = oracle.bnb4_matmul(A, pack_bnb4_flat(Q), absmax, CODE, b, N=N, K=K,
                                        block_size=bs)
            check(Y, R, mag, f"bnb4 M{M} N{N} K{K} bs{bs}")


@pytest.mark.parametrize("M", [17, 512])
@pytest.mark.parametrize("s_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("bs", [16, 64, 256])
def test_bnb4_prefill_rows_on_the_tensor_core_kernel(dev, M, s_dtype, bs):
    """Above 16 rows with bf16 activations: the tensor-core kernel's code-book
    mode (ragged N, K of several blocks); seeded rows at M = 512."""
    N, K = 300, 10 * bs
    Q, absmax, A, b = problem(M, N, K, bs, torch.bfloat16, s_dtype, True, M + bs)
    w = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(Q)).to(dev), absmax.to(dev), N, K, bs)
    Y = mnb.mnb_matmul_bnb4(A.to(dev), w, torch.tensor(CODE).to(dev), b.to(dev))
    torch.cuda.synchronize()
    rows = None if M <= 64 else np.sort(np.random.default_rng(M).choice(M, 40, replace=False))
    R, mag = oracle.bnb4_matmul(A, pack_bnb4_flat(Q), absmax, CODE, b, N=N, K=K,
                                block_size=bs, rows=rows)
    check(Y if rows is None else Y[rows], R, mag, f"bnb4 prefill M{M} bs{bs}")


@pytest.mark.parametrize("M", [1, 8, 17, 200])
@pytest.mark.parametrize("a_f32", [False, True], ids=["abf16", "af32"])
def test_bnb4_adversarial_code_book_within_stated_bound(dev, M, a_f32):
    bs, N = 64, 40
    A, Q, code = aligned_rounding_codebook(M, N, bs, 6, seed=M)
    if a_f32:
        A = A.float()
    K = Q.shape[1]
    absmax = torch.full((N * K // bs,), 0.5)
    w = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(Q)).to(dev), absmax.to(dev), N, K, bs)
    Y = mnb.mnb_matmul_bnb4(A.to(dev), w, code.to(dev))
    torch.cuda.synchronize()
    R, mag = oracle.bnb4_matmul(A, pack_bnb4_flat(Q), absmax, code.numpy(), None, N=N, K=K,
                                block_size=bs)
    check(Y, R, mag, f"bnb4 adversarial M{M}")


@pytest.mark.parametrize("bs", [16, 64, 256])
def test_bnb4_relayout_is_the_matmulnbits_plan_of_the_same_codes(dev, bs):
    N, K = 37, 3 * bs
    Q, absmax, _, _ = problem(1, N, K, bs, torch.float32, torch.float32, False, bs)
    w = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(Q)).to(dev), absmax.to(dev), N, K,
                             bs)
    B, S, Z = mnb.mnb_unprepack(w)
    torch.cuda.synchronize()
    assert Z is None
    assert np.array_equal(B.cpu().numpy().reshape(-1), pack_codes(Q, bs).reshape(-1))
    assert torch.equal(S.cpu(), absmax.reshape(N, K // bs))


def test_qwen3_4b_lm_head_shape(dev):
    """The LM head at full size (151936 x 2560, bs 64, bf16 A and absmax),
    M = 1: 512 seeded columns."""
    N, K, bs = 151936, 2560, 64
    Q, absmax, A, _ = problem(1, N, K, bs, torch.bfloat16, torch.bfloat16, False, 9)
    w = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(Q)).to(dev), absmax.to(dev), N, K,
                             bs)
    Y = mnb.mnb_matmul_bnb4(A.to(dev), w, torch.tensor(CODE).to(dev))
    torch.cuda.synchronize()
    cols = np.sort(np.random.default_rng(1).choice(N, 512, replace=False))
    R, mag = oracle.bnb4_matmul(A, pack_bnb4_flat(Q), absmax, CODE, None, N=N, K=K,
                                block_size=bs, cols=cols)
    check(Y[:, cols], R, mag, "bnb4 lm_head")


def test_blocks_straddling_rows_are_refused(dev):
    B = torch.zeros((16 * 40 + 1) // 2, dtype=torch.uint8, device=dev)
    absmax = torch.ones(16 * 40 // 16, device=dev)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_prepack_bnb4(B, absmax, 16, 40, 16)
    assert e.value.status == -8
