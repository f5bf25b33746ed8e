"""Pins for the CPU oracle (no GPU).

The oracle is the definition of MatMulNBits written out in double precision
(page "Qwen3 CPU Inference Critical Path", section "Exact kernel inventory",
MatMulNBits row; section "Prepared weight-only plan"). Each test here checks
it against something other than itself: a hand-worked fixture, exact integer
arithmetic on logical codes packed by an independent packer, a dense float64
library GEMM, and invariants that hold by the mathematics. The mutation tests
at the end prove the pins are not vacuous: plausible slips planted in a copy
of the oracle each fail at least one pin.
"""
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.packing import dense_weights, pack_codes, pack_zero_points

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "hand_worked_k5_bs4.json")) as f:
        return json.load(f)


def _run_golden(lib, g, dtype, with_zp):
    A = torch.tensor(g["A"], dtype=torch.float32).to(dtype)
    S = torch.tensor(g["scales"], dtype=torch.float32).to(dtype)
    B = np.array(g["B_bytes"], dtype=np.uint8)
    zp = np.array(g["zero_points_bytes"], dtype=np.uint8) if with_zp else None
    bias = np.array(g["bias"], dtype=np.float32)
    return oracle.matmulnbits(A, B, S, zp, bias, N=g["N"], K=g["K"],
                              block_size=g["block_size"], lib=lib)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [True, False])
def test_hand_worked_fixture(oracle_lib, dtype, with_zp):
    g = _golden()
    case = g["with_zero_points" if with_zp else "default_zero_point_8"]
    Y, mag = _run_golden(oracle_lib, g, dtype, with_zp)
    assert Y.tolist() == case["Y"]
    assert mag.tolist() == case["absdot"]
    B = np.array(g["B_bytes"], dtype=np.uint8)
    zp = np.array(g["zero_points_bytes"], dtype=np.uint8) if with_zp else None
    W = oracle.dequantize(B, torch.tensor(g["scales"]), zp, N=g["N"], K=g["K"],
                          block_size=g["block_size"], lib=oracle_lib)
    assert W.tolist() == case["weights"]


def test_golden_bytes_match_independent_packer():
    g = _golden()
    Q = np.array(g["logical_codes"])
    B = pack_codes(Q, g["block_size"], pad_value=0)
    B[0, -1, :] |= 0xF0  # the fixture's padding nibbles in row 0 are 15
    B[0, -1, 1] = 0xFF
    assert B.tolist() == g["B_bytes"]
    Z = np.array(g["zero_points_logical"])
    assert pack_zero_points(Z).tolist() == g["zero_points_bytes"]


# (M, N, K, block_size): tails in K (partial last block, odd K), odd N, tiny
# and several-block cases, every block size the library accepts.
SHAPES = [(1, 1, 1, 16), (3, 7, 31, 16), (2, 5, 33, 32), (4, 3, 100, 32),
          (2, 9, 257, 64), (1, 4, 130, 128), (2, 3, 300, 256), (5, 17, 64, 16)]


def _logical(rng, M, N, K, bs, with_zp):
    nb = -(-K // bs)
    Q = rng.integers(0, 16, size=(N, K))
    Z = rng.integers(0, 16, size=(N, nb)) if with_zp else np.full((N, nb), 8)
    return Q, Z, nb


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_integer_exact_brute_force(oracle_lib, shape, with_zp, dtype):
    """Scale 1 and integer A: the exact result is an integer, computed here in
    int64 from the logical codes; the oracle must reproduce it exactly."""
    M, N, K, bs = shape
    rng = np.random.default_rng(hash((shape, with_zp)) % 2**32)
    Q, Z, nb = _logical(rng, M, N, K, bs, with_zp)
    A_int = rng.integers(-3, 4, size=(M, K))
    bias_int = rng.integers(-5, 6, size=N)
    exact = A_int.astype(np.int64) @ (Q - Z[:, np.arange(K) // bs]).T.astype(np.int64)
    exact = exact + bias_int
    B = pack_codes(Q, bs, pad_value=int(rng.integers(0, 16)))
    zp = pack_zero_points(Z, pad_value=int(rng.integers(0, 16))) if with_zp else None
    A = torch.tensor(A_int, dtype=torch.float32).to(dtype)
    S = torch.ones(N, nb, dtype=dtype)
    Y, mag = oracle.matmulnbits(A, B, S, zp, bias_int.astype(np.float32), N=N,
                                K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(Y, exact.astype(np.float64))
    assert np.array_equal(mag, (np.abs(A_int)[:, None, :] * np.abs(
        Q - Z[:, np.arange(K) // bs])[None, :, :]).sum(-1).astype(np.float64))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_matches_dense_float64_gemm(oracle_lib, shape, dtype):
    """Reduction to a textbook dense GEMM: Y = A @ W^T + bias with W from the
    logical codes, computed by numpy in float64."""
    M, N, K, bs = shape
    rng = np.random.default_rng(7 + K)
    Q, Z, nb = _logical(rng, M, N, K, bs, True)
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(K)).to(dtype)
    S = (torch.rand(N, nb, generator=torch.Generator().manual_seed(N)) * 0.02 - 0.005).to(dtype)
    bias = rng.normal(0, 0.02, size=N).astype(np.float32)
    W = dense_weights(Q, Z, S.double().numpy(), bs)
    ref = A.double().numpy() @ W.T + bias.astype(np.float64)
    Y, mag = oracle.matmulnbits(A, pack_codes(Q, bs), S, pack_zero_points(Z),
                                bias, N=N, K=K, block_size=bs, lib=oracle_lib)
    assert np.allclose(Y, ref, rtol=0, atol=1e-12 * (1 + mag.max()))
    assert np.allclose(mag, np.abs(A.double().numpy()[:, None, :] * W[None]).sum(-1),
                       rtol=1e-12, atol=0)


@pytest.mark.parametrize("with_zp", [False, True])
def test_codes_equal_to_zero_point_give_bias(oracle_lib, with_zp):
    M, N, K, bs = 3, 6, 70, 32
    rng = np.random.default_rng(3)
    nb = -(-K // bs)
    Z = rng.integers(0, 16, size=(N, nb)) if with_zp else np.full((N, nb), 8)
    Q = Z[:, np.arange(K) // bs]
    A = torch.randn(M, K)
    S = torch.rand(N, nb) + 0.1
    bias = rng.normal(size=N).astype(np.float32)
    Y, mag = oracle.matmulnbits(A, pack_codes(Q, bs), S,
                                pack_zero_points(Z) if with_zp else None, bias,
                                N=N, K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(Y, np.broadcast_to(bias.astype(np.float64), (M, N)))
    assert not mag.any()


def test_linearity_in_A(oracle_lib):
    M, N, K, bs = 2, 5, 96, 32
    rng = np.random.default_rng(11)
    Q, Z, nb = _logical(rng, M, N, K, bs, True)
    B, zp = pack_codes(Q, bs), pack_zero_points(Z)
    S = torch.rand(N, nb) * 0.02 + 0.005
    bias = rng.normal(size=N).astype(np.float32)
    # dyadic activations keep al*A1 + be*A2 exact in fp32
    A1 = torch.randint(-512, 512, (M, K)).float() / 64
    A2 = torch.randint(-512, 512, (M, K)).float() / 64
    al, be = 0.75, -1.5
    f = lambda A: oracle.matmulnbits(A, B, S, zp, bias, N=N, K=K, block_size=bs,
                                     lib=oracle_lib)[0]
    lhs = f(al * A1 + be * A2)
    rhs = al * f(A1) + be * f(A2) - (al + be - 1) * bias.astype(np.float64)
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)


@pytest.mark.parametrize("with_zp", [False, True])
def test_reblocking_invariance(oracle_lib, with_zp):
    """A bs=128 quantization re-expressed at bs=32 with each scale and zero
    point repeated four times is the same matrix: identical Y, bit for bit."""
    M, N, K = 3, 7, 512
    rng = np.random.default_rng(5)
    Q = rng.integers(0, 16, size=(N, K))
    Z128 = rng.integers(0, 16, size=(N, 4)) if with_zp else np.full((N, 4), 8)
    S128 = torch.rand(N, 4) * 0.02 + 0.005
    A = torch.randn(M, K)
    Y128, _ = oracle.matmulnbits(A, pack_codes(Q, 128), S128,
                                 pack_zero_points(Z128) if with_zp else None,
                                 None, N=N, K=K, block_size=128, lib=oracle_lib)
    Z32 = np.repeat(Z128, 4, axis=1)
    S32 = S128.repeat_interleave(4, dim=1)
    Y32, _ = oracle.matmulnbits(A, pack_codes(Q, 32), S32,
                                pack_zero_points(Z32) if with_zp else None,
                                None, N=N, K=K, block_size=32, lib=oracle_lib)
    assert np.array_equal(Y128, Y32)


def test_nibble_swap_with_activation_permutation(oracle_lib):
    """Swapping the two nibbles of every byte and the matching pair of A
    columns describes the same products."""
    M, N, K, bs = 2, 4, 128, 32
    rng = np.random.default_rng(9)
    Q, Z, nb = _logical(rng, M, N, K, bs, True)
    B = pack_codes(Q, bs)
    Bs = ((B >> 4) | (B << 4)).astype(np.uint8)
    perm = np.arange(K).reshape(-1, 2)[:, ::-1].reshape(-1)
    A = torch.randn(M, K)
    S = torch.rand(N, nb)
    zp = pack_zero_points(Z)
    Y, _ = oracle.matmulnbits(A, B, S, zp, None, N=N, K=K, block_size=bs, lib=oracle_lib)
    Yp, _ = oracle.matmulnbits(A[:, perm].contiguous(), Bs, S, zp, None, N=N, K=K,
                               block_size=bs, lib=oracle_lib)
    assert np.allclose(Y, Yp, rtol=0, atol=1e-12)


def test_padding_nibbles_are_ignored(oracle_lib):
    M, N, K, bs = 2, 3, 40, 32  # last block holds 8 of 32 elements
    rng = np.random.default_rng(2)
    Q, Z, nb = _logical(rng, M, N, K, bs, True)
    A, S = torch.randn(M, K), torch.rand(N, nb)
    outs = [oracle.matmulnbits(A, pack_codes(Q, bs, pad_value=p), S,
                               pack_zero_points(Z), None, N=N, K=K,
                               block_size=bs, lib=oracle_lib)[0] for p in (0, 15)]
    assert np.array_equal(outs[0], outs[1])


def test_bf16_widening_is_exact(oracle_lib):
    M, N, K, bs = 2, 3, 64, 32
    rng = np.random.default_rng(4)
    Q, Z, nb = _logical(rng, M, N, K, bs, False)
    A16 = torch.randn(M, K).to(torch.bfloat16)
    S16 = (torch.rand(N, nb) * 0.02).to(torch.bfloat16)
    B = pack_codes(Q, bs)
    y16, _ = oracle.matmulnbits(A16, B, S16, None, None, N=N, K=K, block_size=bs,
                                lib=oracle_lib)
    y32, _ = oracle.matmulnbits(A16.float(), B, S16.float(), None, None, N=N, K=K,
                                block_size=bs, lib=oracle_lib)
    assert np.array_equal(y16, y32)


def test_row_and_column_sampling(oracle_lib):
    M, N, K, bs = 6, 11, 96, 32
    rng = np.random.default_rng(8)
    Q, Z, nb = _logical(rng, M, N, K, bs, True)
    args = (torch.randn(M, K), pack_codes(Q, bs), torch.rand(N, nb),
            pack_zero_points(Z), rng.normal(size=N).astype(np.float32))
    full, fmag = oracle.matmulnbits(*args, N=N, K=K, block_size=bs, lib=oracle_lib)
    rows, cols = np.array([5, 0, 3]), np.array([10, 2, 2, 7])
    part, pmag = oracle.matmulnbits(*args, N=N, K=K, block_size=bs, rows=rows,
                                    cols=cols, lib=oracle_lib)
    assert np.array_equal(part, full[np.ix_(rows, cols)])
    assert np.array_equal(pmag, fmag[np.ix_(rows, cols)])


# --- mutation checks: plausible slips planted in a copy of the oracle -------

MUTATIONS = {
    "nibble order swapped": ("(within % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
                             "(within % 2 == 0) ? (byte >> 4) : (byte & 0x0F)"),
    "zero-point default 0": ("if (zp == NULL) return 8;", "if (zp == NULL) return 0;"),
    "zero-point nibble order swapped": ("(b % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
                                        "(b % 2 == 0) ? (byte >> 4) : (byte & 0x0F)"),
    "scale indexed by row only": ("widen(scales, n * nb + b, scale_dtype)",
                                  "widen(scales, n * nb, scale_dtype)"),
    "block index off by row stride": ("B[(n * nb + b) * (bs / 2) + within / 2]",
                                      "B[(n + b) * (bs / 2) + within / 2]"),
    "bias dropped": ("if (bias) acc += (double)bias[n];", ""),
    "sign of zero point flipped": ("return (double)(q - z) * s;", "return (double)(q + z) * s;"),
    "zp byte stride uses nb": ("int64_t zbytes = (nb + 1) / 2;", "int64_t zbytes = nb / 2 + 0;"),
}


def _mutant_lib(tmp_path, name, before, after):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(before) == 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", str(path), "-o",
                    str(so), "-lm"], check=True)
    return oracle.load(str(so))


def _pins_pass(lib):
    """The pins above, condensed: returns False as soon as one fails."""
    g = _golden()
    for with_zp, key in ((True, "with_zero_points"), (False, "default_zero_point_8")):
        Y, _ = _run_golden(lib, g, torch.float32, with_zp)
        if Y.tolist() != g[key]["Y"]:
            return False
    for shape in [(2, 5, 33, 32), (3, 9, 257, 64)]:
        M, N, K, bs = shape
        rng = np.random.default_rng(1)
        for with_zp in (False, True):
            Q, Z, nb = _logical(rng, M, N, K, bs, with_zp)
            A_int = rng.integers(-3, 4, size=(M, K))
            exact = A_int @ (Q - Z[:, np.arange(K) // bs]).T
            Y, _ = oracle.matmulnbits(torch.tensor(A_int, dtype=torch.float32),
                                      pack_codes(Q, bs), torch.ones(N, nb),
                                      pack_zero_points(Z) if with_zp else None,
                                      None, N=N, K=K, block_size=bs, lib=lib)
            if not np.array_equal(Y, exact.astype(np.float64)):
                return False
    return True


def test_pins_pass_on_the_real_oracle(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_each_planted_mistake_fails_a_pin(tmp_path, name):
    before, after = MUTATIONS[name]
    lib = _mutant_lib(tmp_path, name, before, after)
    assert not _pins_pass(lib), f"mutation '{name}' survived every pin"
