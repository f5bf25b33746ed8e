"""CPU pins of the oracle's bitsandbytes-style 4-bit statement (page "Qwen3
CPU Inference Critical Path", com.microsoft operator inventory, row
MatMulBnb4: an alternative bitsandbytes-style 4-bit matrix format to adapt
into the same weight-only plan; the storage readings are listed in the
oracle: the N x K weight flattened row-major, two codes per byte with the
first in the high nibble, one absmax per block_size flattened elements, a
16-value code book, w = code[q] * absmax).

The test-side packer (tests/packing.py, pack_bnb4_flat) is written from that
reading alone and shares no code with the oracle.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.packing import pack_bnb4_flat, pack_codes

SHAPES = [(1, 1, 1, 1), (2, 3, 5, 4), (3, 7, 31, 16), (2, 5, 64, 64), (1, 9, 130, 32),
          (2, 4, 100, 7), (3, 6, 257, 64)]


def _case(rng, M, N, K, bs):
    Q = rng.integers(0, 16, size=(N, K))
    A = rng.integers(-3, 4, size=(M, K))
    nblk = -(-(N * K) // bs)
    return Q, A, nblk


@pytest.mark.parametrize("shape", SHAPES)
def test_integer_code_book_is_exact(oracle_lib, shape):
    """code[q] = q - 7, absmax = 1 or 2, integer A: the exact int64 result,
    with blocks that may straddle rows (K not a multiple of bs)."""
    M, N, K, bs = shape
    rng = np.random.default_rng(hash(shape) % 2**32)
    Q, A, nblk = _case(rng, M, N, K, bs)
    code = (np.arange(16) - 7).astype(np.float32)
    absmax = rng.integers(1, 3, size=nblk).astype(np.float32)
    flat_scale = absmax[np.arange(N * K) // bs].reshape(N, K)
    bias = rng.integers(-4, 5, size=N)
    W = (Q - 7) * flat_scale
    exact = A.astype(np.int64) @ W.T.astype(np.int64) + bias
    Y, mag = oracle.bnb4_matmul(A.astype(np.float32), pack_bnb4_flat(Q), absmax, code,
                                bias.astype(np.float32), N=N, K=K, block_size=bs,
                                lib=oracle_lib)
    assert np.array_equal(Y, exact.astype(np.float64))
    assert np.array_equal(mag, (np.abs(A)[:, None, :] * np.abs(W)[None]).sum(-1))


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_affine_code_book_equals_matmulnbits(oracle_lib, bs, dtype):
    """With code[q] = q - 8 and K a multiple of bs the format is MatMulNBits
    with the default zero point: bitwise the same Y (same products in the
    same k order)."""
    rng = np.random.default_rng(bs)
    M, N, K = 3, 11, 4 * bs
    Q = rng.integers(0, 16, size=(N, K))
    nb = K // bs
    S = torch.rand(N, nb, generator=torch.Generator().manual_seed(bs)) * 0.01 + 0.001
    S = S.to(dtype)
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(bs + 1)).to(dtype)
    code = (np.arange(16) - 8).astype(np.float32)
    absmax = S.reshape(-1)  # block (n, b) is flattened block n*nb + b when K % bs == 0
    Y, mag = oracle.bnb4_matmul(A, pack_bnb4_flat(Q), absmax, code, None, N=N, K=K,
                                block_size=bs, lib=oracle_lib)
    R, rmag = oracle.matmulnbits(A, pack_codes(Q, bs), S, None, None, N=N, K=K, block_size=bs,
                                 lib=oracle_lib)
    assert np.array_equal(Y, R) and np.array_equal(mag, rmag)


def test_zero_code_book_and_zero_activations_give_the_bias(oracle_lib):
    rng = np.random.default_rng(3)
    N, K, bs = 6, 40, 8
    Q = rng.integers(0, 16, size=(N, K))
    bias = rng.standard_normal(N).astype(np.float32)
    absmax = rng.uniform(0.5, 2, size=(N * K) // bs).astype(np.float32)
    Y, _ = oracle.bnb4_matmul(rng.standard_normal((2, K)).astype(np.float32),
                              pack_bnb4_flat(Q), absmax, np.zeros(16, np.float32), bias, N=N,
                              K=K, block_size=bs, lib=oracle_lib)
    assert np.array_equal(Y, np.tile(bias.astype(np.float64), (2, 1)))
    Y, _ = oracle.bnb4_matmul(np.zeros((2, K), np.float32), pack_bnb4_flat(Q), absmax,
                              np.linspace(-1, 1, 16).astype(np.float32), bias, N=N, K=K,
                              block_size=bs, lib=oracle_lib)
    assert np.array_equal(Y, np.tile(bias.astype(np.float64), (2, 1)))


def test_first_code_of_a_byte_is_the_high_nibble(oracle_lib):
    """One byte 0x1F: element 0 is code 1, element 1 is code 15."""
    code = np.arange(16, dtype=np.float32) * 10.0
    Y, _ = oracle.bnb4_matmul(np.array([[1.0, 0.0]], np.float32), np.array([0x1F], np.uint8),
                              np.ones(1, np.float32), code, None, N=1, K=2, block_size=2,
                              lib=oracle_lib)
    assert Y[0, 0] == 10.0
    Y, _ = oracle.bnb4_matmul(np.array([[0.0, 1.0]], np.float32), np.array([0x1F], np.uint8),
                              np.ones(1, np.float32), code, None, N=1, K=2, block_size=2,
                              lib=oracle_lib)
    assert Y[0, 0] == 150.0


MUTATIONS = {
    "low nibble first": ("return (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);",
                         "return (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);"),
    "per-row blocks": ("widen(absmax, flat / bs, absmax_dtype)",
                       "widen(absmax, n * ((K + bs - 1) / bs) + k / bs, absmax_dtype)"),
    "code index off by one": ("(double)code[bnb4_nibble(B, flat)]",
                              "(double)code[(bnb4_nibble(B, flat) + 1) & 15]"),
    "transposed flattening": ("int64_t flat = n * K + k;", "int64_t flat = k * N + n;"),
}


def _pins_pass(lib):
    rng = np.random.default_rng(11)
    for (M, N, K, bs) in [(2, 5, 12, 8), (1, 4, 9, 4)]:
        Q, A, nblk = _case(rng, M, N, K, bs)
        code = (np.arange(16) - 7).astype(np.float32)
        absmax = rng.integers(1, 3, size=nblk).astype(np.float32)
        W = (Q - 7) * absmax[np.arange(N * K) // bs].reshape(N, K)
        exact = A @ W.T
        Y, _ = oracle.bnb4_matmul(A.astype(np.float32), pack_bnb4_flat(Q), absmax, code, None,
                                  N=N, K=K, block_size=bs, lib=lib)
        if not np.array_equal(Y, exact.astype(np.float64)):
            return False
    return True


def test_pins_pass_on_the_real_oracle(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_each_planted_bnb4_mistake_fails_a_pin(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(before) == 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", str(path), "-o", str(so),
                    "-lm"], check=True)
    assert not _pins_pass(oracle.load(str(so))), f"mutation '{name}' survived every pin"
