"""CPU pins of the oracle's QDQ INT4 statement (page "Qwen3 CPU Inference
Critical Path", section "qwen3-int4-qdq": a logical UINT4 initializer in ONNX
row-major, low-nibble-first storage; DequantizeLinear with block_size along
axis 0 for the projections ([K, N] matrix, scales [ceil(K/bs), N]) or axis 1
for the tied LM head ([N, K], scales [N, ceil(K/bs)]); zero points default to
0 when absent).

The test-side packer (tests/packing.py, pack_flat) is written from that
storage description alone (element i of the flattened matrix is nibble i,
low nibble first) and shares no code with the oracle.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from tests.packing import pack_codes, pack_flat, pack_zero_points


SHAPES = [(1, 1, 1, 16), (3, 7, 31, 16), (2, 5, 33, 32), (4, 3, 100, 32),
          (2, 9, 257, 64), (1, 4, 130, 128), (2, 3, 300, 256), (3, 17, 64, 32)]


def _case(rng, M, N, K, bs, with_zp):
    """Logical codes W_q[n,k], zero points Z[n,b] (0 when absent), integer A."""
    nb = -(-K // bs)
    Q = rng.integers(0, 16, size=(N, K))
    Z = rng.integers(0, 16, size=(N, nb)) if with_zp else np.zeros((N, nb), dtype=np.int64)
    A_int = rng.integers(-3, 4, size=(M, K))
    return Q, Z, A_int, nb


def _qdq_inputs(Q, Z, S, axis, with_zp):
    """QDQ storage of the logical weight: axis 0 stores the transposes."""
    if axis == 0:
        return pack_flat(Q.T), np.ascontiguousarray(S.T), (pack_flat(Z.T) if with_zp else None)
    return pack_flat(Q), np.ascontiguousarray(S), (pack_flat(Z) if with_zp else None)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("axis", [0, 1])
@pytest.mark.parametrize("with_zp", [False, True])
def test_qdq_integer_exact_brute_force(oracle_lib, shape, axis, with_zp):
    """Scale 1 and integer A: the exact int64 result of A (Q - Z)^T + bias;
    absent zero points are 0."""
    M, N, K, bs = shape
    rng = np.random.default_rng(hash((shape, axis, with_zp)) % 2**32)
    Q, Z, A_int, nb = _case(rng, M, N, K, bs, with_zp)
    bias = rng.integers(-5, 6, size=N)
    exact = A_int.astype(np.int64) @ (Q - Z[:, np.arange(K) // bs]).T.astype(np.int64) + bias
    Bq, S, zp = _qdq_inputs(Q, Z, np.ones((N, nb), dtype=np.float32), axis, with_zp)
    Y, mag = oracle.qdq_matmul(torch.tensor(A_int, dtype=torch.float32), Bq, S, zp,
                               bias.astype(np.float32), N=N, K=K, block_size=bs, axis=axis,
                               lib=oracle_lib)
    assert np.array_equal(Y, exact.astype(np.float64))
    assert np.array_equal(mag, (np.abs(A_int)[:, None, :] * np.abs(
        Q - Z[:, np.arange(K) // bs])[None, :, :]).sum(-1).astype(np.float64))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_qdq_equals_matmulnbits_of_the_transposed_weight(oracle_lib, shape, with_zp, dtype):
    """The same logical weight stored both ways (QDQ axis 0 and 1, and
    MatMulNBits with explicit zero points) gives bitwise the same Y: the two
    statements add the same products in the same k order."""
    M, N, K, bs = shape
    rng = np.random.default_rng(hash((shape, with_zp, str(dtype))) % 2**32)
    Q, Z, _, nb = _case(rng, M, N, K, bs, with_zp)
    A = torch.randn(M, K, generator=torch.Generator().manual_seed(M + K)).to(dtype)
    S = (torch.rand(N, nb, generator=torch.Generator().manual_seed(N)) * 0.01 + 0.001).to(dtype)
    S_np = S.view(torch.int16).numpy().view(np.uint16) if dtype == torch.bfloat16 else S.numpy()
    ref, rmag = oracle.matmulnbits(A, pack_codes(Q, bs), S, pack_zero_points(Z), None, N=N,
                                   K=K, block_size=bs, lib=oracle_lib)
    for axis in (0, 1):
        Bq, S_q, zp = _qdq_inputs(Q, Z, S_np, axis, with_zp)
        Y, mag = oracle.qdq_matmul(A, Bq, S_q, zp, None, N=N, K=K, block_size=bs, axis=axis,
                                   lib=oracle_lib)
        assert np.array_equal(Y, ref), axis
        assert np.array_equal(mag, rmag), axis


def test_qdq_rejects_a_bad_axis(oracle_lib):
    with pytest.raises(ValueError):
        oracle.qdq_matmul(np.zeros((1, 4), np.float32), np.zeros(2, np.uint8),
                          np.ones((1, 1), np.float32), None, None, N=1, K=4, block_size=16,
                          axis=2, lib=oracle_lib)


# --- planted mistakes in a copy of the oracle's QDQ statement ------------------

MUTATIONS = {
    "code index not transposed on axis 0": ("int64_t ci = axis == 0 ? k * N + n : n * K + k;",
                                            "int64_t ci = n * K + k;"),
    "scale index not transposed on axis 0": ("int64_t si = axis == 0 ? b * N + n : n * nb + b;",
                                             "int64_t si = n * nb + b;"),
    "QDQ nibble order swapped": ("return (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);",
                                 "return (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);"),
    "QDQ zero-point default 8": ("int z = zp ? qdq_nibble(zp, si) : 0;",
                                 "int z = zp ? qdq_nibble(zp, si) : 8;"),
    "QDQ bias dropped": ("if (bias != NULL) acc += (double)bias[n];", ""),
    "QDQ zero point subtracted twice": ("return (double)(q - z) * widen(scales, si, scale_dtype);",
                                        "return (double)(q - 2 * z) * widen(scales, si, scale_dtype);"),
}


def _pins_pass(lib):
    for shape in [(2, 5, 33, 32), (3, 9, 70, 16)]:
        M, N, K, bs = shape
        rng = np.random.default_rng(7)
        for axis in (0, 1):
            for with_zp in (False, True):
                Q, Z, A_int, nb = _case(rng, M, N, K, bs, with_zp)
                bias = rng.integers(-5, 6, size=N)
                exact = A_int @ (Q - Z[:, np.arange(K) // bs]).T + bias
                Bq, S, zp = _qdq_inputs(Q, Z, np.ones((N, nb), dtype=np.float32), axis, with_zp)
                Y, _ = oracle.qdq_matmul(torch.tensor(A_int, dtype=torch.float32), Bq, S, zp,
                                         bias.astype(np.float32), N=N, K=K, block_size=bs,
                                         axis=axis, lib=lib)
                if not np.array_equal(Y, exact.astype(np.float64)):
                    return False
    return True


def test_qdq_pins_pass_on_the_real_oracle(oracle_lib):
    assert _pins_pass(oracle_lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_each_planted_qdq_mistake_fails_a_pin(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert src.count(before) == 1, name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", str(path), "-o", str(so),
                    "-lm"], check=True)
    lib = oracle.load(str(so))
    assert not _pins_pass(lib), f"mutation '{name}' survived every pin"
