"""Inputs on which rounding each dequantised weight once to bf16 breaks the
stated bound 2e-3 * sum|a w| + 1e-5.

With bf16 scales, w = (q - z) * s is exact in 12 bits, and its nearest bf16
value can be off by up to 3.86e-3 relative (found by enumerating every
(q - z, s) pair). These problems use two such pairs:
  P blocks:  q - z = 7, s = 1.15625:   w = 8.09375 rounds UP to 8.125,
             paired with a = +r (r a power of two, per row);
  N blocks:  q - z = 3, s = 1.359375:  w = 4.078125 rounds DOWN to 4.0625,
             paired with a = -r.
Every product's rounding error then has the same sign, while the products
themselves nearly cancel (one P block per two N blocks): a single rounding
leaves about 1.9 times the stated bound, yet every value involved is exact
in bf16 and fp32, so an exact split of each weight gives the exact result.

The same for a code book (MatMulBnb4): code values 1 + 3 * 2^-8 (rounds up
to 1 + 2^-6) under a = +r, and 1 + 2^-8 (rounds down to 1) under a = -r, in
alternating blocks.
Only the inputs are built here; the expected values come from the oracle.
"""
import numpy as np
import torch

from int4_weight_only_matmulnbits_gb300.workloads import Problem
from tests.packing import pack_codes, pack_zero_points

P_D, P_S = 7, 1.15625
N_D, N_S = 3, 1.359375


def aligned_rounding_problem(M: int, N: int, block_size: int, repeats: int, *,
                             scale_dtype: torch.dtype, zero_points: bool,
                             seed: int) -> Problem:
    rng = np.random.default_rng(seed)
    nb = 3 * repeats
    K = nb * block_size
    kind = np.tile(np.array([0, 1, 1]), repeats)          # 0 = P block, 1 = N block
    d = np.where(kind == 0, P_D, N_D)
    s = np.where(kind == 0, P_S, N_S)
    r = 2.0 ** rng.integers(-2, 3, size=M)                 # exact in bf16
    sign = np.repeat(np.where(kind == 0, 1.0, -1.0), block_size)
    A = torch.tensor(r[:, None] * sign[None, :], dtype=torch.float32).to(torch.bfloat16)
    if zero_points:
        Z = rng.integers(0, 16 - P_D, size=(N, nb))
    else:
        Z = np.full((N, nb), 8)
    blk = np.arange(K) // block_size
    Q = Z[:, blk] + d[blk][None, :]
    assert Q.max() <= 15
    B = torch.from_numpy(pack_codes(Q, block_size))
    S = torch.tensor(np.broadcast_to(s, (N, nb)).copy(), dtype=torch.float32).to(scale_dtype)
    zp = torch.from_numpy(pack_zero_points(Z)) if zero_points else None
    return Problem(M, N, K, block_size, A, B, S, zp, None)


BNB_UP, BNB_DOWN = 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8


def aligned_rounding_codebook(M: int, N: int, block_size: int, repeats: int, *, seed: int):
    """(A bf16 [M, K], logical codes [N, K], code book fp32 [16]) for the
    code-book form: codes 1 (value BNB_UP) under a = +r and 2 (BNB_DOWN)
    under a = -r, in alternating blocks; other entries arbitrary."""
    rng = np.random.default_rng(seed)
    nb = 2 * repeats
    K = nb * block_size
    kind = np.tile(np.array([0, 1]), repeats)
    r = 2.0 ** rng.integers(-2, 3, size=M)
    sign = np.repeat(np.where(kind == 0, 1.0, -1.0), block_size)
    A = torch.tensor(r[:, None] * sign[None, :], dtype=torch.float32).to(torch.bfloat16)
    Q = np.broadcast_to(np.repeat(np.where(kind == 0, 1, 2), block_size), (N, K)).copy()
    code = torch.tensor(np.linspace(-1.0, 1.0, 16), dtype=torch.float32)
    code[1], code[2] = BNB_UP, BNB_DOWN
    return A, Q, code
