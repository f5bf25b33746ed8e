"""Test-side packer: logical 4-bit codes -> MatMulNBits byte storage.

Written for the tests from the storage description alone (element k of row n
in byte (k mod bs)/2 of block k/bs, low nibble for even k; zero points two
blocks per byte, low nibble for the even block). It runs in the opposite
direction to the oracle's unpacking and shares no code with it, so an index
or nibble-order slip in either shows up as a mismatch.
"""
import numpy as np


def pack_codes(Q: np.ndarray, block_size: int, pad_value: int = 0) -> np.ndarray:
    """Q int [N, K] in 0..15 -> uint8 [N, nb, bs/2]."""
    N, K = Q.shape
    nb = -(-K // block_size)
    full = np.full((N, nb * block_size), pad_value, dtype=np.uint8)
    full[:, :K] = Q.astype(np.uint8)
    even = full[:, 0::2]
    odd = full[:, 1::2]
    packed = (even | (odd << 4)).astype(np.uint8)
    return packed.reshape(N, nb, block_size // 2)


def pack_zero_points(Z: np.ndarray, pad_value: int = 0) -> np.ndarray:
    """Z int [N, nb] in 0..15 -> uint8 [N, ceil(nb/2)]."""
    N, nb = Z.shape
    full = np.full((N, 2 * (-(-nb // 2))), pad_value, dtype=np.uint8)
    full[:, :nb] = Z.astype(np.uint8)
    return (full[:, 0::2] | (full[:, 1::2] << 4)).astype(np.uint8)


def dense_weights(Q, Z, S, block_size):
    """float64 W[n,k] = (Q[n,k] - Z[n,k//bs]) * S[n,k//bs] from logical arrays."""
    N, K = Q.shape
    blk = np.arange(K) // block_size
    return (Q.astype(np.float64) - Z[:, blk].astype(np.float64)) * S[:, blk].astype(np.float64)


def pack_flat(Q: np.ndarray) -> np.ndarray:
    """Logical UINT4 array (any shape) -> uint8 bytes in ONNX row-major,
    low-nibble-first storage: element i of the flattened array is nibble i;
    an odd count leaves the last high nibble 0."""
    flat = np.asarray(Q, dtype=np.uint8).reshape(-1)
    if flat.size % 2:
        flat = np.concatenate([flat, np.zeros(1, dtype=np.uint8)])
    return (flat[0::2] | (flat[1::2] << 4)).astype(np.uint8)


def pack_bnb4_flat(Q: np.ndarray) -> np.ndarray:
    """Logical 4-bit codes (any shape) -> uint8 bytes with two codes per byte,
    the FIRST of each pair in the HIGH nibble (the bitsandbytes-style order
    read for MatMulBnb4); an odd count leaves the last low nibble 0."""
    flat = np.asarray(Q, dtype=np.uint8).reshape(-1)
    if flat.size % 2:
        flat = np.concatenate([flat, np.zeros(1, dtype=np.uint8)])
    return ((flat[0::2] << 4) | flat[1::2]).astype(np.uint8)
