"""MatMulNBits oracle (test infrastructure only).

A ctypes wrapper around ``oracle.c``: a plain double-precision CPU statement
of the weight-only INT4 blockwise MatMul from the page "Qwen3 CPU Inference
Critical Path" (section "Exact kernel inventory", MatMulNBits row; section
"Prepared weight-only plan"). Only the tests, the package smoke check and the
CPU-baseline leg of the benchmark may import this package. It shares no code
with the CUDA library and never imports it.

Arrays are numpy arrays or CPU torch tensors. bf16 data is passed as torch
bfloat16 tensors (or as raw uint16 numpy bit patterns with the dtype named
explicitly); it is widened exactly to double inside the C code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", _SRC,
                    "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load(path: str | None = None):
    """Load the compiled oracle (building it first if needed)."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_matmulnbits.argtypes = [p, i32, p, p, i32, p, p, i64, i64,
                                           i64, i32, p, i64, p, i64, p, p]
        lib.oracle_matmulnbits.restype = i32
        lib.oracle_dequantize.argtypes = [p, p, i32, p, i64, i64, i32, p]
        lib.oracle_dequantize.restype = i32
        lib.oracle_qdq_matmul.argtypes = [p, i32, p, p, i32, p, p, i32, i64, i64,
                                          i64, i32, p, i64, p, i64, p, p]
        lib.oracle_qdq_matmul.restype = i32
        lib.oracle_rms_normalize.argtypes = [p, i32, p, ctypes.c_double, i64, i64, p]
        lib.oracle_rms_normalize.restype = i32
        lib.oracle_bnb4_matmul.argtypes = [p, i32, p, p, i32, p, p, i64, i64, i64, i32, p,
                                           i64, p, i64, p, p]
        lib.oracle_bnb4_matmul.restype = i32
        if path is None:
            _lib = lib
        return lib


def _as_array(x, name):
    """numpy view of x plus its oracle dtype code (F32 or BF16)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float32:
                return x.numpy(), F32
            if x.dtype == torch.float64:
                return x.numpy(), F64
            if x.dtype == torch.uint8:
                return x.numpy(), None
            raise TypeError(f"{name}: unsupported torch dtype {x.dtype}")
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.uint8:
        return x, None
    raise TypeError(f"{name}: unsupported numpy dtype {x.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def matmulnbits(A, B, scales, zero_points=None, bias=None, *, N: int, K: int,
                block_size: int, rows=None, cols=None, lib=None):
    """Y[m,n] = sum_k A[m,k] (q[n,k] - z[n,k/bs]) s[n,k/bs] + bias[n].

    Returns (Y, absdot) as float64 arrays of shape [len(rows), len(cols)]
    (all rows / columns when None), absdot = sum_k |A[m,k] w[n,k]|.
    """
    lib = lib or load()
    a, a_t = _as_array(A, "A")
    b, _ = _as_array(B, "B")
    s, s_t = _as_array(scales, "scales")
    z = None if zero_points is None else _as_array(zero_points, "zero_points")[0]
    bi = None
    if bias is not None:
        bi, bt = _as_array(bias, "bias")
        if bt != F32:
            raise TypeError("bias must be fp32")
    if a.ndim != 2 or a.shape[1] != K:
        raise ValueError("A must be a 2-D [M, K] array")
    M = a.shape[0]
    nb = (K + block_size - 1) // block_size
    if b.size != N * nb * (block_size // 2):
        raise ValueError("B has the wrong number of bytes")
    if s.size != N * nb:
        raise ValueError("scales has the wrong number of elements")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    Y = np.zeros((nr, nc), dtype=np.float64)
    mag = np.zeros((nr, nc), dtype=np.float64)
    rc = lib.oracle_matmulnbits(_ptr(a), a_t, _ptr(b), _ptr(s), s_t, _ptr(z),
                                _ptr(bi), M, N, K, block_size, _ptr(r),
                                0 if r is None else r.size, _ptr(c),
                                0 if c is None else c.size, _ptr(Y), _ptr(mag))
    if rc != 0:
        raise ValueError(f"oracle_matmulnbits rejected its arguments ({rc})")
    return Y, mag


def dequantize(B, scales, zero_points=None, *, N: int, K: int,
               block_size: int, lib=None):
    """W[n,k] = (q[n,k] - z[n,k/bs]) * s[n,k/bs] as a float64 [N, K] array."""
    lib = lib or load()
    b, _ = _as_array(B, "B")
    s, s_t = _as_array(scales, "scales")
    z = None if zero_points is None else _as_array(zero_points, "zero_points")[0]
    W = np.zeros((N, K), dtype=np.float64)
    rc = lib.oracle_dequantize(_ptr(b), _ptr(s), s_t, _ptr(z), N, K,
                               block_size, _ptr(W))
    if rc != 0:
        raise ValueError(f"oracle_dequantize rejected its arguments ({rc})")
    return W


def qdq_matmul(A, Bq, scales, zero_points=None, bias=None, *, N: int, K: int,
               block_size: int, axis: int = 0, rows=None, cols=None, lib=None):
    """Y[m,n] = sum_k A[m,k] w[n,k] + bias[n] for the QDQ INT4 encoding: a
    logical UINT4 matrix ([K, N] for axis 0, [N, K] for axis 1) stored
    flattened, low nibble first, DequantizeLinear along that axis with
    block_size (scales / zero points of the block-reduced shape; absent zero
    points are 0). Returns (Y, absdot) like matmulnbits."""
    lib = lib or load()
    a, a_t = _as_array(A, "A")
    b, _ = _as_array(Bq, "Bq")
    s, s_t = _as_array(scales, "scales")
    z = None if zero_points is None else _as_array(zero_points, "zero_points")[0]
    bi = None
    if bias is not None:
        bi, bt = _as_array(bias, "bias")
        if bt != F32:
            raise TypeError("bias must be fp32")
    if a.ndim != 2 or a.shape[1] != K:
        raise ValueError("A must be a 2-D [M, K] array")
    M = a.shape[0]
    nb = (K + block_size - 1) // block_size
    if b.size != (K * N + 1) // 2:
        raise ValueError("Bq has the wrong number of bytes")
    if s.size != N * nb:
        raise ValueError("scales has the wrong number of elements")
    if z is not None and z.size != (N * nb + 1) // 2:
        raise ValueError("zero_points has the wrong number of bytes")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    Y = np.zeros((nr, nc), dtype=np.float64)
    mag = np.zeros((nr, nc), dtype=np.float64)
    rc = lib.oracle_qdq_matmul(_ptr(a), a_t, _ptr(b), _ptr(s), s_t, _ptr(z), _ptr(bi), axis,
                               M, N, K, block_size, _ptr(r), 0 if r is None else r.size,
                               _ptr(c), 0 if c is None else c.size, _ptr(Y), _ptr(mag))
    if rc != 0:
        raise ValueError(f"oracle_qdq_matmul rejected its arguments ({rc})")
    return Y, mag


def gate_up(A, gate, up, *, N: int, K: int, block_size: int, rows=None, cols=None, lib=None):
    """Gated-MLP pair (page "Qwen3 CPU Inference Critical Path": the fusion
    "gate projection, SiLU, and gate/up multiplication"; SiLU is x * Sigmoid(x)
    in the audited graph): with g = the MatMulNBits result of A and gate and
    u = that of A and up (each a tuple (B, scales, zero_points, bias)),
    Y = g * sigmoid(g) * u, all in double.

    Returns (Y, g, u, absdot_g, absdot_u)."""
    g, mg = matmulnbits(A, *gate, N=N, K=K, block_size=block_size, rows=rows, cols=cols,
                        lib=lib)
    u, mu = matmulnbits(A, *up, N=N, K=K, block_size=block_size, rows=rows, cols=cols,
                        lib=lib)
    sig = 1.0 / (1.0 + np.exp(-g))
    return g * sig * u, g, u, mg, mu


def rms_normalize(A, gamma=None, *, eps: float = 1e-6, lib=None):
    """RMS-style row normalization (page "Qwen3 CPU Inference Critical Path":
    SimplifiedLayerNormalization / RMSNormalization, FP32 over the last axis,
    epsilon 1e-6): out[m,k] = A[m,k] / sqrt(mean_k A[m,k]^2 + eps) * gamma[k],
    in double. Returns a float64 [M, K] array."""
    lib = lib or load()
    a, a_t = _as_array(A, "A")
    if a.ndim != 2:
        raise ValueError("A must be a 2-D [M, K] array")
    M, K = a.shape
    g = None
    if gamma is not None:
        g, gt = _as_array(gamma, "gamma")
        if gt != F32 or g.size != K:
            raise TypeError("gamma must be fp32 [K]")
    out = np.zeros((M, K), dtype=np.float64)
    rc = lib.oracle_rms_normalize(_ptr(a), a_t, _ptr(g), float(eps), M, K, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_rms_normalize rejected its arguments ({rc})")
    return out


def rmsnorm_matmul(A, gamma, eps, B, scales, zero_points=None, bias=None, *, N: int, K: int,
                   block_size: int, rows=None, cols=None, lib=None):
    """The projection of a normalized row (the page's fusion "RMSNorm into
    packed projection input"): matmulnbits of rms_normalize(A, gamma, eps).
    Returns (Y, absdot) with absdot = sum_k |a'[m,k] w[n,k]| over the
    normalized activations a'."""
    An = rms_normalize(A, gamma, eps=eps, lib=lib)
    return matmulnbits(An, B, scales, zero_points, bias, N=N, K=K, block_size=block_size,
                       rows=rows, cols=cols, lib=lib)


def lm_head_argmax(Y):
    """Greedy token choice (the page's fusion "final RMSNorm, LM-head GEMV, and
    greedy ArgMax"): the index of the largest logit of each row, the first
    one on ties (numpy's argmax)."""
    return np.argmax(np.asarray(Y), axis=1)


def bnb4_matmul(A, B, absmax, code, bias=None, *, N: int, K: int, block_size: int, rows=None,
                cols=None, lib=None):
    """The bitsandbytes-style 4-bit matrix (page "Qwen3 CPU Inference Critical
    Path", MatMulBnb4 row): B is the N x K weight flattened row-major, two
    codes per byte with the first in the high nibble; absmax holds one scale
    per block_size consecutive flattened elements; code is the 16-value fp32
    code book; w[n,k] = code[q] * absmax. Returns (Y, absdot) like
    matmulnbits."""
    lib = lib or load()
    a, a_t = _as_array(A, "A")
    b, _ = _as_array(B, "B")
    s, s_t = _as_array(absmax, "absmax")
    c, c_t = _as_array(code, "code")
    if c_t != F32 or c.size != 16:
        raise TypeError("code must be 16 fp32 values")
    bi = None
    if bias is not None:
        bi, bt = _as_array(bias, "bias")
        if bt != F32:
            raise TypeError("bias must be fp32")
    if a.ndim != 2 or a.shape[1] != K:
        raise ValueError("A must be a 2-D [M, K] array")
    M = a.shape[0]
    if b.size != (N * K + 1) // 2:
        raise ValueError("B has the wrong number of bytes")
    if s.size != -(-(N * K) // block_size):
        raise ValueError("absmax has the wrong number of elements")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cc = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if cc is None else cc.size
    Y = np.zeros((nr, nc), dtype=np.float64)
    mag = np.zeros((nr, nc), dtype=np.float64)
    rc = lib.oracle_bnb4_matmul(_ptr(a), a_t, _ptr(b), _ptr(s), s_t, _ptr(c), _ptr(bi), M, N,
                                K, block_size, _ptr(r), 0 if r is None else r.size, _ptr(cc),
                                0 if cc is None else cc.size, _ptr(Y), _ptr(mag))
    if rc != 0:
        raise ValueError(f"oracle_bnb4_matmul rejected its arguments ({rc})")
    return Y, mag
