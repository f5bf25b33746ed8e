"""Thin ctypes binding of libmnb.so (include/mnb.h), same names as the C ABI.

Argument marshalling only: tensors are turned into device pointers, outputs
are allocated with torch (device memory is plumbing here), and every
computation runs in the library's CUDA kernels. A missing library raises
immediately; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import torch

from . import _build

MNB_OK = 0
MNB_ERR_NULL = -1
MNB_ERR_SHAPE = -2
MNB_ERR_BLOCKSIZE = -3
MNB_ERR_DTYPE = -4
MNB_ERR_ALIGN = -5
MNB_ERR_ALIAS = -6
MNB_ERR_CUDA = -7
MNB_ERR_UNSUPPORTED = -8
MNB_ERR_DEVICE = -9
MNB_ERR_LAYOUT = -10
MNB_CODES_AFFINE, MNB_CODES_CODEBOOK = 0, 1
MNB_PACKED_MAGIC = 0x4B43415034424E4D
MNB_PACKED_HEADER_BYTES = 256
MNB_F32, MNB_BF16 = 0, 1
MNB_PATH = {"auto": 0, "gemv": 1, "gemm": 2, "gemm_streamk": 3, "gemm_pair": 4}

# Every entry point include/mnb.h declares.
EXPORTS = ("mnb_status_string", "mnb_last_error_string", "mnb_version",
           "mnb_prepacked_sizes", "mnb_prepack", "mnb_unprepack", "mnb_matmul",
           "mnb_matmul_path", "mnb_matmul_from_host",
           "mnb_set_programmatic_launch", "mnb_fault_status", "mnb_matmul_grouped",
           "mnb_prepack_qdq", "mnb_matmul_gate_up", "mnb_chain_build", "mnb_chain_run", "mnb_chain_run_noalloc",
           "mnb_matmul_rmsnorm", "mnb_prepack_bnb4", "mnb_matmul_bnb4",
           "mnb_matmul_workspace_size", "mnb_matmul_ws", "mnb_matmul_plan",
           "mnb_packed_header_make", "mnb_packed_register", "mnb_packed_read_header",
           "mnb_packed_forget", "mnb_graph_build", "mnb_graph_info", "mnb_graph_run",
           "mnb_graph_run_from_host", "mnb_graph_destroy", "mnb_test_wait_fault")

_lock = threading.Lock()
_lib = None


class PlanInfoC(ctypes.Structure):
    """mnb_matmul_plan_info (include/mnb.h)."""
    _fields_ = [("path", ctypes.c_int32), ("m_slices", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("k_split", ctypes.c_int32),
                ("stream_k", ctypes.c_int32), ("tf32", ctypes.c_int32),
                ("tma_store", ctypes.c_int32), ("pair_cols", ctypes.c_int32),
                ("ctas", ctypes.c_int64)]


class PackedHeaderC(ctypes.Structure):
    """mnb_packed_header (include/mnb.h)."""
    _fields_ = [("magic", ctypes.c_uint64), ("version", ctypes.c_uint32),
                ("codes", ctypes.c_uint32), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("scale_dtype", ctypes.c_int32),
                ("has_zero_points", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("packed_b_bytes", ctypes.c_uint64), ("packed_scales_bytes", ctypes.c_uint64),
                ("packed_zp_bytes", ctypes.c_uint64), ("check", ctypes.c_uint64)]


class ChainOpC(ctypes.Structure):
    """mnb_chain_op (include/mnb.h)."""
    _fields_ = [("A", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("packed_b", ctypes.c_void_p), ("packed_scales", ctypes.c_void_p),
                ("packed_zp", ctypes.c_void_p), ("bias", ctypes.c_void_p),
                ("packed_b_up", ctypes.c_void_p), ("packed_scales_up", ctypes.c_void_p),
                ("packed_zp_up", ctypes.c_void_p), ("bias_up", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("deps", ctypes.c_int32 * 4)]


class ChainInfoC(ctypes.Structure):
    """mnb_chain_info (include/mnb.h)."""
    _fields_ = [("plan_bytes", ctypes.c_uint64)] + [
        (f, ctypes.c_int32) for f in ("n_ops", "n_segments", "grid", "smem_bytes", "M",
                                      "block_size", "a_dtype", "scale_dtype",
                                      "has_zero_points", "ring_stages", "k_max",
                                      "tiles_per_segment", "ctas_per_sm")] + [
        ("check", ctypes.c_uint64)]


class MnbError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        msg = f"{where}: {status_string(status)}"
        if detail:
            msg += f" [{detail}]"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load libmnb.so and declare its signatures. Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            _build.build_library()
        lib = ctypes.CDLL(path)
        p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        lib.mnb_status_string.argtypes = [i32]
        lib.mnb_status_string.restype = ctypes.c_char_p
        lib.mnb_last_error_string.argtypes = []
        lib.mnb_last_error_string.restype = ctypes.c_char_p
        lib.mnb_version.argtypes = []
        lib.mnb_version.restype = i32
        lib.mnb_prepacked_sizes.argtypes = [i64, i64, i32, i32, i32,
                                            ctypes.POINTER(sz), ctypes.POINTER(sz),
                                            ctypes.POINTER(sz)]
        lib.mnb_prepacked_sizes.restype = i32
        lib.mnb_prepack.argtypes = [p, p, p, i64, i64, i32, i32, p, p, p, p]
        lib.mnb_prepack.restype = i32
        lib.mnb_matmul_gate_up.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i64, i32, p,
                                           i32, i32, p]
        lib.mnb_matmul_gate_up.restype = i32
        lib.mnb_prepack_qdq.argtypes = [p, p, p, i32, i64, i64, i32, i32, p, p, p, p]
        lib.mnb_prepack_qdq.restype = i32
        lib.mnb_unprepack.argtypes = [p, p, p, i64, i64, i32, i32, p, p, p, p]
        lib.mnb_unprepack.restype = i32
        lib.mnb_matmul.argtypes = [p, p, p, p, p, i64, i64, i64, i32, p, i32, i32, p]
        lib.mnb_matmul.restype = i32
        lib.mnb_matmul_path.argtypes = [p, p, p, p, p, i64, i64, i64, i32, p, i32,
                                        i32, i32, p]
        lib.mnb_matmul_path.restype = i32
        lib.mnb_matmul_workspace_size.argtypes = []
        lib.mnb_matmul_workspace_size.restype = sz
        lib.mnb_matmul_ws.argtypes = [p, p, p, p, p, i64, i64, i64, i32, p, i32, i32, i32, p,
                                      sz, p]
        lib.mnb_matmul_ws.restype = i32
        lib.mnb_matmul_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, sz, i32,
                                        ctypes.POINTER(PlanInfoC)]
        lib.mnb_matmul_plan.restype = i32
        lib.mnb_matmul_from_host.argtypes = [p, p, p, p, p, p, i64, i64, i64, i32,
                                             p, p, i32, i32, p]
        lib.mnb_matmul_from_host.restype = i32
        lib.mnb_set_programmatic_launch.argtypes = [i32]
        lib.mnb_set_programmatic_launch.restype = None
        lib.mnb_matmul_grouped.argtypes = [p, i32, p, p, p, p, p, p, i64, i64, i32,
                                           i32, i32, p]
        lib.mnb_matmul_grouped.restype = i32
        lib.mnb_fault_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.mnb_fault_status.restype = i32
        lib.mnb_chain_build.argtypes = [ctypes.POINTER(ChainOpC), i32, i64, i32, i32, i32, p,
                                        sz, ctypes.POINTER(ChainInfoC), p]
        lib.mnb_chain_build.restype = i32
        lib.mnb_chain_run.argtypes = [p, ctypes.POINTER(ChainInfoC), p]
        lib.mnb_chain_run.restype = i32
        lib.mnb_chain_run_noalloc.argtypes = [ctypes.POINTER(ChainOpC), i32, i64, i32, i32,
                                              i32, p]
        lib.mnb_chain_run_noalloc.restype = i32
        lib.mnb_matmul_rmsnorm.argtypes = [p, i32, p, ctypes.c_float, p, p, p, p, i64, i64,
                                           i64, i32, p, p, i32, i32, p]
        lib.mnb_matmul_rmsnorm.restype = i32
        lib.mnb_packed_header_make.argtypes = [i64, i64, i32, i32, i32, i32,
                                               ctypes.POINTER(PackedHeaderC)]
        lib.mnb_packed_header_make.restype = i32
        lib.mnb_packed_register.argtypes = [p, ctypes.POINTER(PackedHeaderC)]
        lib.mnb_packed_register.restype = i32
        lib.mnb_packed_read_header.argtypes = [p, sz, ctypes.POINTER(PackedHeaderC), p]
        lib.mnb_packed_read_header.restype = i32
        lib.mnb_packed_forget.argtypes = [p]
        lib.mnb_packed_forget.restype = i32
        lib.mnb_graph_build.argtypes = [ctypes.POINTER(ChainOpC), i32, i64, i32, i32, i32,
                                        ctypes.POINTER(p)]
        lib.mnb_graph_build.restype = i32
        lib.mnb_graph_info.argtypes = [p, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.POINTER(ctypes.c_int32)]
        lib.mnb_graph_info.restype = i32
        lib.mnb_graph_run.argtypes = [p, p]
        lib.mnb_graph_run.restype = i32
        lib.mnb_graph_run_from_host.argtypes = [p, p, p, sz, p, p, sz, p]
        lib.mnb_graph_run_from_host.restype = i32
        lib.mnb_test_wait_fault.argtypes = [i32]
        lib.mnb_test_wait_fault.restype = None
        lib.mnb_graph_destroy.argtypes = [p]
        lib.mnb_graph_destroy.restype = i32
        lib.mnb_prepack_bnb4.argtypes = [p, p, i64, i64, i32, i32, p, p, p]
        lib.mnb_prepack_bnb4.restype = i32
        lib.mnb_matmul_bnb4.argtypes = [p, p, p, p, p, i64, i64, i64, i32, p, i32, i32, p]
        lib.mnb_matmul_bnb4.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().mnb_status_string(status).decode()


def _check(status: int, where: str):
    if status != MNB_OK:
        detail = load().mnb_last_error_string().decode()
        raise MnbError(status, where, detail)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return MNB_F32
    if dt == torch.bfloat16:
        return MNB_BF16
    raise TypeError(f"unsupported dtype {dt}: fp32 or bf16")


@dataclass
class PackedWeight:
    """Caller-owned prepacked buffers of one N x K MatMulNBits weight."""
    packed_b: torch.Tensor
    packed_scales: torch.Tensor
    packed_zp: torch.Tensor | None
    N: int
    K: int
    block_size: int
    scale_dtype: torch.dtype

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.packed_b, self.packed_scales, self.packed_zp) if t is not None)


def mnb_version() -> int:
    return load().mnb_version()


def mnb_set_programmatic_launch(enable: bool) -> None:
    load().mnb_set_programmatic_launch(1 if enable else 0)


def mnb_test_wait_fault(stop_stage: int = -1) -> None:
    """Test-only failure injection in the decode kernel (see include/mnb.h);
    the default turns it off."""
    load().mnb_test_wait_fault(stop_stage)


def mnb_fault_status() -> int:
    """Fault bits recorded by kernels whose bounded waits ran out (cleared)."""
    v = ctypes.c_uint()
    _check(load().mnb_fault_status(ctypes.byref(v)), "mnb_fault_status")
    return v.value


def mnb_prepacked_sizes(N: int, K: int, block_size: int, scale_dtype: torch.dtype,
                        has_zero_points: bool) -> tuple[int, int, int]:
    b, s, z = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mnb_prepacked_sizes(N, K, block_size, _dtype_code(scale_dtype),
                                      int(has_zero_points), ctypes.byref(b),
                                      ctypes.byref(s), ctypes.byref(z)),
           "mnb_prepacked_sizes")
    return b.value, s.value, z.value


def mnb_prepack(B: torch.Tensor, scales: torch.Tensor, zero_points: torch.Tensor | None,
                N: int, K: int, block_size: int, *, stream=None) -> PackedWeight:
    """Prepack one weight given in MatMulNBits layout (device tensors)."""
    for name, t in (("B", B), ("scales", scales), ("zero_points", zero_points)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    sb, ss, sz = mnb_prepacked_sizes(N, K, block_size, scales.dtype,
                                     zero_points is not None)
    dev = B.device
    packed_b = torch.empty(sb, dtype=torch.uint8, device=dev)
    packed_s = torch.empty(ss, dtype=torch.uint8, device=dev)
    packed_z = (torch.empty(sz, dtype=torch.uint8, device=dev)
                if zero_points is not None else None)
    _check(load().mnb_prepack(_ptr(B), _ptr(scales), _ptr(zero_points), N, K, block_size,
                              _dtype_code(scales.dtype), _ptr(packed_b), _ptr(packed_s),
                              _ptr(packed_z), _stream(stream)), "mnb_prepack")
    return PackedWeight(packed_b, packed_s, packed_z, N, K, block_size, scales.dtype)


def mnb_prepack_qdq(B_qdq: torch.Tensor, scales: torch.Tensor,
                    zero_points: torch.Tensor | None, N: int, K: int, block_size: int, *,
                    axis: int = 0, stream=None) -> PackedWeight:
    """Prepack one weight given in the QDQ INT4 encoding (device tensors): a
    logical UINT4 [K, N] (axis 0) or [N, K] (axis 1) matrix stored flattened
    low-nibble-first, scales / zero points of the block-reduced shape, absent
    zero points meaning 0. The result always carries packed zero points."""
    for name, t in (("B_qdq", B_qdq), ("scales", scales), ("zero_points", zero_points)):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    sb, ss, sz = mnb_prepacked_sizes(N, K, block_size, scales.dtype, True)
    dev = B_qdq.device
    packed_b = torch.empty(sb, dtype=torch.uint8, device=dev)
    packed_s = torch.empty(ss, dtype=torch.uint8, device=dev)
    packed_z = torch.empty(sz, dtype=torch.uint8, device=dev)
    _check(load().mnb_prepack_qdq(_ptr(B_qdq), _ptr(scales), _ptr(zero_points), axis, N, K,
                                  block_size, _dtype_code(scales.dtype), _ptr(packed_b),
                                  _ptr(packed_s), _ptr(packed_z), _stream(stream)),
           "mnb_prepack_qdq")
    return PackedWeight(packed_b, packed_s, packed_z, N, K, block_size, scales.dtype)


def mnb_packed_header_make(N: int, K: int, block_size: int, scale_dtype: torch.dtype,
                           has_zero_points: bool, codes: int = MNB_CODES_AFFINE) -> PackedHeaderC:
    """The header a prepack call writes for these arguments (host only)."""
    h = PackedHeaderC()
    _check(load().mnb_packed_header_make(N, K, block_size, _dtype_code(scale_dtype),
                                         int(has_zero_points), codes, ctypes.byref(h)),
           "mnb_packed_header_make")
    return h


def mnb_packed_read_header(w: PackedWeight | torch.Tensor, *, stream=None) -> PackedHeaderC:
    """The header stored at the end of a packed_b buffer (read from the device)."""
    pb = w.packed_b if isinstance(w, PackedWeight) else w
    h = PackedHeaderC()
    _check(load().mnb_packed_read_header(_ptr(pb), pb.numel() * pb.element_size(),
                                         ctypes.byref(h), _stream(stream)),
           "mnb_packed_read_header")
    return h


def mnb_packed_register(packed_b: torch.Tensor | int, header: PackedHeaderC) -> None:
    """Record `header` for the packed weight at packed_b (a restored weight)."""
    ptr = ctypes.c_void_p(packed_b) if isinstance(packed_b, int) else _ptr(packed_b)
    _check(load().mnb_packed_register(ptr, ctypes.byref(header)), "mnb_packed_register")


def mnb_packed_forget(packed_b: torch.Tensor | int) -> None:
    ptr = ctypes.c_void_p(packed_b) if isinstance(packed_b, int) else _ptr(packed_b)
    _check(load().mnb_packed_forget(ptr), "mnb_packed_forget")


def mnb_unprepack(w: PackedWeight, *, stream=None):
    """Recover (B, scales, zero_points) in MatMulNBits layout from w."""
    nb = -(-w.K // w.block_size)
    dev = w.packed_b.device
    B = torch.empty(w.N, nb, w.block_size // 2, dtype=torch.uint8, device=dev)
    S = torch.empty(w.N, nb, dtype=w.scale_dtype, device=dev)
    Z = (torch.empty(w.N, (nb + 1) // 2, dtype=torch.uint8, device=dev)
         if w.packed_zp is not None else None)
    _check(load().mnb_unprepack(_ptr(w.packed_b), _ptr(w.packed_scales), _ptr(w.packed_zp),
                                w.N, w.K, w.block_size, _dtype_code(w.scale_dtype),
                                _ptr(B), _ptr(S), _ptr(Z), _stream(stream)),
           "mnb_unprepack")
    return B, S, Z


def mnb_matmul_plan(M: int, N: int, K: int, block_size: int, *,
                    a_dtype: torch.dtype = torch.bfloat16,
                    scale_dtype: torch.dtype | None = None, zero_points: bool = False,
                    path: str = "auto", workspace_bytes: int = 0,
                    sm_count: int = 0) -> dict:
    """What mnb_matmul(..., workspace) would launch (host arithmetic only):
    {"path": "gemv" | "gemm", "m_slices", "tile_rows", "k_split", "stream_k",
    "tf32", "tma_store", "pair_cols", "ctas"}; pair_cols > 0 names the
    persistent CTA-pair kernel and its tile width. sm_count 0 asks the current
    device."""
    info = PlanInfoC()
    sd = a_dtype if scale_dtype is None else scale_dtype
    _check(load().mnb_matmul_plan(M, N, K, block_size, _dtype_code(a_dtype), _dtype_code(sd),
                                  int(bool(zero_points)), MNB_PATH[path], workspace_bytes,
                                  sm_count, ctypes.byref(info)), "mnb_matmul_plan")
    return {"path": "gemv" if info.path == MNB_PATH["gemv"] else "gemm",
            "m_slices": info.m_slices, "tile_rows": info.tile_rows,
            "k_split": info.k_split, "stream_k": bool(info.stream_k), "tf32": bool(info.tf32),
            "tma_store": bool(info.tma_store), "pair_cols": info.pair_cols, "ctas": info.ctas}


def mnb_matmul_workspace(device=None) -> torch.Tensor:
    """A zero-filled workspace for mnb_matmul's stream-K schedule on `device`
    (mnb_matmul_workspace_size() bytes). Calls that use one must be ordered
    one after another (one stream, or a CUDA graph)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    with torch.cuda.device(dev):
        n = load().mnb_matmul_workspace_size()
    if n == 0:
        raise MnbError(MNB_ERR_DEVICE, "mnb_matmul_workspace", "no usable CUDA device")
    return torch.zeros(n, dtype=torch.uint8, device=dev)


# One workspace per (device, stream): calls on one stream run one after another.
_workspaces: dict = {}


def _default_workspace(A: torch.Tensor, stream) -> torch.Tensor:
    s = torch.cuda.current_stream(A.device) if stream is None else stream
    key = (A.device.index, s.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None:
        ws = _workspaces[key] = mnb_matmul_workspace(A.device)
    return ws


def mnb_matmul(A: torch.Tensor, w: PackedWeight, bias: torch.Tensor | None = None, *,
               out: torch.Tensor | None = None, path: str = "auto", workspace="auto",
               stream=None) -> torch.Tensor:
    """Y[M, N] = A[M, K] @ dequant(w)^T + bias, on the GPU.

    workspace: "auto" (above 16 rows: a zero-filled workspace kept per device
    and stream, which lets the tensor-core kernel use its stream-K schedule
    where that is faster), None (no workspace: whole-tile CTAs only), or a
    tensor from mnb_matmul_workspace()."""
    if A.dim() != 2 or A.shape[1] != w.K:
        raise ValueError(f"A must be [M, {w.K}]")
    if not A.is_cuda or not A.is_contiguous():
        raise ValueError("A must be a contiguous CUDA tensor")
    M = A.shape[0]
    if out is None:
        out = torch.empty(M, w.N, dtype=A.dtype, device=A.device)
    if bias is not None and (bias.dtype != torch.float32 or not bias.is_cuda):
        raise ValueError("bias must be a CUDA float32 tensor")
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a tensor')
        workspace = _default_workspace(A, stream) if M > 16 and path != "gemv" else None
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().mnb_matmul_ws(_ptr(A), _ptr(w.packed_b), _ptr(w.packed_scales),
                                _ptr(w.packed_zp), _ptr(bias), M, w.N, w.K,
                                w.block_size, _ptr(out), _dtype_code(A.dtype),
                                _dtype_code(w.scale_dtype), MNB_PATH[path],
                                _ptr(workspace), ws_bytes, _stream(stream)), "mnb_matmul")
    return out


def mnb_matmul_from_host(A_host: torch.Tensor, A_dev: torch.Tensor, w: PackedWeight,
                         Y_dev: torch.Tensor, Y_host: torch.Tensor,
                         bias: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """Host A in, host Y out: copies and product enqueued on one stream."""
    M = A_host.shape[0]
    _check(load().mnb_matmul_from_host(
        _ptr(A_host), _ptr(A_dev), _ptr(w.packed_b), _ptr(w.packed_scales),
        _ptr(w.packed_zp), _ptr(bias), M, w.N, w.K, w.block_size, _ptr(Y_dev),
        _ptr(Y_host), _dtype_code(A_host.dtype), _dtype_code(w.scale_dtype),
        _stream(stream)), "mnb_matmul_from_host")
    return Y_host


def mnb_matmul_grouped(A: torch.Tensor, ws: list[PackedWeight],
                       biases: list[torch.Tensor | None] | None = None, *,
                       outs: list[torch.Tensor] | None = None,
                       stream=None) -> list[torch.Tensor]:
    """Fused-N projections: [A @ dequant(w)^T + b for w, b in zip(ws, biases)]."""
    n = len(ws)
    if A.dim() != 2 or not A.is_cuda or not A.is_contiguous():
        raise ValueError("A must be a contiguous 2-D CUDA tensor")
    M, K = A.shape
    if any(w.K != K or w.block_size != ws[0].block_size or
           w.scale_dtype != ws[0].scale_dtype for w in ws):
        raise ValueError("grouped weights must share K, block size and scale dtype")
    if outs is None:
        outs = [torch.empty(M, w.N, dtype=A.dtype, device=A.device) for w in ws]
    biases = biases or [None] * n
    VP = ctypes.c_void_p * n
    vp = lambda ts: VP(*[None if t is None else t.data_ptr() for t in ts])
    zps = [w.packed_zp for w in ws]
    _check(load().mnb_matmul_grouped(
        _ptr(A), n, vp([w.packed_b for w in ws]), vp([w.packed_scales for w in ws]),
        None if zps[0] is None else vp(zps), vp(biases),
        (ctypes.c_int64 * n)(*[w.N for w in ws]), vp(outs), M, K, ws[0].block_size,
        _dtype_code(A.dtype), _dtype_code(ws[0].scale_dtype), _stream(stream)),
        "mnb_matmul_grouped")
    return outs


def mnb_matmul_gate_up(A: torch.Tensor, gate: PackedWeight, up: PackedWeight,
                       bias_gate: torch.Tensor | None = None,
                       bias_up: torch.Tensor | None = None, *,
                       out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = silu(A @ gate^T + bias_gate) * (A @ up^T + bias_up), silu(x) =
    x * sigmoid(x), in one launch per 16 rows."""
    if (gate.N, gate.K, gate.block_size, gate.scale_dtype) != (up.N, up.K, up.block_size,
                                                              up.scale_dtype):
        raise ValueError("gate and up must have the same N, K, block size and scale dtype")
    if A.dim() != 2 or A.shape[1] != gate.K or not A.is_cuda or not A.is_contiguous():
        raise ValueError(f"A must be a contiguous CUDA [M, {gate.K}] tensor")
    for b in (bias_gate, bias_up):
        if b is not None and (b.dtype != torch.float32 or not b.is_cuda):
            raise ValueError("biases must be fp32 CUDA tensors")
    M = A.shape[0]
    if out is None:
        out = torch.empty(M, gate.N, dtype=A.dtype, device=A.device)
    _check(load().mnb_matmul_gate_up(
        _ptr(A), _ptr(gate.packed_b), _ptr(gate.packed_scales), _ptr(gate.packed_zp),
        _ptr(bias_gate), _ptr(up.packed_b), _ptr(up.packed_scales), _ptr(up.packed_zp),
        _ptr(bias_up), M, gate.N, gate.K, gate.block_size, _ptr(out), _dtype_code(A.dtype),
        _dtype_code(gate.scale_dtype), _stream(stream)), "mnb_matmul_gate_up")
    return out


@dataclass
class ChainOp:
    """One projection of a decode chain: out = A @ dequant(weight)^T + bias,
    or, with `up`, silu(A @ gate^T + bias) * (A @ up^T + bias_up). `deps`
    lists earlier ops (indices) whose outputs must be complete before this
    op reads A."""
    A: torch.Tensor
    weight: PackedWeight
    out: torch.Tensor
    bias: torch.Tensor | None = None
    up: PackedWeight | None = None
    bias_up: torch.Tensor | None = None
    deps: tuple = ()


class MnbChain:
    """A built decode chain: the device plan buffer (torch-allocated) and its
    launch description. Holds references to every tensor of its ops."""

    def __init__(self, ops: list, plan: torch.Tensor, info: ChainInfoC):
        self.ops = list(ops)
        self.plan = plan
        self.info = info

    def describe(self) -> dict:
        return {f: getattr(self.info, f) for f, _ in ChainInfoC._fields_}

    def run(self, stream=None) -> None:
        mnb_chain_run(self, stream=stream)


def _chain_structs(ops: list):
    arr = (ChainOpC * len(ops))()
    first = ops[0]
    M = first.A.shape[0]
    for j, o in enumerate(ops):
        w, up = o.weight, o.up
        if o.A.dim() != 2 or o.A.shape != (M, w.K) or not o.A.is_contiguous():
            raise ValueError(f"op {j}: A must be a contiguous [{M}, {w.K}] tensor")
        if o.out.shape != (M, w.N) or o.out.dtype != first.A.dtype or not o.out.is_contiguous():
            raise ValueError(f"op {j}: out must be a contiguous [{M}, {w.N}] tensor of A's dtype")
        if len(o.deps) > 4:
            raise ValueError(f"op {j}: at most 4 deps")
        if up is not None and (up.N, up.K) != (w.N, w.K):
            raise ValueError(f"op {j}: up must match the gate's N and K")
        deps = list(o.deps) + [-1] * (4 - len(o.deps))
        c = arr[j]
        c.A, c.Y = o.A.data_ptr(), o.out.data_ptr()
        c.packed_b, c.packed_scales = w.packed_b.data_ptr(), w.packed_scales.data_ptr()
        c.packed_zp = None if w.packed_zp is None else w.packed_zp.data_ptr()
        c.bias = None if o.bias is None else o.bias.data_ptr()
        if up is not None:
            c.packed_b_up, c.packed_scales_up = up.packed_b.data_ptr(), up.packed_scales.data_ptr()
            c.packed_zp_up = None if up.packed_zp is None else up.packed_zp.data_ptr()
            c.bias_up = None if o.bias_up is None else o.bias_up.data_ptr()
        c.N, c.K = w.N, w.K
        for k in range(4):
            c.deps[k] = deps[k]
    return arr, M


def mnb_chain_build(ops: list, *, stream=None) -> MnbChain:
    """Plan a chain of projections (one persistent launch per run). All ops
    share the block size, activation dtype, scale dtype and zero-point
    presence; M (rows of A) is 1..8."""
    if not ops:
        raise ValueError("empty chain")
    lib = load()
    arr, M = _chain_structs(ops)
    w0 = ops[0].weight
    info = ChainInfoC()
    args = (arr, len(ops), M, w0.block_size, _dtype_code(ops[0].A.dtype),
            _dtype_code(w0.scale_dtype))
    _check(lib.mnb_chain_build(*args, None, 0, ctypes.byref(info), _stream(stream)),
           "mnb_chain_build")
    plan = torch.empty(int(info.plan_bytes), dtype=torch.uint8, device=ops[0].A.device)
    _check(lib.mnb_chain_build(*args, ctypes.c_void_p(plan.data_ptr()), plan.numel(),
                               ctypes.byref(info), _stream(stream)), "mnb_chain_build")
    return MnbChain(ops, plan, info)


def mnb_chain_run(chain: MnbChain, *, stream=None) -> None:
    """Run every op of a built chain in one cooperative launch on `stream`."""
    _check(load().mnb_chain_run(ctypes.c_void_p(chain.plan.data_ptr()), ctypes.byref(chain.info),
                                _stream(stream)), "mnb_chain_run")


class MnbGraph:
    """A sequence of projections recorded as one CUDA graph by the library
    (mnb_graph_build). Holds references to every tensor of its ops; the graph
    reads their current contents each run."""

    def __init__(self, ops: list, handle: int):
        self.ops = list(ops)
        self._handle = ctypes.c_void_p(handle)
        calls, kernels = ctypes.c_int32(), ctypes.c_int32()
        _check(load().mnb_graph_info(self._handle, ctypes.byref(calls), ctypes.byref(kernels)),
               "mnb_graph_info")
        self.calls, self.kernels = calls.value, kernels.value

    def run(self, stream=None) -> None:
        _check(load().mnb_graph_run(self._handle, _stream(stream)), "mnb_graph_run")

    def run_from_host(self, in_host: torch.Tensor | None, in_dev: torch.Tensor | None,
                      out_dev: torch.Tensor | None, out_host: torch.Tensor | None,
                      stream=None) -> None:
        """Copy in_host -> in_dev, run, copy out_dev -> out_host (one stream)."""
        nb = lambda t: 0 if t is None else t.numel() * t.element_size()
        if nb(in_host) != nb(in_dev) or nb(out_dev) != nb(out_host):
            raise ValueError("host and device buffers of a copy must have the same size")
        _check(load().mnb_graph_run_from_host(self._handle, _ptr(in_host), _ptr(in_dev),
                                              nb(in_dev), _ptr(out_dev), _ptr(out_host),
                                              nb(out_dev), _stream(stream)),
               "mnb_graph_run_from_host")

    def __del__(self):
        if getattr(self, "_handle", None) and self._handle.value and _lib is not None:
            _lib.mnb_graph_destroy(self._handle)
            self._handle = None


def mnb_graph_build(ops: list) -> MnbGraph:
    """Record the projections `ops` (ChainOp; run in list order, deps ignored)
    as one CUDA graph on the current device: consecutive ops reading the same
    activations fuse into one grouped call, gated pairs run as one call."""
    if not ops:
        raise ValueError("empty sequence")
    arr, M = _chain_structs(ops)
    w0 = ops[0].weight
    h = ctypes.c_void_p()
    _check(load().mnb_graph_build(arr, len(ops), M, w0.block_size, _dtype_code(ops[0].A.dtype),
                                  _dtype_code(w0.scale_dtype), ctypes.byref(h)),
           "mnb_graph_build")
    return MnbGraph(ops, h.value)


def mnb_chain_run_noalloc(ops: list, *, stream=None) -> None:
    """Plan and run a chain with the plan in the library's fixed device
    array: no device memory is allocated (for callers that cannot allocate;
    at most one such call in flight at a time)."""
    if not ops:
        raise ValueError("empty chain")
    arr, M = _chain_structs(ops)
    w0 = ops[0].weight
    _check(load().mnb_chain_run_noalloc(arr, len(ops), M, w0.block_size,
                                        _dtype_code(ops[0].A.dtype), _dtype_code(w0.scale_dtype),
                                        _stream(stream)), "mnb_chain_run_noalloc")


def mnb_matmul_rmsnorm(A: torch.Tensor, w: PackedWeight, bias: torch.Tensor | None = None, *,
                       gamma: torch.Tensor | None = None, eps: float = 1e-6,
                       normalize: bool = True, logits: bool = True, argmax: bool = False,
                       out: torch.Tensor | None = None, stream=None):
    """Y = rmsnorm(A; gamma, eps) @ dequant(w)^T + bias (normalize=False: plain
    A), and optionally the greedy ArgMax of each row: one decode launch for
    M <= 16, the tensor-core kernel for bf16 prefill rows, 16-row decode
    slices otherwise. Returns (Y or None, argmax int64 [M] or None)."""
    if A.dim() != 2 or A.shape[1] != w.K or not A.is_cuda or not A.is_contiguous():
        raise ValueError(f"A must be a contiguous CUDA [M, {w.K}] tensor")
    for name, t in (("bias", bias), ("gamma", gamma)):
        if t is not None and (t.dtype != torch.float32 or not t.is_cuda):
            raise ValueError(f"{name} must be an fp32 CUDA tensor")
    if not logits and not argmax:
        raise ValueError("ask for the logits, the argmax or both")
    M = A.shape[0]
    Y = None
    if logits:
        Y = out if out is not None else torch.empty(M, w.N, dtype=A.dtype, device=A.device)
    idx = torch.empty(M, dtype=torch.int64, device=A.device) if argmax else None
    _check(load().mnb_matmul_rmsnorm(
        _ptr(A), 1 if normalize else 0, _ptr(gamma), float(eps), _ptr(w.packed_b),
        _ptr(w.packed_scales), _ptr(w.packed_zp), _ptr(bias), M, w.N, w.K, w.block_size,
        _ptr(Y), _ptr(idx), _dtype_code(A.dtype), _dtype_code(w.scale_dtype), _stream(stream)),
        "mnb_matmul_rmsnorm")
    return Y, idx


def mnb_prepack_bnb4(B: torch.Tensor, absmax: torch.Tensor, N: int, K: int, block_size: int,
                     *, stream=None) -> PackedWeight:
    """Re-lay out a bitsandbytes-style 4-bit matrix (flattened N x K codes,
    first of a pair in the high nibble; absmax per block_size flattened
    elements) into the packed plan; K must be a multiple of block_size."""
    if B.dtype != torch.uint8 or not B.is_cuda or not absmax.is_cuda:
        raise ValueError("B must be a CUDA uint8 tensor and absmax a CUDA tensor")
    b, s, _ = mnb_prepacked_sizes(N, K, block_size, absmax.dtype, False)
    pb = torch.empty(b, dtype=torch.uint8, device=B.device)
    ps = torch.empty(s // absmax.element_size(), dtype=absmax.dtype, device=B.device)
    _check(load().mnb_prepack_bnb4(_ptr(B), _ptr(absmax.contiguous()), N, K, block_size,
                                   _dtype_code(absmax.dtype), _ptr(pb), _ptr(ps),
                                   _stream(stream)), "mnb_prepack_bnb4")
    return PackedWeight(pb, ps, None, N, K, block_size, absmax.dtype)


def mnb_matmul_bnb4(A: torch.Tensor, w: PackedWeight, code: torch.Tensor,
                    bias: torch.Tensor | None = None, *, out: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Y = A @ (code[q] * absmax)^T + bias for a packed bitsandbytes-style
    weight; code: the 16 fp32 code-book values (CUDA)."""
    if A.dim() != 2 or A.shape[1] != w.K or not A.is_cuda or not A.is_contiguous():
        raise ValueError(f"A must be a contiguous CUDA [M, {w.K}] tensor")
    if code.dtype != torch.float32 or code.numel() != 16 or not code.is_cuda:
        raise ValueError("code must be 16 fp32 values on the GPU")
    M = A.shape[0]
    if out is None:
        out = torch.empty(M, w.N, dtype=A.dtype, device=A.device)
    _check(load().mnb_matmul_bnb4(_ptr(A), _ptr(w.packed_b), _ptr(w.packed_scales),
                                  _ptr(code.contiguous()), _ptr(bias), M, w.N, w.K,
                                  w.block_size, _ptr(out), _dtype_code(A.dtype),
                                  _dtype_code(w.scale_dtype), _stream(stream)),
           "mnb_matmul_bnb4")
    return out
