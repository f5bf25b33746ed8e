"""C-ABI checks that need no GPU: the library loads, exports every entry
point include/mnb.h declares, and rejects invalid arguments on the host
before touching a device, including a packed weight whose recorded header
does not match the call (fake device addresses: the header records are
host-side, so registering one needs no device)."""
import ctypes
import os
import re

import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
from int4_weight_only_matmulnbits_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mnb.build_library()
    return mnb.load()


def declared_entry_points():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"MNB_API\s+[\w\s\*]*?\b(mnb_\w+)\s*\(", text))
    return names


def test_header_declares_the_binding_names():
    assert declared_entry_points() == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert mnb.mnb_version() >> 16 == 1
    for code in range(-10, 1):
        assert mnb.status_string(code).startswith("MNB_")
    assert "unknown" in mnb.status_string(42)


@pytest.mark.parametrize("N,K,bs,zp", [(3072, 1024, 32, False), (7, 33, 16, True),
                                       (151936, 2560, 128, False), (1, 1, 256, True)])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_prepacked_sizes(lib, N, K, bs, zp, dt):
    b, s, z = mnb.mnb_prepacked_sizes(N, K, bs, dt, zp)
    n16, k64, nb = -(-N // 16), -(-K // 64), -(-K // bs)
    assert b == n16 * k64 * 512 + 256  # the codes, then the packed-weight header
    assert s == n16 * nb * 16 * (4 if dt == torch.float32 else 2)
    assert z == (n16 * (-(-nb // 2) * 2) * 8 if zp else 0)


def test_packed_storage_within_bound_for_qwen_shapes(lib):
    """Packed weights + scales + zero points stay within 1.25x the serialized
    UINT4 codes + scales + zero points (page "Qwen3 CPU Inference Critical
    Path", section "Benchmark gates", INT4 memory row)."""
    from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_0P6B, QWEN3_4B
    for model, bs, dt, zp in ((QWEN3_0P6B, 32, torch.float32, True),
                              (QWEN3_4B, 128, torch.bfloat16, False)):
        for p in model["projections"] + [model["lm_head"]]:
            nb = -(-p.K // bs)
            serial = p.N * nb * bs // 2 + p.N * nb * (4 if dt == torch.float32 else 2)
            serial += p.N * ((nb + 1) // 2) if zp else 0
            packed = sum(mnb.mnb_prepacked_sizes(p.N, p.K, bs, dt, zp))
            assert packed <= 1.25 * serial, (p, packed / serial)


def _call_matmul(lib, **kw):
    args = dict(A=16, packed_b=256, scales=256, zp=None, bias=None, M=1, N=16, K=64,
                bs=32, Y=1 << 20, a_t=0, s_t=0, path=0)
    args.update(kw)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.mnb_matmul_path(v(args["A"]), v(args["packed_b"]), v(args["scales"]),
                               v(args["zp"]), v(args["bias"]), args["M"], args["N"],
                               args["K"], args["bs"], v(args["Y"]), args["a_t"],
                               args["s_t"], args["path"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(A=None), -1), (dict(packed_b=None), -1), (dict(scales=None), -1),
    (dict(Y=None), -1), (dict(M=0), -2), (dict(N=0), -2), (dict(K=-1), -2),
    (dict(M=1 << 31), -2), (dict(bs=0), -3), (dict(bs=48), -3), (dict(bs=512), -3),
    (dict(bs=8), -3), (dict(a_t=7), -4), (dict(s_t=2), -4), (dict(packed_b=264), -5),
    (dict(scales=260), -5), (dict(zp=1000), -5), (dict(A=17), -5), (dict(bias=2), -5),
    (dict(path=9), -8), (dict(path=1, M=17), -8),
    (dict(Y=16), -6), (dict(Y=300), -6),
])
def test_matmul_rejects_invalid_arguments_on_host(lib, kw, status):
    assert _call_matmul(lib, **kw) == status


def test_prepack_rejects_invalid_arguments_on_host(lib):
    v = ctypes.c_void_p
    ok = dict(B=v(4096), S=v(1 << 16), Z=None, N=16, K=64, bs=32, st=0,
              pb=v(1 << 20), ps=v(1 << 21), pz=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.mnb_prepack(a["B"], a["S"], a["Z"], a["N"], a["K"], a["bs"], a["st"],
                               a["pb"], a["ps"], a["pz"], None)
    assert call(B=None) == -1
    assert call(Z=v(8192), pz=None) == -1
    assert call(N=0) == -2
    assert call(bs=24) == -3
    assert call(st=5) == -4
    assert call(pb=v((1 << 20) + 8)) == -5
    assert call(pb=v(4096 + 16)) == -6  # packed output overlaps B
    assert call(ps=v((1 << 20) + 256)) == -6  # the two outputs overlap
    assert lib.mnb_prepacked_sizes(16, 64, 32, 0, 0, None, None, None) == -1


def test_prepack_qdq_rejects_invalid_arguments_on_host(lib):
    """QDQ re-layout: the same argument checks, plus the axis (0 or 1) and a
    packed zero-point output that is always required."""
    v = ctypes.c_void_p
    ok = dict(B=v(4096), S=v(1 << 16), Z=None, axis=0, N=16, K=64, bs=32, st=1,
              pb=v(1 << 20), ps=v(1 << 21), pz=v(1 << 22))

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.mnb_prepack_qdq(a["B"], a["S"], a["Z"], a["axis"], a["N"], a["K"], a["bs"],
                                   a["st"], a["pb"], a["ps"], a["pz"], None)
    assert call(B=None) == -1
    assert call(pz=None) == -1
    assert call(axis=2) == -2
    assert call(axis=-1) == -2
    assert call(K=0) == -2
    assert call(bs=48) == -3
    assert call(st=7) == -4
    assert call(pz=v((1 << 22) + 4)) == -5
    assert call(pb=v(4096)) == -6  # packed output overlaps B


# --- decode chain: host-side validation -------------------------------------------

def _chain_ops(n, deps=None, over=None):
    """n independent ops of N=16, K=64 (bf16, bs 32) on disjoint fake device
    addresses; `over` maps op index -> dict of field overrides."""
    from int4_weight_only_matmulnbits_gb300.binding import ChainOpC
    arr = (ChainOpC * n)()
    for j in range(n):
        base = (j + 1) << 24
        c = arr[j]
        c.A, c.Y = base, base + (1 << 20)
        c.packed_b, c.packed_scales = base + (2 << 20), base + (3 << 20)
        c.N, c.K = 16, 64
        for k in range(4):
            c.deps[k] = -1
        for k, d in enumerate((deps or {}).get(j, ())):
            c.deps[k] = d
        for name, val in (over or {}).get(j, {}).items():
            setattr(c, name, val)
    return arr


def _build(lib, arr, n=None, M=1, bs=32, a_t=1, s_t=1, plan=None, plan_bytes=0):
    from int4_weight_only_matmulnbits_gb300.binding import ChainInfoC
    info = ChainInfoC()
    n = len(arr) if n is None else n
    return lib.mnb_chain_build(arr, n, M, bs, a_t, s_t,
                               None if plan is None else ctypes.c_void_p(plan), plan_bytes,
                               ctypes.byref(info), None)


NO_DEVICE = (-7, -9)  # validation passed; the call then needs a device


def _register(lib, ptr, N, K, bs, s_t, zp, codes=0):
    """Records, for a fake device address, the header a prepack call would write."""
    h = binding.PackedHeaderC()
    assert lib.mnb_packed_header_make(N, K, bs, s_t, int(zp), codes, ctypes.byref(h)) == 0
    assert lib.mnb_packed_register(ctypes.c_void_p(ptr), ctypes.byref(h)) == 0
    return h


def test_chain_build_rejects_invalid_arguments_on_host(lib):
    assert lib.mnb_chain_build(None, 1, 1, 32, 1, 1, None, 0, None, None) == -1
    assert _build(lib, _chain_ops(2), n=0) == -2
    assert _build(lib, _chain_ops(2), M=9) == -2
    assert _build(lib, _chain_ops(2), M=0) == -2
    assert _build(lib, _chain_ops(2), bs=48) == -3
    assert _build(lib, _chain_ops(2), a_t=3) == -4
    assert _build(lib, _chain_ops(2, over={1: {"A": None}})) == -1
    assert _build(lib, _chain_ops(2, over={1: {"packed_zp": 1 << 30}})) == -1  # mixed zp
    assert _build(lib, _chain_ops(2, over={0: {"packed_scales_up": 1 << 30}})) == -1
    assert _build(lib, _chain_ops(2, over={1: {"K": 0}})) == -2
    assert _build(lib, _chain_ops(2, over={1: {"packed_b": (2 << 24) + (2 << 20) + 8}})) == -5
    assert _build(lib, _chain_ops(2, over={0: {"A": (1 << 24) + 1}})) == -5
    assert _build(lib, _chain_ops(2, deps={0: (0,)})) == -2   # not an earlier op
    assert _build(lib, _chain_ops(2, deps={1: (2,)})) == -2
    assert _build(lib, _chain_ops(2, deps={1: (-2,)})) == -2


def test_chain_build_checks_hazards_on_host(lib):
    for j in range(3):
        _register(lib, ((j + 1) << 24) + (2 << 20), 16, 64, 32, 1, False)
    y0 = (1 << 24) + (1 << 20)
    a0 = 1 << 24
    # op 1 reads op 0's output: needs the dependency
    assert _build(lib, _chain_ops(2, over={1: {"A": y0}})) == -6
    assert _build(lib, _chain_ops(2, deps={1: (0,)}, over={1: {"A": y0}})) in NO_DEVICE
    # op 1 overwrites op 0's activations, or its output: needs the dependency
    assert _build(lib, _chain_ops(2, over={1: {"Y": a0}})) == -6
    assert _build(lib, _chain_ops(2, over={1: {"Y": y0}})) == -6
    assert _build(lib, _chain_ops(2, deps={1: (0,)}, over={1: {"Y": a0}})) in NO_DEVICE
    # a transitive dependency is enough
    y1 = (2 << 24) + (1 << 20)
    assert _build(lib, _chain_ops(3, deps={1: (0,), 2: (1,)},
                                  over={2: {"A": y0}})) in NO_DEVICE
    assert _build(lib, _chain_ops(3, deps={2: (1,)}, over={2: {"A": y0}})) == -6
    assert _build(lib, _chain_ops(3, deps={2: (1,)}, over={2: {"A": y1}})) in NO_DEVICE
    # an output over any weight of the chain, or over its own activations
    assert _build(lib, _chain_ops(2, over={1: {"Y": (1 << 24) + (2 << 20)}})) == -6
    assert _build(lib, _chain_ops(2, over={0: {"Y": a0 + 32}})) == -6


def test_chain_run_rejects_an_altered_description(lib):
    from int4_weight_only_matmulnbits_gb300.binding import ChainInfoC
    info = ChainInfoC()
    assert lib.mnb_chain_run(None, ctypes.byref(info), None) == -1
    assert lib.mnb_chain_run(ctypes.c_void_p(1 << 20), None, None) == -1
    info.n_ops, info.grid, info.check = 3, 304, 12345
    assert lib.mnb_chain_run(ctypes.c_void_p(1 << 20), ctypes.byref(info), None) == -2


def test_matmul_rmsnorm_rejects_invalid_arguments_on_host(lib):
    v = ctypes.c_void_p
    ok = dict(A=v(1 << 16), nrm=1, gamma=v(1 << 17), eps=1e-6, pb=v(1 << 20), ps=v(1 << 21),
              pz=None, bias=None, M=1, N=16, K=64, bs=32, Y=v(1 << 22), am=v(1 << 23),
              a_t=1, s_t=1)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.mnb_matmul_rmsnorm(a["A"], a["nrm"], a["gamma"], a["eps"], a["pb"], a["ps"],
                                      a["pz"], a["bias"], a["M"], a["N"], a["K"], a["bs"],
                                      a["Y"], a["am"], a["a_t"], a["s_t"], None)
    assert call(A=None) == -1
    assert call(Y=None, am=None) == -1
    assert call(nrm=2) == -2
    assert call(eps=-1.0) == -2
    assert call(eps=float("inf")) == -2
    assert call(M=0) == -2
    assert call(bs=40) == -3
    assert call(a_t=5) == -4
    assert call(gamma=v((1 << 17) + 2)) == -5
    assert call(am=v((1 << 23) + 4)) == -5
    assert call(Y=v(1 << 16)) == -6            # Y over A
    assert call(am=v((1 << 22) + 8)) == -6     # argmax over Y
    assert call(gamma=v(1 << 22)) == -6        # Y over gamma
    _register(lib, 1 << 20, 16, 64, 32, 1, False)
    assert call(nrm=0, gamma=v(1 << 22)) in (-7, -9)  # gamma unused without normalize
    assert call(bs=64) == -10                  # packed with block_size 32


def test_bnb4_rejects_invalid_arguments_on_host(lib):
    v = ctypes.c_void_p
    assert lib.mnb_prepack_bnb4(None, v(1 << 16), 16, 64, 32, 0, v(1 << 20), v(1 << 21),
                                None) == -1
    assert lib.mnb_prepack_bnb4(v(4096), v(1 << 16), 16, 40, 16, 0, v(1 << 20), v(1 << 21),
                                None) == -8  # K not a multiple of the block size
    assert lib.mnb_prepack_bnb4(v(4096), v(1 << 16), 16, 64, 48, 0, v(1 << 20), v(1 << 21),
                                None) == -3
    assert lib.mnb_prepack_bnb4(v(4096), v(1 << 16), 16, 64, 32, 0, v((1 << 20) + 8),
                                v(1 << 21), None) == -5
    assert lib.mnb_matmul_bnb4(v(16), v(256), v(256), None, None, 1, 16, 64, 32, v(1 << 20),
                               0, 0, None) == -1
    assert lib.mnb_matmul_bnb4(v(16), v(256), v(256), v(2), None, 1, 16, 64, 32, v(1 << 20),
                               0, 0, None) == -5


def _call_matmul_ws(lib, ws, ws_bytes, **kw):
    args = dict(A=16, packed_b=256, scales=256, zp=None, bias=None, M=64, N=16, K=64,
                bs=32, Y=1 << 20, a_t=1, s_t=1, path=3)
    args.update(kw)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.mnb_matmul_ws(v(args["A"]), v(args["packed_b"]), v(args["scales"]),
                             v(args["zp"]), v(args["bias"]), args["M"], args["N"], args["K"],
                             args["bs"], v(args["Y"]), args["a_t"], args["s_t"], args["path"],
                             v(ws), ws_bytes, None)


def test_matmul_ws_checks_its_workspace_on_host(lib):
    """Workspace alignment (256 bytes) and overlap with every input and the
    output are refused before any device work; argument errors come first."""
    far = 1 << 30
    assert _call_matmul_ws(lib, far + 128, 1 << 20) == -5
    assert _call_matmul_ws(lib, 256, 1 << 16) == -6          # covers B and the scales
    assert _call_matmul_ws(lib, (1 << 20) - 256, 512) == -6  # covers the start of Y
    assert _call_matmul_ws(lib, far, 1 << 20, A=None) == -1
    assert _call_matmul_ws(lib, far, 1 << 20, path=5) == -8
    # A valid request reaches the device query, which fails without a GPU
    # (MNB_ERR_CUDA, or MNB_ERR_DEVICE for another architecture).
    assert _call_matmul_ws(lib, far, 1 << 20, packed_b=1 << 12) == -10  # no header recorded
    import torch
    _register(lib, 256, 16, 64, 32, 1, False)
    if not torch.cuda.is_available():
        assert _call_matmul_ws(lib, far, 1 << 20) in (-7, -9)
        assert lib.mnb_matmul_workspace_size() == 0


# --- packed-weight headers -------------------------------------------------------

def test_packed_header_fields(lib):
    h = _register(lib, 1 << 32, 3072, 1024, 32, 0, True)
    assert h.magic == binding.MNB_PACKED_MAGIC and h.version == 1 and h.codes == 0
    assert (h.N, h.K, h.block_size, h.scale_dtype, h.has_zero_points) == (3072, 1024, 32, 0, 1)
    sizes = mnb.mnb_prepacked_sizes(3072, 1024, 32, torch.float32, True)
    assert (h.packed_b_bytes, h.packed_scales_bytes, h.packed_zp_bytes) == sizes
    assert bytes(h)[:8] == b"MNB4PACK"
    h2 = binding.PackedHeaderC()
    # a code-book weight carries no zero points; unknown code forms are refused
    assert lib.mnb_packed_header_make(16, 64, 32, 0, 1, 1, ctypes.byref(h2)) == -8
    assert lib.mnb_packed_header_make(16, 64, 32, 0, 0, 2, ctypes.byref(h2)) == -8
    assert lib.mnb_packed_header_make(16, 64, 24, 0, 0, 0, ctypes.byref(h2)) == -3
    assert lib.mnb_packed_header_make(16, 64, 32, 0, 0, 0, None) == -1


def test_register_refuses_a_damaged_header(lib):
    h = binding.PackedHeaderC()
    assert lib.mnb_packed_header_make(160, 640, 64, 1, 0, 0, ctypes.byref(h)) == 0
    ptr = ctypes.c_void_p(3 << 32)
    for field, value in (("magic", 1), ("version", 2), ("N", 161), ("check", h.check ^ 1),
                         ("packed_b_bytes", h.packed_b_bytes + 16)):
        bad = binding.PackedHeaderC.from_buffer_copy(h)
        setattr(bad, field, value)
        assert lib.mnb_packed_register(ptr, ctypes.byref(bad)) == -10, field
    assert lib.mnb_packed_register(None, ctypes.byref(h)) == -1
    assert lib.mnb_packed_register(ptr, None) == -1


@pytest.mark.parametrize("kw", [dict(N=32), dict(K=128), dict(bs=64), dict(s_t=0),
                                dict(zp=1 << 23)])
def test_matmul_refuses_a_layout_mismatch_before_any_launch(lib, kw):
    """A weight packed with N=16, K=64, bs=32, bf16 scales and no zero points,
    called with one of those changed: MNB_ERR_LAYOUT, nothing enqueued (the
    same call with the recorded layout goes on to the device query)."""
    pb = 5 << 32
    _register(lib, pb, 16, 64, 32, 1, False)
    base = dict(packed_b=pb, scales=(5 << 32) + (1 << 20), A=6 << 32, Y=7 << 32, a_t=1, s_t=1)
    assert _call_matmul(lib, **base) in NO_DEVICE
    base.update(kw)
    assert _call_matmul(lib, **base) == -10
    assert "differs in" in lib.mnb_last_error_string().decode()


def test_layout_checks_cover_every_reader_of_a_packed_weight(lib):
    v = ctypes.c_void_p
    pb, ps = 9 << 32, (9 << 32) + (1 << 20)
    A, Y = v(10 << 32), v(11 << 32)
    _register(lib, pb, 16, 64, 32, 1, False)
    # unknown packed_b, and a forgotten one
    assert _call_matmul(lib, packed_b=12 << 32, scales=ps, A=10 << 32, Y=11 << 32, a_t=1,
                        s_t=1) == -10
    assert lib.mnb_packed_forget(v(pb)) == 0
    assert _call_matmul(lib, packed_b=pb, scales=ps, A=10 << 32, Y=11 << 32, a_t=1,
                        s_t=1) == -10
    _register(lib, pb, 16, 64, 32, 1, False)
    # grouped (second weight's K differs), gated pair (up unknown)
    arr = (ctypes.c_void_p * 2)(pb, pb)
    sc = (ctypes.c_void_p * 2)(ps, ps)
    ns = (ctypes.c_int64 * 2)(16, 16)
    ys = (ctypes.c_void_p * 2)(11 << 32, (11 << 32) + (1 << 20))
    assert lib.mnb_matmul_grouped(A, 2, arr, sc, None, None, ns, ys, 1, 64, 32, 1, 1,
                                  None) in NO_DEVICE
    assert lib.mnb_matmul_grouped(A, 2, arr, sc, None, None, ns, ys, 1, 128, 32, 1, 1,
                                  None) == -10
    assert lib.mnb_matmul_gate_up(A, v(pb), v(ps), None, None, v(13 << 32), v(ps), None,
                                  None, 1, 16, 64, 32, Y, 1, 1, None) == -10
    # the code-book form is not the affine one, either way round
    assert lib.mnb_matmul_bnb4(A, v(pb), v(ps), v(14 << 32), None, 1, 16, 64, 32, Y, 1, 1,
                               None) == -10
    _register(lib, 15 << 32, 16, 64, 32, 1, False, codes=1)
    assert lib.mnb_matmul_bnb4(A, v(15 << 32), v(ps), v(14 << 32), None, 1, 16, 64, 32, Y,
                               1, 1, None) in NO_DEVICE
    assert _call_matmul(lib, packed_b=15 << 32, scales=ps, A=10 << 32, Y=11 << 32, a_t=1,
                        s_t=1) == -10
    # unprepack, and a chain op whose weight has zero points it was not packed with
    assert lib.mnb_unprepack(v(pb), v(ps), None, 16, 64, 64, 1, v(16 << 32), v(17 << 32),
                             None, None) == -10
    ops = _chain_ops(1, over={0: {"packed_b": pb, "packed_scales": ps}})
    assert _build(lib, ops) in NO_DEVICE
    assert _build(lib, ops, bs=64) == -10


def test_graph_calls_reject_invalid_arguments_on_host(lib):
    v = ctypes.c_void_p
    h = v()
    assert lib.mnb_graph_build(None, 1, 1, 32, 1, 1, ctypes.byref(h)) == -1
    assert lib.mnb_graph_build(_chain_ops(1), 1, 1, 32, 1, 1, None) == -1
    assert lib.mnb_graph_build(_chain_ops(1), 0, 1, 32, 1, 1, ctypes.byref(h)) == -2
    assert lib.mnb_graph_build(_chain_ops(1), 1, 0, 32, 1, 1, ctypes.byref(h)) == -2
    assert lib.mnb_graph_build(_chain_ops(2, over={1: {"Y": None}}), 2, 1, 32, 1, 1,
                               ctypes.byref(h)) == -1
    assert not h.value  # nothing built
    for fn in (lib.mnb_graph_run, lib.mnb_graph_destroy):
        assert (fn(None, None) if fn is lib.mnb_graph_run else fn(None)) == -1
    assert lib.mnb_graph_info(None, None, None) == -1
    assert lib.mnb_graph_run_from_host(None, None, None, 0, None, None, 0, None) == -1
