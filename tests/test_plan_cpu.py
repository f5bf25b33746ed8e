"""Host logic of the kernel choice (mnb_matmul_plan): the dispatch of a6
and the tensor-core kernel's tile height, K split, stream-K schedule and
TMA-store epilogue, for a GB300 (152 SMs), without a GPU.

The expected decisions are the measured ones (timing of the Qwen3-4B
prefill shapes, bs 128, zero points, on GB300, each weight as an exact hi +
lo bf16 pair): the stream-K schedule beat whole tiles on down at every M
(79.1 / 162.1 / 288.1 us against 81.7 / 228.3 / 433.5 at M = 512 / 2048 /
4096) and on o at M = 2048 and 4096 (90.7 / 138.1 against 100.9 / 190.6),
and lost on q, k, v, gate and up at every M and on o at M = 512.
"""
import ctypes

import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
from int4_weight_only_matmulnbits_gb300 import binding
from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B

SMS = 152
WS = 4096 + 2 * SMS * 2 * 256 * 128 * 4  # what mnb_matmul_workspace_size() gives on GB300


@pytest.fixture(scope="module")
def lib():
    mnb.build_library()
    return mnb.load()


def plan(M, N, K, bs=128, **kw):
    kw.setdefault("sm_count", SMS)
    return mnb.mnb_matmul_plan(M, N, K, bs, **kw)


def test_struct_layout_matches_the_header(lib):
    assert ctypes.sizeof(binding.PlanInfoC) == 40


@pytest.mark.parametrize("M", [512, 2048, 4096])
def test_stream_k_only_where_it_was_measured_to_win(lib, M):
    wins = {512: {"down"}, 2048: {"o", "down"}, 4096: {"o", "down"}}[M]
    for p in QWEN3_4B["projections"]:
        r = plan(M, p.N, p.K, zero_points=True, workspace_bytes=WS)
        assert r["path"] == "gemm" and not r["tf32"]
        assert r["stream_k"] == (p.name in wins), (M, p.name, r)
        if r["stream_k"]:
            assert r["tile_rows"] == 256 and r["k_split"] == 1 and r["ctas"] == 2 * SMS
            assert not r["tma_store"]
        # Without a workspace the whole-tile schedule, always.
        assert not plan(M, p.N, p.K, zero_points=True)["stream_k"]


def test_whole_tile_shapes_and_grids(lib):
    # gate 2560 -> 9728 at M = 2048: 8 x 76 tiles of 256 x 128, two waves.
    g = plan(2048, 9728, 2560, zero_points=True, workspace_bytes=WS)
    assert (g["tile_rows"], g["k_split"], g["ctas"], g["tma_store"]) == (256, 1, 608, True)
    # down without a workspace: 160 tiles of 256 rows.
    d = plan(2048, 2560, 9728, zero_points=True)
    assert (d["tile_rows"], d["k_split"], d["ctas"]) == (256, 1, 160)
    # k 2560 -> 1024 at M = 2048: too few 256-row tiles; 128-row tiles split over K.
    k = plan(2048, 1024, 2560, zero_points=True)
    assert k["tile_rows"] == 128 and k["k_split"] > 1 and not k["tma_store"]


def test_dispatch_by_rows_and_activation_dtype(lib):
    assert plan(16, 9728, 2560)["path"] == "gemv"
    r = plan(17, 9728, 2560)
    assert r["path"] == "gemm" and r["tile_rows"] in (128, 256)
    f = plan(64, 9728, 2560, a_dtype=torch.float32)
    assert f["path"] == "gemm" and f["tf32"] and f["tile_rows"] == 128
    # Rows the TMA cannot address (K not a multiple of 4 fp32 / 8 bf16
    # elements): the decode kernel over 16-row slices.
    s = plan(64, 9728, 2562, a_dtype=torch.float32)
    assert s["path"] == "gemv" and s["m_slices"] == 4
    s = plan(100, 1000, 2564)
    assert s["path"] == "gemv" and s["m_slices"] == 7


def test_forced_paths(lib):
    with pytest.raises(mnb.MnbError) as e:  # stream-K needs a workspace
        plan(2048, 2560, 9728, path="gemm_streamk")
    assert e.value.status == -8
    with pytest.raises(mnb.MnbError) as e:  # and bf16 activations
        plan(2048, 2560, 9728, path="gemm_streamk", a_dtype=torch.float32, workspace_bytes=WS)
    assert e.value.status == -8
    # Room for 20 CTAs caps the grid; forced even where it would not pay.
    r = plan(2048, 2560, 9728, path="gemm_streamk", workspace_bytes=4096 + 20 * 262144)
    assert r["stream_k"] and r["ctas"] == 20
    assert plan(512, 4096, 2560, path="gemm_streamk", workspace_bytes=WS)["stream_k"]
    # The decode kernel up to 16 rows only; the tensor-core kernel at any M.
    with pytest.raises(mnb.MnbError) as e:
        plan(17, 256, 256, path="gemv")
    assert e.value.status == -8
    assert plan(1, 256, 256, path="gemm")["path"] == "gemm"


def test_tma_store_needs_16_byte_rows_of_y(lib):
    assert plan(2048, 2560, 9728)["tma_store"]
    assert not plan(2048, 2561, 9728)["tma_store"]


def test_argument_errors(lib):
    info = binding.PlanInfoC()
    assert lib.mnb_matmul_plan(64, 256, 256, 128, 1, 1, 0, 0, 0, SMS, None) == -1
    assert lib.mnb_matmul_plan(0, 256, 256, 128, 1, 1, 0, 0, 0, SMS, ctypes.byref(info)) == -2
    assert lib.mnb_matmul_plan(64, 256, 256, 48, 1, 1, 0, 0, 0, SMS, ctypes.byref(info)) == -3
    assert lib.mnb_matmul_plan(64, 256, 256, 128, 5, 1, 0, 0, 0, SMS, ctypes.byref(info)) == -4
    assert lib.mnb_matmul_plan(64, 256, 256, 128, 1, 1, 0, 9, 0, SMS, ctypes.byref(info)) == -8
    if not torch.cuda.is_available():  # sm_count 0 asks the device
        assert lib.mnb_matmul_plan(64, 256, 256, 128, 1, 1, 0, 0, 0, 0,
                                   ctypes.byref(info)) in (-7, -9)


def test_pair_kernel_tile_widths_fill_the_pairs(lib):
    """The CTA-pair kernel's tile width (32 nt columns, nt = 4..8 weight
    tiles per CTA) for the Qwen3-4B shapes at M = 2048 on 76 pairs: the
    fewest rounds of tiles times the work per tile."""
    want = {1024: (128, 128), 2560: (160, 152), 4096: (224, 152), 9728: (256, 152)}
    for N, (cols, ctas) in want.items():
        r = plan(2048, N, 2560, path="gemm_pair", zero_points=True)
        assert (r["path"], r["tile_rows"], r["k_split"]) == ("gemm", 256, 1)
        assert (r["pair_cols"], r["ctas"]) == (cols, ctas), N
    # A single tile: one pair; past the pairs, every pair is launched.
    assert plan(17, 16, 264, path="gemm_pair")["ctas"] == 2
    assert plan(8192, 151936, 2560, path="gemm_pair")["ctas"] == SMS


def test_pair_kernel_refusals(lib):
    with pytest.raises(mnb.MnbError) as e:
        plan(2048, 2560, 2560, path="gemm_pair", a_dtype=torch.float32)
    assert e.value.status == -8
    assert plan(2048, 2560, 2560, path="gemm")["pair_cols"] == 0
