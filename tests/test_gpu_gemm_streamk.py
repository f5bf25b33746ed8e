"""GPU parity of the tensor-core kernel's stream-K schedule (mnb_matmul_ws,
path MNB_PATH_GEMM_STREAMK) against the oracle, through the C ABI.

The schedule splits the product's (256 x 128 output tile, 64-wide k stage)
units evenly over two CTAs per SM; a tile that several CTAs share is
completed by whichever of them finishes last, adding the fp32 partial tiles
in the order of their k stages. Each product is the one the whole-tile
kernel computes (each dequantised weight as an exact bf16 hi + lo pair,
fp32 accumulation), summed in a different but fixed order, so the same
stated bound applies (tests/tolerance.py), also on inputs built so that a
single rounding of every weight would err the same way
(tests/adversarial.py), and repeated runs are bitwise equal.

The shapes cover: one tile split over many CTAs (one output tile, 64 k
stages), CTAs whose ranges cross tiles (many tiles of few stages), ragged M,
N and K, a partial last block, zero points, fp32 scales and every block
size; a workspace too small for the full grid; replay in a CUDA graph with
new activations (the counters must be clear again after every run); and
the host's refusals.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300 import binding
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.adversarial import aligned_rounding_problem
from tests.tolerance import check

pytestmark = pytest.mark.gpu

COUNT_BYTES = 4096
CTA_BYTES = 2 * 256 * 128 * 4  # two parked partial tiles


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def prepack(prob, dev):
    f = lambda t: None if t is None else t.to(dev)
    return mnb.mnb_prepack(f(prob.B), f(prob.scales), f(prob.zero_points), prob.N, prob.K,
                           prob.block_size)


def ref(prob, rows=None, cols=None):
    return oracle.matmulnbits(prob.A, prob.B, prob.scales, prob.zero_points, prob.bias,
                              N=prob.N, K=prob.K, block_size=prob.block_size,
                              rows=rows, cols=cols)


def flags_clear(ws):
    return int(ws[:COUNT_BYTES].count_nonzero()) == 0


# (M, N, K): one tile over 16 CTAs; tiles of 9 stages crossed by CTA ranges,
# ragged M and N, partial last block; a mid-size ragged product.
SHAPES = [(200, 100, 4096), (777, 1000, 520), (300, 2000, 1000)]


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("scale_f32", [False, True])
def test_streamk_tiles_and_tails(dev, bs, with_zp, scale_f32):
    ws = mnb.mnb_matmul_workspace(dev)
    for j, (M, N, K) in enumerate(SHAPES):
        prob = make_problem(M, N, K, bs, dtype=torch.bfloat16, zero_points=with_zp,
                            bias=(j != 1), seed=40 * bs + 7 * j + with_zp + 2 * scale_f32)
        if scale_f32:
            prob.scales = prob.scales.float()
        w = prepack(prob, dev)
        Y = mnb.mnb_matmul(prob.A.to(dev), w, None if prob.bias is None else prob.bias.to(dev),
                           path="gemm_streamk", workspace=ws)
        torch.cuda.synchronize()
        R, mag = ref(prob)
        check(Y, R, mag, f"streamk M{M} N{N} K{K} bs{bs} zp{with_zp} sf32{scale_f32}")
        assert flags_clear(ws)
    assert mnb.mnb_fault_status() == 0


@pytest.mark.parametrize("scale_dtype", [torch.bfloat16, torch.float32], ids=["sbf16", "sf32"])
def test_streamk_adversarial_rounding_within_stated_bound(dev, scale_dtype):
    ws = mnb.mnb_matmul_workspace(dev)
    prob = aligned_rounding_problem(300, 700, 64, 8, scale_dtype=scale_dtype,
                                    zero_points=True, seed=3)
    w = prepack(prob, dev)
    Y = mnb.mnb_matmul(prob.A.to(dev), w, None, path="gemm_streamk", workspace=ws)
    torch.cuda.synchronize()
    R, mag = ref(prob)
    check(Y, R, mag, "streamk adversarial")
    assert flags_clear(ws)


def test_streamk_and_whole_tiles_agree_and_repeat_bitwise(dev):
    """Both schedules within the bound of the oracle on the same product; the
    stream-K result is bitwise the same on a second run."""
    prob = make_problem(1000, 2560, 4096, 128, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=11, scale_range=(0.002, 0.01))
    w = prepack(prob, dev)
    A, bias = prob.A.to(dev), prob.bias.to(dev)
    ws = mnb.mnb_matmul_workspace(dev)
    Y1 = mnb.mnb_matmul(A, w, bias, path="gemm_streamk", workspace=ws)
    Y2 = mnb.mnb_matmul(A, w, bias, path="gemm_streamk", workspace=ws)
    Yc = mnb.mnb_matmul(A, w, bias, path="gemm", workspace=None)
    torch.cuda.synchronize()
    assert torch.equal(Y1, Y2)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 255, 256, 999], rng.choice(1000, 12, replace=False)]))
    cols = np.unique(np.concatenate([[0, 127, 128, 2559], rng.choice(2560, 60, replace=False)]))
    R, mag = ref(prob, rows=rows, cols=cols)
    check(Y1[rows][:, cols], R, mag, "streamk")
    check(Yc[rows][:, cols], R, mag, "whole tiles")
    assert flags_clear(ws)


def test_streamk_with_a_small_workspace(dev):
    """Room for 20 CTAs caps the grid at 20."""
    prob = make_problem(600, 1500, 2048, 64, dtype=torch.bfloat16, zero_points=True,
                        bias=True, seed=13)
    w = prepack(prob, dev)
    ws = torch.zeros(COUNT_BYTES + 20 * CTA_BYTES, dtype=torch.uint8, device=dev)
    Y = mnb.mnb_matmul(prob.A.to(dev), w, prob.bias.to(dev), path="gemm_streamk",
                       workspace=ws)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    rows = np.sort(rng.choice(600, 24, replace=False))
    R, mag = ref(prob, rows=rows)
    check(Y[rows], R, mag, "streamk, 20 CTAs")
    assert flags_clear(ws)


def test_streamk_replays_in_a_cuda_graph(dev):
    """Captured once, replayed with new activations: every replay finds the
    flags clear and computes the new product."""
    M, N, K = 512, 2560, 9728
    prob = make_problem(M, N, K, 128, dtype=torch.bfloat16, zero_points=False, bias=True,
                        seed=17, scale_range=(0.002, 0.01))
    w = prepack(prob, dev)
    A = prob.A.to(dev)
    bias = prob.bias.to(dev)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = mnb.mnb_matmul_workspace(dev)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        mnb.mnb_matmul(A, w, bias, out=Y, path="gemm_streamk", workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        mnb.mnb_matmul(A, w, bias, out=Y, path="gemm_streamk", workspace=ws)
    gen = torch.Generator().manual_seed(18)
    rng = np.random.default_rng(7)
    for rep in range(3):
        prob.A = torch.randn(M, K, generator=gen).to(torch.bfloat16)
        A.copy_(prob.A.to(dev))
        g.replay()
        torch.cuda.synchronize()
        rows = np.sort(rng.choice(M, 6, replace=False))
        cols = np.sort(rng.choice(N, 96, replace=False))
        R, mag = ref(prob, rows=rows, cols=cols)
        check(Y[rows][:, cols], R, mag, f"graph replay {rep}")
        assert flags_clear(ws)
    assert mnb.mnb_fault_status() == 0


def test_streamk_refusals(dev):
    """Host-side checks only: nothing is launched."""
    prob = make_problem(64, 256, 512, 64, dtype=torch.bfloat16, seed=19)
    w = prepack(prob, dev)
    A = prob.A.to(dev)
    with pytest.raises(mnb.MnbError) as e:  # no workspace
        mnb.mnb_matmul(A, w, path="gemm_streamk", workspace=None)
    assert e.value.status == -8
    with pytest.raises(mnb.MnbError) as e:  # fp32 activations
        mnb.mnb_matmul(A.float(), w, path="gemm_streamk", workspace=mnb.mnb_matmul_workspace(dev))
    assert e.value.status == -8
    ws = mnb.mnb_matmul_workspace(dev)
    with pytest.raises(mnb.MnbError) as e:  # not 256-byte aligned
        mnb.mnb_matmul(A, w, path="gemm_streamk", workspace=ws[16:])
    assert e.value.status == -5
    buf = torch.zeros(ws.numel() + 64 * 256 * 2, dtype=torch.uint8, device=dev)
    Y = buf[-64 * 256 * 2:].view(torch.bfloat16).view(64, 256)
    with pytest.raises(mnb.MnbError) as e:  # workspace overlaps Y
        mnb.mnb_matmul(A, w, out=Y, path="gemm_streamk", workspace=buf)
    assert e.value.status == -6


def test_auto_workspace_is_kept_per_stream(dev):
    """The binding's default workspace: one per (device, stream), zero-filled."""
    prob = make_problem(300, 2560, 1024, 128, dtype=torch.bfloat16, seed=23)
    w = prepack(prob, dev)
    A = prob.A.to(dev)
    Y = mnb.mnb_matmul(A, w)
    torch.cuda.synchronize()  # one product at a time
    s2 = torch.cuda.Stream(dev)
    with torch.cuda.stream(s2):
        Y2 = mnb.mnb_matmul(A, w)
    torch.cuda.synchronize()
    keys = [k for k in binding._workspaces if k[0] == dev.index]
    assert len(keys) >= 2
    assert all(flags_clear(binding._workspaces[k]) for k in keys)
    assert torch.equal(Y, Y2)
