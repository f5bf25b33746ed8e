"""GPU checks of the packed-weight header (page "Qwen3 CPU Inference Critical
Path", section "Prepared weight-only plan": the plan captures N, K, the
nibble order and the block size).

Every prepack call writes the header into the last 256 bytes of packed_b and
records it in the library. A weight saved and restored into new device
buffers is unknown to the library until its stored header is read back and
registered; after that it computes exactly what the original computes. A call
whose N, K, block size, scale dtype, zero-point presence or code form differs
from the header is refused with MNB_ERR_LAYOUT, and nothing runs: the output
buffer keeps its contents.
"""
import dataclasses

import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.packing import pack_bnb4_flat, pack_flat

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def fields(h):
    return {f: getattr(h, f) for f, _ in h._fields_}


def test_every_prepack_writes_its_header(dev):
    p = make_problem(1, 300, 520, 64, dtype=torch.bfloat16, zero_points=True, seed=1)
    w = mnb.mnb_prepack(p.B.to(dev), p.scales.to(dev), p.zero_points.to(dev), 300, 520, 64)
    assert fields(mnb.mnb_packed_read_header(w)) == fields(
        mnb.mnb_packed_header_make(300, 520, 64, torch.bfloat16, True))
    q = mnb.mnb_prepack_qdq(torch.tensor(pack_flat(np.zeros((520, 300), np.uint8))).to(dev),
                            p.scales.float().t().contiguous().to(dev), None, 300, 520, 64)
    assert fields(mnb.mnb_packed_read_header(q)) == fields(
        mnb.mnb_packed_header_make(300, 520, 64, torch.float32, True))
    b = mnb.mnb_prepack_bnb4(torch.tensor(pack_bnb4_flat(np.ones((30, 128), np.uint8))).to(dev),
                             torch.ones(30 * 128 // 64, device=dev), 30, 128, 64)
    assert fields(mnb.mnb_packed_read_header(b)) == fields(
        mnb.mnb_packed_header_make(30, 128, 64, torch.float32, False, mnb.MNB_CODES_CODEBOOK))


def test_restored_weight_runs_once_its_header_is_registered(dev):
    p = make_problem(3, 1000, 777, 32, dtype=torch.float32, zero_points=True, bias=True,
                     seed=2)
    w = mnb.mnb_prepack(p.B.to(dev), p.scales.to(dev), p.zero_points.to(dev), 1000, 777, 32)
    A, bias = p.A.to(dev), p.bias.to(dev)
    Y0 = mnb.mnb_matmul(A, w, bias)
    saved = [t.cpu() for t in (w.packed_b, w.packed_scales, w.packed_zp)]
    r = dataclasses.replace(w, packed_b=saved[0].to(dev), packed_scales=saved[1].to(dev),
                            packed_zp=saved[2].to(dev))
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul(A, r, bias)
    assert e.value.status == -10
    mnb.mnb_packed_register(r.packed_b, mnb.mnb_packed_read_header(r))
    assert torch.equal(mnb.mnb_matmul(A, r, bias), Y0)
    mnb.mnb_packed_forget(r.packed_b)
    with pytest.raises(mnb.MnbError):
        mnb.mnb_matmul(A, r, bias)


@pytest.mark.parametrize("change", [dict(block_size=64), dict(N=999), dict(K=700),
                                    dict(packed_zp=None), dict(scale_dtype=torch.float32)])
def test_a_call_that_disagrees_with_the_header_runs_nothing(dev, change):
    p = make_problem(2, 1000, 768, 32, dtype=torch.bfloat16, zero_points=True, seed=3)
    w = mnb.mnb_prepack(p.B.to(dev), p.scales.to(dev), p.zero_points.to(dev), 1000, 768, 32)
    bad = dataclasses.replace(w, **change)
    A = p.A.to(dev)[:, :bad.K].contiguous()
    Y = torch.full((2, bad.N), 7.0, dtype=torch.bfloat16, device=dev)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_matmul(A, bad, None, out=Y)
    assert e.value.status == -10
    torch.cuda.synchronize()
    assert bool((Y == 7.0).all())
