"""GPU checks of the CUDA-graph executor (mnb_graph_*): a sequence of
projections recorded once and run as one graph launch per step.

The graph records the launches the single-call entry points make, so its
outputs are bitwise those of the same calls made one by one, and within the
stated bound of the oracle. Consecutive ops reading the same activations fuse
into one grouped call and a gated pair is one call (checked by the recorded
call count); the run framed by host copies returns the same outputs in host
memory; a sequence with an invalid op builds nothing and reports that op's
error.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.tolerance import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def sequence(dev, M, dtype, bs, zp, seed):
    """q/k/v-like ops on one activation row set, a gated pair, then a single
    op reading its own rows: (ops, problems per op, the A tensors)."""
    probs, ops = [], []
    K = 512
    A0 = make_problem(M, 1, K, bs, dtype=dtype, seed=seed).A.to(dev)
    for i, N in enumerate((384, 128, 128)):
        p = make_problem(M, N, K, bs, dtype=dtype, zero_points=zp, bias=(i == 1),
                         seed=seed + 1 + i)
        p.A = A0.cpu()
        w = mnb.mnb_prepack(p.B.to(dev), p.scales.to(dev),
                            None if p.zero_points is None else p.zero_points.to(dev), N, K, bs)
        ops.append(mnb.ChainOp(A0, w, torch.empty(M, N, dtype=dtype, device=dev),
                               None if p.bias is None else p.bias.to(dev)))
        probs.append(p)
    A1 = make_problem(M, 1, K, bs, dtype=dtype, seed=seed + 9).A.to(dev)
    g = make_problem(M, 256, K, bs, dtype=dtype, zero_points=zp, seed=seed + 10)
    u = make_problem(M, 256, K, bs, dtype=dtype, zero_points=zp, seed=seed + 11)
    pk = lambda p: mnb.mnb_prepack(p.B.to(dev), p.scales.to(dev),
                                   None if p.zero_points is None else p.zero_points.to(dev),
                                   p.N, p.K, bs)
    ops.append(mnb.ChainOp(A1, pk(g), torch.empty(M, 256, dtype=dtype, device=dev), up=pk(u)))
    g.A = u.A = A1.cpu()
    probs.append((g, u))
    s = make_problem(M, 200, 768, bs, dtype=dtype, zero_points=zp, bias=True, seed=seed + 12)
    A2 = s.A.to(dev)
    ops.append(mnb.ChainOp(A2, pk(s), torch.empty(M, 200, dtype=dtype, device=dev),
                           s.bias.to(dev)))
    probs.append(s)
    return ops, probs


def one_by_one(ops):
    """The same calls the graph records: the first three ops as one grouped
    call, the gated pair, the single op."""
    outs = mnb.mnb_matmul_grouped(ops[0].A, [o.weight for o in ops[:3]],
                                  [o.bias for o in ops[:3]])
    outs.append(mnb.mnb_matmul_gate_up(ops[3].A, ops[3].weight, ops[3].up))
    outs.append(mnb.mnb_matmul(ops[4].A, ops[4].weight, ops[4].bias, workspace=None))
    return outs


@pytest.mark.parametrize("M,dtype,bs,zp", [(1, torch.bfloat16, 128, False),
                                           (3, torch.float32, 32, True),
                                           (16, torch.bfloat16, 64, True)])
def test_graph_matches_the_calls_and_the_oracle(dev, M, dtype, bs, zp):
    ops, probs = sequence(dev, M, dtype, bs, zp, seed=M * 100 + bs)
    g = mnb.mnb_graph_build(ops)
    assert g.calls == 3  # q/k/v grouped, the gated pair, the single op
    assert g.kernels >= 3
    for o in ops:
        o.out.fill_(0)
    g.run()
    ref = one_by_one(ops)
    torch.cuda.synchronize()
    for o, r in zip(ops, ref):
        assert torch.equal(o.out, r)
    for o, p in zip(ops, probs):
        if isinstance(p, tuple):
            continue  # the gated pair is compared bitwise above
        R, mag = oracle.matmulnbits(p.A, p.B, p.scales, p.zero_points, p.bias, N=p.N, K=p.K,
                                    block_size=bs)
        check(o.out, R, mag, f"graph op N{p.N}")


def test_graph_run_from_host(dev):
    ops, _ = sequence(dev, 1, torch.bfloat16, 128, False, seed=7)
    g = mnb.mnb_graph_build(ops)
    # Inputs: the first op's activations; outputs: the last op's.
    A_dev, Y_dev = ops[0].A, ops[-1].out
    A_host = torch.randn(A_dev.shape).to(A_dev.dtype).pin_memory()
    Y_host = torch.zeros(Y_dev.shape, dtype=Y_dev.dtype).pin_memory()
    g.run_from_host(A_host, A_dev, Y_dev, Y_host)
    torch.cuda.synchronize()
    assert torch.equal(A_dev.cpu(), A_host)
    assert torch.equal(Y_host, Y_dev.cpu())
    ref = one_by_one(ops)
    torch.cuda.synchronize()
    assert torch.equal(ops[0].out, ref[0])


def test_graph_build_reports_the_failing_op(dev):
    ops, _ = sequence(dev, 1, torch.bfloat16, 128, False, seed=11)
    import dataclasses
    # zero points the weight was not packed with
    bad = dataclasses.replace(ops[-1].weight,
                              packed_zp=torch.zeros(1 << 16, dtype=torch.uint8, device=dev))
    ops[-1] = mnb.ChainOp(ops[-1].A, bad, ops[-1].out)
    with pytest.raises(mnb.MnbError) as e:
        mnb.mnb_graph_build(ops)
    assert e.value.status == -10
