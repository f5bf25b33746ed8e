"""The allocation-free chain entry point, mnb_chain_run_noalloc.

Some callers cannot call cudaMalloc: a plugin whose host runtime owns every
device allocation through its own pool, or a process that reserves all its
device memory up front for weights and caches and must not allocate while
it serves. They cannot hand mnb_chain_build a plan buffer, so this entry
point keeps the plan in a fixed 1 MiB array inside the library.

This file is collected last on purpose. It calls the entry point through the
C ABI twice in a row (the second time with new activations, so a stale plan
or stale counters from the first call would show) and compares each result
with the caller-buffer chain (mnb_chain_build + mnb_chain_run) on the same
ops, within the suite's tolerance; it also checks that a chain too large for
the array is refused with a clear message.
"""

import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300 import binding
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.tolerance import bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def _prepack(p, dev):
    f = lambda t: None if t is None else t.to(dev)
    return mnb.mnb_prepack(f(p.B), f(p.scales), f(p.zero_points), p.N, p.K, p.block_size)


def _noalloc(ops):
    arr, M = binding._chain_structs(ops)
    w = ops[0].weight
    return mnb.load().mnb_chain_run_noalloc(arr, len(ops), M, w.block_size,
                                            binding._dtype_code(ops[0].A.dtype),
                                            binding._dtype_code(w.scale_dtype), None)


def test_noalloc_chain_matches_the_caller_buffer_chain_twice(dev):
    M, bs, dt = 2, 64, torch.bfloat16
    shapes = [(1000, 640), (640, 1000), (257, 640), (96, 257)]
    probs = [make_problem(M, N, K, bs, dtype=dt, zero_points=True, bias=(j % 2 == 0),
                          seed=900 + j) for j, (N, K) in enumerate(shapes)]
    up = make_problem(M, 640, 1000, bs, dtype=dt, zero_points=True, bias=False, seed=950)
    As = [p.A.to(dev) for p in probs]
    outs = [torch.full((M, p.N), float("nan"), dtype=dt, device=dev) for p in probs]
    ops = [mnb.ChainOp(As[0], _prepack(probs[0], dev), outs[0], probs[0].bias.to(dev)),
           mnb.ChainOp(As[1], _prepack(probs[1], dev), outs[1], None, _prepack(up, dev),
                       deps=(0,)),
           mnb.ChainOp(As[2], _prepack(probs[2], dev), outs[2], probs[2].bias.to(dev),
                       deps=(1,)),
           mnb.ChainOp(As[3], _prepack(probs[3], dev), outs[3], None, deps=(0, 2))]
    chain = mnb.mnb_chain_build(ops)
    g = torch.Generator().manual_seed(31)
    for call in range(2):
        if call == 1:
            for j, p in enumerate(probs):
                As[j].copy_(torch.randn(M, p.K, generator=g).to(dt).to(dev))
        for o in outs:
            o.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        want = [o.clone() for o in outs]
        for o in outs:
            o.fill_(float("nan"))
        assert _noalloc(ops) == 0, mnb.load().mnb_last_error_string().decode()
        torch.cuda.synchronize()
        for j, p in enumerate(probs):
            got = outs[j].float().cpu().double().numpy()
            ref = want[j].float().cpu().double().numpy()
            assert np.all(np.isfinite(got)), (call, j)
            # The suite's bound on this op's own activations; for the gated
            # pair, the bound of silu(g) * u given g and u within the matmul
            # bound (|silu'| <= 1.1).
            A = As[j].cpu()
            if j == 1:
                R, gv, uv, mg, mu = oracle.gate_up(
                    A, (p.B, p.scales, p.zero_points, None),
                    (up.B, up.scales, up.zero_points, None), N=p.N, K=p.K, block_size=bs)
                eg, eu = 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5
                silu = gv / (1 + np.exp(-gv))
                b = (1.1 * eg * (np.abs(uv) + eu) + (np.abs(silu) + 1.1 * eg) * eu
                     + 2.0 ** -8 * (np.abs(R) + np.abs(ref)) + 1e-6)
            else:
                _, mag = oracle.matmulnbits(A, p.B, p.scales, p.zero_points, None, N=p.N,
                                            K=p.K, block_size=bs)
                b = bound(mag, ref, dt)
            assert np.all(np.abs(got - ref) <= b), (call, j, float(np.max(np.abs(got - ref) / b)))
    assert mnb.mnb_fault_status() == 0


def test_noalloc_chain_refuses_a_plan_larger_than_its_array(dev):
    """4096 ops of 16 tiles each need far more than the 1 MiB array."""
    p = make_problem(1, 256, 64, 32, dtype=torch.bfloat16, seed=5)
    w = _prepack(p, dev)
    A = p.A.to(dev)
    Y = torch.empty(4096, 256, dtype=torch.bfloat16, device=dev)
    ops = [mnb.ChainOp(A, w, Y[j:j + 1]) for j in range(4096)]
    st = _noalloc(ops)
    assert st == -8
    msg = mnb.load().mnb_last_error_string().decode()
    assert "fixed plan array" in msg and "1048576" in msg, msg
