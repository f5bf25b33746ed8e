"""The allocation-free chain entry point, mnb_chain_run_noalloc.

Some callers cannot call cudaMalloc: a plugin whose host runtime owns every
device allocation through its own pool, or a process that reserves all its
device memory up front for weights and caches and must not allocate while
it serves. They cannot hand mnb_chain_build a plan buffer, so this entry
point keeps the plan in a fixed 1 MiB array inside the library.

This file is collected last on purpose. It calls the entry point through the
C ABI twice in a row (the second time with new activations, so a stale plan
or stale counters from the first call would show) and compares every output
with the oracle, within the suite's tolerance; it also runs a chain whose
plan just fits the array, and checks that a chain one op larger than that is
refused with a clear message.
"""
import ctypes

import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300 import binding
from int4_weight_only_matmulnbits_gb300.workloads import make_problem
from tests.tolerance import bound

pytestmark = pytest.mark.gpu

ARRAY_BYTES = 1 << 20  # the library's fixed plan array


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def _prepack(p, dev):
    f = lambda t: None if t is None else t.to(dev)
    return mnb.mnb_prepack(f(p.B), f(p.scales), f(p.zero_points), p.N, p.K, p.block_size)


def _args(ops):
    arr, M = binding._chain_structs(ops)
    w = ops[0].weight
    return (arr, len(ops), M, w.block_size, binding._dtype_code(ops[0].A.dtype),
            binding._dtype_code(w.scale_dtype))


def _noalloc(ops):
    return mnb.load().mnb_chain_run_noalloc(*_args(ops), None)


def _plan_bytes(ops):
    """The plan size a query-only mnb_chain_build reports (no device memory)."""
    info = binding.ChainInfoC()
    st = mnb.load().mnb_chain_build(*_args(ops), None, 0, ctypes.byref(info), None)
    assert st == binding.MNB_OK, mnb.load().mnb_last_error_string().decode()
    return int(info.plan_bytes)


def test_noalloc_chain_matches_the_oracle_twice(dev):
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
    g = torch.Generator().manual_seed(31)
    for call in range(2):
        if call == 1:
            for j, p in enumerate(probs):
                As[j].copy_(torch.randn(M, p.K, generator=g).to(dt).to(dev))
        for o in outs:
            o.fill_(float("nan"))
        st = _noalloc(ops)
        assert st == binding.MNB_OK, mnb.load().mnb_last_error_string().decode()
        torch.cuda.synchronize()
        for j, p in enumerate(probs):
            got = outs[j].float().cpu().double().numpy()
            assert np.all(np.isfinite(got)), (call, j)
            A = As[j].cpu()
            bias = probs[j].bias if j % 2 == 0 else None
            if j == 1:
                # Gated pair: g and u each within the matmul bound, then
                # silu(g) * u (|silu'| <= 1.1) and one bf16 rounding.
                R, gv, uv, mg, mu = oracle.gate_up(
                    A, (p.B, p.scales, p.zero_points, None),
                    (up.B, up.scales, up.zero_points, None), N=p.N, K=p.K, block_size=bs)
                eg, eu = 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5
                silu = gv / (1 + np.exp(-gv))
                b = (1.1 * eg * (np.abs(uv) + eu) + (np.abs(silu) + 1.1 * eg) * eu
                     + 2.0 ** -8 * np.abs(R) + 1e-6 * (np.abs(R) + 1))
            else:
                R, mag = oracle.matmulnbits(A, p.B, p.scales, p.zero_points, bias, N=p.N,
                                            K=p.K, block_size=bs)
                b = bound(mag, R, dt)
            err = np.abs(got - R)
            assert np.all(err <= b), (call, j, float(np.max(err / b)))
    assert mnb.mnb_fault_status() == 0


def test_noalloc_chain_at_the_array_limit(dev):
    """The largest chain of one small op repeated whose plan fits the array
    runs and matches the oracle on every op; one more op is refused with
    MNB_ERR_UNSUPPORTED and a message giving both sizes."""
    p = make_problem(1, 256, 64, 32, dtype=torch.bfloat16, seed=5)
    w = _prepack(p, dev)
    A = p.A.to(dev)
    Y = torch.full((4096, 256), float("nan"), dtype=torch.bfloat16, device=dev)
    ops_of = lambda n: [mnb.ChainOp(A, w, Y[j:j + 1]) for j in range(n)]
    assert _plan_bytes(ops_of(4096)) > ARRAY_BYTES
    lo, hi = 1, 4096  # plan(lo) fits, plan(hi) does not
    assert _plan_bytes(ops_of(lo)) <= ARRAY_BYTES
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _plan_bytes(ops_of(mid)) <= ARRAY_BYTES:
            lo = mid
        else:
            hi = mid
    fits = ops_of(lo)
    assert _plan_bytes(fits) > ARRAY_BYTES - 4096, "the search should end near the limit"
    st = _noalloc(fits)
    assert st == binding.MNB_OK, mnb.load().mnb_last_error_string().decode()
    torch.cuda.synchronize()
    R, mag = oracle.matmulnbits(p.A, p.B, p.scales, None, None, N=p.N, K=p.K, block_size=32)
    got = Y[:lo].float().cpu().double().numpy()
    err = np.abs(got - R)
    assert np.all(err <= bound(mag, R, torch.bfloat16)), float(np.max(err))
    # One op more: refused before anything is enqueued.
    over = ops_of(hi)
    assert _plan_bytes(over) > ARRAY_BYTES
    Y[lo:hi].fill_(float("nan"))
    st = _noalloc(over)
    assert st == binding.MNB_ERR_UNSUPPORTED
    msg = mnb.load().mnb_last_error_string().decode()
    assert "fixed plan array" in msg and str(ARRAY_BYTES) in msg, msg
    assert bool(torch.isnan(Y[lo:hi].float()).all()), "a refused call wrote its output"
    assert mnb.mnb_fault_status() == 0
