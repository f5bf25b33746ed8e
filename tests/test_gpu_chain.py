"""GPU parity of the decode chain (mnb_chain_build / mnb_chain_run): many
MatMulNBits projections, and gated-MLP pairs, in one persistent launch.

Every op's result is compared with the double-precision oracle on the same
host inputs. Where an op reads an earlier op's output, the comparison uses
a composed bound computed from oracle quantities only: with R_prev the
oracle's previous output and B_prev its bound, the GPU's input differs from
R_prev by at most B_prev, so

  |Y - R| <= 2e-3 * sum|(|R_prev| + B_prev) w| + 1e-5 + sum|w| B_prev
             + u_out * (|R| + sum|w| B_prev)

(the matmul tolerance on the perturbed input, its propagation through the
weights, and the output rounding)."""
import numpy as np
import pytest
import torch

import int4_weight_only_matmulnbits_gb300 as mnb
import oracle
from int4_weight_only_matmulnbits_gb300.workloads import QWEN3_4B, make_problem
from tests.tolerance import U_OUT, check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mnb.build_library()
    mnb.load()
    return torch.device("cuda:0")


def f(t, dev):
    return None if t is None else t.to(dev)


def prepack(prob, dev):
    return mnb.mnb_prepack(f(prob.B, dev), f(prob.scales, dev), f(prob.zero_points, dev),
                           prob.N, prob.K, prob.block_size)


def pair_bound(gv, uv, R, eg, eu, dtype):
    """Bound of silu(g) * u given |g - gv| <= eg, |u - uv| <= eu (|silu'| <= 1.1)."""
    silu = gv / (1 + np.exp(-gv))
    return (1.1 * eg * (np.abs(uv) + eu) + (np.abs(silu) + 1.1 * eg) * eu
            + (2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24) * np.abs(R)
            + 1e-6 * (np.abs(R) + 1))


def independent_ops(dev, shapes, M, bs, dtype, with_zp, seed):
    """One op per (N, K, paired) with its own seeded inputs."""
    ops, refs = [], []
    for i, (N, K, paired) in enumerate(shapes):
        g = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp, bias=(i % 2 == 0),
                         seed=seed + 10 * i)
        A = f(g.A, dev)
        out = torch.full((M, N), float("nan"), dtype=dtype, device=dev)
        if paired:
            u = make_problem(M, N, K, bs, dtype=dtype, zero_points=with_zp, bias=(i % 2 == 0),
                             seed=seed + 10 * i + 1)
            ops.append(mnb.ChainOp(A, prepack(g, dev), out, f(g.bias, dev), prepack(u, dev),
                                   f(u.bias, dev)))
            refs.append(("pair", g, u))
        else:
            ops.append(mnb.ChainOp(A, prepack(g, dev), out, f(g.bias, dev)))
            refs.append(("single", g, None))
    return ops, refs


def check_independent(ops, refs, what):
    for j, (kind, g, u) in enumerate(refs):
        Y = ops[j].out
        if kind == "single":
            R, mag = oracle.matmulnbits(g.A, g.B, g.scales, g.zero_points, g.bias, N=g.N,
                                        K=g.K, block_size=g.block_size)
            check(Y, R, mag, f"{what} op {j}")
        else:
            R, gv, uv, mg, mu = oracle.gate_up(
                g.A, (g.B, g.scales, g.zero_points, g.bias),
                (u.B, u.scales, u.zero_points, u.bias), N=g.N, K=g.K,
                block_size=g.block_size)
            Yh = Y.float().cpu().double().numpy()
            b = pair_bound(gv, uv, R, 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5, Y.dtype)
            err = np.abs(Yh - R)
            assert np.all(np.isfinite(Yh)), (what, j)
            assert np.all(err <= b), (what, j, float(np.max(err / b)))


RAGGED = [(7, 33, False), (129, 257, True), (1000, 700, False), (33, 1000, True),
          (16, 64, False), (5, 130, False), (300, 17, True), (1, 1, False)]


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_zp", [False, True])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_chain_independent_ops(dev, bs, dtype, with_zp, M):
    """Ragged N and K, partial last blocks, single ops and gated pairs, no
    dependencies between ops."""
    ops, refs = independent_ops(dev, RAGGED, M, bs, dtype, with_zp, seed=1000 * bs + M)
    chain = mnb.mnb_chain_build(ops)
    chain.run()
    torch.cuda.synchronize()
    check_independent(ops, refs, f"bs{bs} M{M}")


@pytest.mark.parametrize("bs", [32, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chain_declared_deps_and_reruns(dev, bs, dtype):
    """The same ops with every op depending on the one before (the schedule
    then serialises them); three runs give bitwise identical outputs, so
    the completion counters are reset between launches."""
    ops, refs = independent_ops(dev, RAGGED, 2, bs, dtype, True, seed=77 + bs)
    for j in range(1, len(ops)):
        ops[j].deps = (j - 1,)
    chain = mnb.mnb_chain_build(ops)
    outs = []
    for _ in range(3):
        for o in ops:
            o.out.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        outs.append([o.out.clone() for o in ops])
    check_independent(ops, refs, f"deps bs{bs}")
    for r in outs[1:]:
        for a, b in zip(outs[0], r):
            assert torch.equal(a, b)
    assert mnb.mnb_fault_status() == 0


def chained_problem(dims, M, bs, dtype, with_zp, seed):
    """Weights of a chain where op j reads op j-1's output: dims = [K0, N0=K1,
    N1=K2, ...]; op 0 reads a seeded A."""
    probs = []
    for j in range(len(dims) - 1):
        probs.append(make_problem(M, dims[j + 1], dims[j], bs, dtype=dtype,
                                  zero_points=with_zp, bias=(j % 2 == 1), seed=seed + j))
    return probs


def dequant(p):
    return oracle.dequantize(p.B, p.scales, p.zero_points, N=p.N, K=p.K,
                             block_size=p.block_size)


def lin_bound(p, A, B, bias):
    """Oracle output for a double input A known to within B, and the bound
    (matmul tolerance on the perturbed input plus propagation), before the
    output rounding. The dense products are numpy's, on the oracle's
    dequantized weight."""
    W = dequant(p)
    R = A @ W.T + (0.0 if bias is None else bias.double().numpy())
    mag_in = (np.abs(A) + B) @ np.abs(W).T
    prop = B @ np.abs(W).T
    return R, 2e-3 * mag_in + 1e-5 + prop, prop


def composed_refs(probs, A0):
    """Oracle chain in double, with the composed bound of each output."""
    refs = []
    A = A0.double().numpy()
    B = np.zeros_like(A)
    for p in probs:
        R, e, prop = lin_bound(p, A, B, p.bias)
        bound = e + U_OUT[p.A.dtype] * (np.abs(R) + prop)
        refs.append((R, bound))
        A, B = R, bound
    return refs


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 4])
def test_chain_reads_earlier_outputs(dev, bs, dtype, M):
    """Op j reads op j-1's output (outputs start as NaN, so reading one too
    early is caught), across ragged widths; each run also restages the
    first op's new activations."""
    dims = [700, 1000, 257, 2560, 129, 640]
    probs = chained_problem(dims, M, bs, dtype, True, seed=500 + bs + M)
    A0 = f(probs[0].A, dev)
    outs = [torch.full((M, p.N), float("nan"), dtype=dtype, device=dev) for p in probs]
    ops = []
    for j, p in enumerate(probs):
        A = A0 if j == 0 else outs[j - 1]
        ops.append(mnb.ChainOp(A, prepack(p, dev), outs[j], f(p.bias, dev),
                               deps=(() if j == 0 else (j - 1,))))
    chain = mnb.mnb_chain_build(ops)
    for trial in range(2):
        if trial == 1:
            g = torch.Generator().manual_seed(4242)
            newA = torch.randn(M, dims[0], generator=g).to(dtype)
            A0.copy_(newA.to(dev))
            probs[0].A = newA
            for o in outs:
                o.fill_(float("nan"))
        chain.run()
        torch.cuda.synchronize()
        refs = composed_refs(probs, probs[0].A)
        for j, (R, bound) in enumerate(refs):
            Y = outs[j].float().cpu().double().numpy()
            assert np.all(np.isfinite(Y)), (trial, j)
            err = np.abs(Y - R)
            assert np.all(err <= bound), (trial, j, float(np.max(err / bound)))


def test_chain_gated_pair_reads_earlier_output(dev):
    """A gated pair whose activations are an earlier op's output, followed
    by the down projection reading the pair's output."""
    M, bs, dtype = 2, 64, torch.bfloat16
    x = make_problem(M, 640, 300, bs, dtype=dtype, zero_points=False, bias=True, seed=5)
    gt = make_problem(M, 1000, 640, bs, dtype=dtype, zero_points=False, bias=False, seed=6)
    up = make_problem(M, 1000, 640, bs, dtype=dtype, zero_points=False, bias=True, seed=7)
    dn = make_problem(M, 200, 1000, bs, dtype=dtype, zero_points=False, bias=False, seed=8)
    A0 = f(x.A, dev)
    y0 = torch.full((M, 640), float("nan"), dtype=dtype, device=dev)
    y1 = torch.full((M, 1000), float("nan"), dtype=dtype, device=dev)
    y2 = torch.full((M, 200), float("nan"), dtype=dtype, device=dev)
    ops = [mnb.ChainOp(A0, prepack(x, dev), y0, f(x.bias, dev)),
           mnb.ChainOp(y0, prepack(gt, dev), y1, None, prepack(up, dev), f(up.bias, dev),
                       deps=(0,)),
           mnb.ChainOp(y1, prepack(dn, dev), y2, None, deps=(1,))]
    chain = mnb.mnb_chain_build(ops)
    chain.run()
    torch.cuda.synchronize()
    # op 0
    (R0, B0), = composed_refs([x], x.A)
    Y0 = y0.float().cpu().double().numpy()
    assert np.all(np.abs(Y0 - R0) <= B0)
    # op 1: g, u perturbed through their inputs, then the pair bound
    gv, eg, _ = lin_bound(gt, R0, B0, gt.bias)
    uv, eu, _ = lin_bound(up, R0, B0, up.bias)
    R1 = gv / (1 + np.exp(-gv)) * uv
    B1 = pair_bound(gv, uv, R1, eg, eu, dtype)
    Y1 = y1.float().cpu().double().numpy()
    assert np.all(np.abs(Y1 - R1) <= B1), float(np.max(np.abs(Y1 - R1) / B1))
    # op 2
    R2, e2, prop2 = lin_bound(dn, R1, B1, None)
    B2 = e2 + 2.0 ** -8 * (np.abs(R2) + prop2)
    Y2 = y2.float().cpu().double().numpy()
    assert np.all(np.abs(Y2 - R2) <= B2), float(np.max(np.abs(Y2 - R2) / B2))


def test_chain_qwen3_4b_layers(dev):
    """Two Qwen3-4B decoder layers' projections and the LM head at full
    shapes (M = 1, bf16, bs 128, no zero points), with the decoder's
    dependency structure: q/k/v <- previous down, o <- q, k, v, gate/up <- o,
    down <- gate/up, lm_head <- last down. Every op reads its own seeded
    activations; outputs are checked on seeded column samples."""
    proj = {p.name: p for p in QWEN3_4B["projections"]}
    ops, refs = [], []
    prev_down = -1
    seed = 3000
    for layer in range(2):
        base = len(ops)
        for name in ("q", "k", "v"):
            p = proj[name]
            pr = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed,
                              scale_range=(0.002, 0.01))
            seed += 1
            out = torch.full((1, p.N), float("nan"), dtype=torch.bfloat16, device=dev)
            ops.append(mnb.ChainOp(f(pr.A, dev), prepack(pr, dev), out,
                                   deps=(() if prev_down < 0 else (prev_down,))))
            refs.append(("single", pr, None))
        p = proj["o"]
        pr = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed,
                          scale_range=(0.002, 0.01))
        seed += 1
        ops.append(mnb.ChainOp(f(pr.A, dev), prepack(pr, dev),
                               torch.empty((1, p.N), dtype=torch.bfloat16, device=dev),
                               deps=(base, base + 1, base + 2)))
        refs.append(("single", pr, None))
        p = proj["gate"]
        g = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed,
                         scale_range=(0.002, 0.01))
        u = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed + 1,
                         scale_range=(0.002, 0.01))
        u.A = g.A
        seed += 2
        ops.append(mnb.ChainOp(f(g.A, dev), prepack(g, dev),
                               torch.empty((1, p.N), dtype=torch.bfloat16, device=dev),
                               None, prepack(u, dev), deps=(base + 3,)))
        refs.append(("pair", g, u))
        p = proj["down"]
        pr = make_problem(1, p.N, p.K, 128, dtype=torch.bfloat16, seed=seed,
                          scale_range=(0.002, 0.01))
        seed += 1
        ops.append(mnb.ChainOp(f(pr.A, dev), prepack(pr, dev),
                               torch.empty((1, p.N), dtype=torch.bfloat16, device=dev),
                               deps=(base + 4,)))
        refs.append(("single", pr, None))
        prev_down = base + 5
    lm = make_problem(1, 151936, 2560, 128, dtype=torch.bfloat16, seed=seed,
                      scale_range=(0.002, 0.01))
    ops.append(mnb.ChainOp(f(lm.A, dev), prepack(lm, dev),
                           torch.empty((1, 151936), dtype=torch.bfloat16, device=dev),
                           deps=(prev_down,)))
    refs.append(("single", lm, None))
    chain = mnb.mnb_chain_build(ops)
    chain.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    rows = np.array([0])
    for j, (kind, g, u) in enumerate(refs):
        cols = np.sort(rng.choice(g.N, min(g.N, 256), replace=False))
        Y = ops[j].out
        if kind == "single":
            R, mag = oracle.matmulnbits(g.A, g.B, g.scales, None, None, N=g.N, K=g.K,
                                        block_size=128, rows=rows, cols=cols)
            check(Y[:, cols], R, mag, f"qwen3-4b op {j}")
        else:
            R, gv, uv, mg, mu = oracle.gate_up(g.A, (g.B, g.scales, None, None),
                                               (u.B, u.scales, None, None), N=g.N, K=g.K,
                                               block_size=128, rows=rows, cols=cols)
            Yh = Y[:, cols].float().cpu().double().numpy()
            b = pair_bound(gv, uv, R, 2e-3 * mg + 1e-5, 2e-3 * mu + 1e-5, Y.dtype)
            assert np.all(np.abs(Yh - R) <= b), j
    assert mnb.mnb_fault_status() == 0
