"""Failure detection on the GPU, without a GPU fault: a bounded wait is made
to run out on purpose and must come back as a status, not as a hang or a
trap.

mnb_test_wait_fault makes CTA 0's producer of the decode kernel stop before
its first weight stage, in a separate instantiation of the kernel with a
short wait cap (2^16 iterations). Its consumers then wait for a
stage that never arrives, give up after the cap, record fault bit 1 and end
the launch; every copy that was issued (the activation row) has landed by
then. The test checks that the launch ends, that mnb_fault_status reports the
bit (and clears it), and that the next normal call on the same stream
matches the oracle: the context stays usable.
"""
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


def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_correct(dev):
    # Many 16-row tiles: the decode kernel works without clusters here; bf16
    # activations and scales, bs 128, no zero points: the probed configuration.
    prob = make_problem(1, 32768, 1024, 128, dtype=torch.bfloat16, seed=21,
                        scale_range=(0.002, 0.01))
    w = mnb.mnb_prepack(prob.B.to(dev), prob.scales.to(dev), None, 32768, 1024, 128)
    A = prob.A.to(dev)
    torch.cuda.synchronize()
    assert mnb.mnb_fault_status() == 0
    mnb.mnb_test_wait_fault(stop_stage=0)
    try:
        mnb.mnb_matmul(A, w)
        torch.cuda.synchronize()  # the launch ends: every wait is bounded
    finally:
        mnb.mnb_test_wait_fault()
    assert mnb.mnb_fault_status() & 1
    assert mnb.mnb_fault_status() == 0  # reading the bits clears them
    Y = mnb.mnb_matmul(A, w)
    torch.cuda.synchronize()
    R, mag = oracle.matmulnbits(prob.A, prob.B, prob.scales, None, None, N=32768, K=1024,
                                block_size=128)
    check(Y, R, mag, "after the reported fault")
    assert mnb.mnb_fault_status() == 0
