"""Failure detection of the bounded waits, on the GPU, without a fault.

With injection point 1 the full-K rotation prepass expects the first stage
(the TMA box of R and the rows of x) but never requests it: every CTA's
bounded wait for it runs out (one wait limit, about 2 s), the kernel records
the timeout in the device error word and returns without writing its outputs;
its other copies in flight are drained, the stage that was never requested is
not waited for again, all CTAs of each cluster still meet at the cluster
barriers, and no CTA writes once any CTA of its cluster has timed out, so
nothing hangs and nothing is written. The
host then reads QMM_ERR_TIMEOUT, and the same call without injection runs on
the same context and matches the oracle.
"""

import numpy as np
import pytest

import qmm_synth
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


def test_rotation_wait_runs_out_and_context_survives(torch_cuda, orc):
    torch = torch_cuda
    q = gc.lib()
    dev = gc.dev()
    M, K, group = 2, 256, 128
    R = qmm_synth.orthogonal_f32(0, "fault/R", K)
    x = qmm_synth.activations_f32(0, "fault/x", M, K)
    Rt, xt = gc.t(R), gc.t(x)
    a = torch.full((M, K), 99, dtype=torch.int8, device=dev)
    sx = torch.full((M, K // group), -1.0, dtype=torch.float32, device=dev)
    assert q.qmm_device_status() == 0
    q.qmm_set_fault_injection(1)
    try:
        q.qmm_prep_act_rotated(M, K, group, Rt, xt, 0, a=a, sx=sx)
    finally:
        q.qmm_set_fault_injection(0)
    flags = q.qmm_device_status()          # synchronises; reads and clears the word
    assert flags & 1, flags                # the timeout bit
    assert (a.cpu().numpy() == 99).all() and (sx.cpu().numpy() == -1.0).all()   # nothing written
    assert q.qmm_device_status() == 0      # cleared
    # the same call without injection, on the same context
    q.qmm_prep_act_rotated(M, K, group, Rt, xt, 0, a=a, sx=sx)
    ra, rsx, _, _ = orc.prep_rotated(R, x, group)
    assert np.array_equal(a.cpu().numpy(), ra)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))
    assert q.qmm_device_status() == 0
