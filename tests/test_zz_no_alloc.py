"""The allocation-free GEMV entry point (qmm_gemv_static_scratch).

It is for callers that cannot allocate device memory, such as code running
inside a host program that owns every device allocation, or a latency-critical
loop that must not reach cudaMalloc. It must give the same results as qmm_gemv
with a caller-provided workspace, call after call, although every call reuses
the library's one fixed scratch array. This file is collected last so that a
run stopping at its first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest

from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

CASES = [
    (1536, 6144, 64, 64),     # down: the largest split over K
    (12288, 1536, 64, 64),    # gate_up
    (1024, 1024, 64, 0),
    (200, 192, 64, 64),       # ragged rows
    (256, 512, 128, 128),
]


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.mark.parametrize("N,K,group,had", CASES)
def test_static_scratch_matches_workspace_gemv_twice(torch_cuda, orc, N, K, group, had):
    torch = torch_cuda
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(21, f"noalloc/{N}/{K}", N, K, group, had, 1, 0.01)
    d, packed = gc.pack(0, N, K, group, qb, sw)
    assert 0 < q.qmm_gemv_workspace_size(d) <= (1 << 20)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, had)
    ref = gc.gemv(d, packed, a, sx, workspace=True).cpu().numpy()
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    for call in range(2):
        y = gc.guarded((N,), torch.float32, float("nan"))
        # through the C ABI directly
        st = q.library().qmm_gemv_static_scratch(ctypes.byref(d), packed.data_ptr(), a.data_ptr(),
                                                 sx.data_ptr(), y.data_ptr(),
                                                 torch.cuda.current_stream().cuda_stream)
        assert st == 0, q.status_string(st)
        out = y.cpu().numpy()
        ok, worst = gc.within_w4a8(out[None, :], Y, Ym)
        assert ok, f"call {call}: worst error / bound = {worst}"
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-5 * float(np.abs(Ym).max()) + 1e-6)
    assert q.qmm_device_status() == 0


def test_static_scratch_rejects_without_touching_the_device(torch_cuda):
    q = gc.lib()
    L = q.library()
    # affine weights have no GEMV; misaligned pointers are refused
    d_aff = q.weight_desc(1, 256, 256, 64)
    assert L.qmm_gemv_static_scratch(ctypes.byref(d_aff), 256, 256, 256, 256, None) == 2
    d = q.weight_desc(0, 1536, 6144, 64)
    assert L.qmm_gemv_static_scratch(ctypes.byref(d), 256, 257, 256, 256, None) == 4
    assert L.qmm_gemv_static_scratch(None, 256, 256, 256, 256, None) == 1
