"""GPU parity of the full-K orthogonal rotation prepass and the orthogonal
lm_head built on it (weights stored as W R^T, one norm per row viewed as
128-wide groups).

Bit-exact: the int8 codes, their fp16 image, the activation scales and the
code sums (z = R x is accumulated by ascending fused multiply-adds on both
sides). Tolerance of the fp32 outputs, as for the symmetric variant:
|d| <= 1e-5 * sum_g |cb_scale sw sx P| + 1e-6.
"""

import numpy as np
import pytest

import qmm_synth
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

W4A8, CQ4 = 0, 2


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


_ROT = {}


def rotation(K):
    if K not in _ROT:
        _ROT[K] = qmm_synth.orthogonal_f32(0, f"rot/R/{K}", K)
    return _ROT[K]


def _input(x, x_dtype):
    import torch
    xt = torch.from_numpy(x)
    if x_dtype == 1:
        xt = xt.to(torch.float16)
    elif x_dtype == 2:
        xt = xt.to(torch.bfloat16)
    return xt, xt.float().numpy()


def prep_rotated(R, xin, M, K, group, x_dtype):
    import torch
    q = gc.lib()
    dev = gc.dev()
    G = K // group
    a = gc.guarded((M, K), torch.int8, 99)
    a16 = gc.guarded((M, K), torch.float16, 99.0)
    sx = gc.guarded((M, G), torch.float32, float("nan"))
    asum = gc.guarded((M, G), torch.int32, -1)
    q.qmm_prep_act_rotated(M, K, group, gc.t(R), xin.to(dev), x_dtype, a=a, a16=a16, sx=sx, asum=asum)
    assert q.qmm_last_kernel_id() == 12
    return a, a16, sx, asum


CASES = [
    (1, 1536, 128, 0.01),    # lm_head decode row
    (1, 128, 128, 0.0),      # one k-chunk, one cluster
    (3, 256, 64, 0.01),      # group 64: two groups per cluster
    (9, 384, 128, 0.0),      # two row blocks, ragged
    (17, 1536, 64, 0.01),
    (33, 1536, 128, 0.01),   # lm_head batch: five row blocks
    (2, 2048, 128, 0.0),     # more k-chunks than ring stages (16 > 8)
]


@pytest.mark.parametrize("M,K,group,outl", CASES)
@pytest.mark.parametrize("x_dtype", [0, 1, 2])
def test_prep_rotated_bit_exact(torch_cuda, orc, M, K, group, outl, x_dtype):
    if x_dtype and M > 9:
        pytest.skip("dtype variants on the small shapes only")
    R = rotation(K)
    x = qmm_synth.activations_f32(4, f"rot/x/{M}/{K}", M, K, outlier_frac=outl)
    if M > 1:
        x[1, :] = 0.0        # an all-zero row: zero codes, zero scales
    xin, xval = _input(x, x_dtype)
    a, a16, sx, asum = prep_rotated(R, xin, M, K, group, x_dtype)
    ra, rsx, rsum, _ = orc.prep_rotated(R, xval, group)
    assert np.array_equal(a.cpu().numpy(), ra)
    assert np.array_equal(a16.cpu().numpy(), ra.astype(np.float16))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))
    assert np.array_equal(asum.cpu().numpy(), rsum)


def test_prep_rotated_order_fixture(torch_cuda, orc):
    """The hand-worked summation-order case of the oracle's fixture on the GPU:
    output 0 sums 2^24, 1, -2^24, 1 (ascending, fused: 1; any other order: 2)
    and is the group's largest value, so sx = fp32(z0 / 127) tells the orders
    apart; outputs 4.. carry small values whose codes depend on sx too."""
    import torch
    K, group = 128, 128
    R = np.eye(K, dtype=np.float32)
    R[0, :4] = 1.0
    R[1:4, 1:4] = 0.0
    x = np.zeros((1, K), dtype=np.float32)
    x[0, :4] = [16777216.0, 1.0, -16777216.0, 1.0]
    x[0, 4:] = (0.01 * qmm_synth.normal(7, "rot/fixture", K - 4)).astype(np.float32)
    a, a16, sx, asum = prep_rotated(R, torch.from_numpy(x), 1, K, group, 0)
    ra, rsx, rsum, z = orc.prep_rotated(R, x, group)
    assert z[0, 0] == 1.0 and rsx[0, 0] == np.float32(1.0) / np.float32(127.0)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))
    assert np.array_equal(a.cpu().numpy(), ra) and np.array_equal(asum.cpu().numpy(), rsum)


def test_prep_rotated_control_orientation_is_detected(torch_cuda, orc):
    """Control: the codes of R^T x differ from those of R x."""
    K, group = 256, 64
    R = rotation(K)
    x = qmm_synth.activations_f32(5, "rot/control", 2, K)
    a, _, _, _ = prep_rotated(R, _input(x, 0)[0], 2, K, group, 0)
    ra, _, _, _ = orc.prep_rotated(np.ascontiguousarray(R.T), x, group)
    assert not np.array_equal(a.cpu().numpy(), ra)


def _orth_lm_head(N, K, seed):
    """CQ4 weights of W R^T with one fp16 norm per row, repeated in every
    128-wide group (the virtual group view)."""
    idx, _, C, cb, _ = gc.cq4_case(seed, f"orth/{N}/{K}", N, K, 128, 0, 1)
    norms = qmm_synth.uniform_f16(seed, f"orth/{N}/{K}/norms", (N, 1), 0.005, 0.02)
    sw = np.ascontiguousarray(np.repeat(norms, K // 128, axis=1))
    return idx, sw, C, cb


@pytest.mark.parametrize("N,K,M,rows", [(4096, 1536, 1, None), (2000, 1536, 5, None),
                                        (262144, 1536, 1, 512)])
def test_orth_lm_head_end_to_end(torch_cuda, orc, N, K, M, rows):
    """Rotated prepass then the GEMV (M = 1) or GEMM on the rotated weights,
    against the oracle's own prepass and output; at the full lm_head size on
    sampled rows (the first, the last and a seeded spread)."""
    import torch
    R = rotation(K)
    idx, sw, C, cb = _orth_lm_head(N, K, 6)
    x = qmm_synth.activations_f32(6, f"orth/x/{N}", M, K, outlier_frac=0.01)
    a, a16, sx, _ = prep_rotated(R, torch.from_numpy(x), M, K, 128, 0)
    d, packed = gc.pack_cq4(N, K, 128, idx, C, cb, sw)
    if M == 1:
        y = gc.gemv(d, packed, a.reshape(-1), sx.reshape(-1)).cpu().numpy()[None]
    else:
        y = gc.gemm(d, packed, M, a16, sx).cpu().numpy()
    ra, rsx, _, _ = orc.prep_rotated(R, x, 128)
    if rows is None:
        sel = np.arange(N)
    else:
        sel = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(0).integers(0, N, rows)]))
    Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, 128, rows=sel.astype(np.int32))
    ok, worst = gc.within_w4a8(y[:, sel], Y, Ym)
    assert ok, worst
