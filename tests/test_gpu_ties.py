"""Round-half-to-even on the GPU, by design rather than by chance.

The method quantizes each group of activations as a = clamp(rint(v / s), -127,
127) with s = amax / 127 and ties to even. Random inputs almost never land on
an exact tie, so these inputs are built to: in every group one element is
127 * s with s a power of two (so s = amax / 127 is exact), and the others
are (k + 1/2) * s for half-integers of both signs and both parities, from
+-0.5 up to +-126.5, so v / s is an exact tie. With the in-group Walsh-Hadamard
rotation the tie values are placed on the rotated vector z and x = H z / n is
fed in (every value is a short dyadic fraction, so the kernel's fp32 transform
reproduces z exactly). The codes of qmm_prep_act, of the fused decode GEMV's
prepass and of the full-K rotation prepass (with an identity and a signed
permutation as the rotation, which move values exactly) must equal the
oracle's bit for bit, and the tie positions must round to the even neighbour.
The largest tie is +-126.5: a tie at the clamp edge (+-127.5) cannot occur,
since every |v| is at most amax = 127 s, so |v / s| never exceeds 127 by more
than the division's rounding.
"""

import numpy as np
import pytest

from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

# half-integers k + 1/2: both signs, even and odd k, small and at the edge
HALVES = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, -3.5, 10.5, 11.5, -10.5, -11.5,
                   63.5, 64.5, -63.5, -64.5, 125.5, 126.5, -125.5, -126.5], dtype=np.float64)


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


def _tie_groups(M, K, group, seed):
    """z [M][K] float64 with exact ties in every group, and the tie mask.
    Element 0 of a group (at a seeded position) is +-127 s (the amax); the
    others cycle through HALVES (rotated per group) times s; a few are 0."""
    rng = np.random.default_rng(seed)
    z = np.zeros((M, K), dtype=np.float64)
    tie = np.zeros((M, K), dtype=bool)
    exps = [-3, 0, -7, 2]
    for m in range(M):
        for g0 in range(0, K, group):
            s = 2.0 ** exps[(m + g0 // group) % len(exps)]
            vals = np.roll(HALVES, g0 // group + m)
            idx = rng.permutation(group)
            top = idx[0]
            z[m, g0 + top] = 127.0 * s * (1 if (m + g0) % 2 == 0 else -1)
            for j, p in enumerate(idx[1:group - 4]):
                z[m, g0 + p] = vals[j % len(vals)] * s
                tie[m, g0 + p] = True
    return z, tie


def _check_codes(a_gpu, ra, z, tie, s_of):
    assert np.array_equal(a_gpu, ra), "codes differ from the oracle"
    # the crafted ties round to the even neighbour (np.rint rounds half to even)
    want = np.rint(z / s_of)
    assert np.array_equal(a_gpu[tie].astype(np.float64), want[tie])
    assert (np.abs(a_gpu[tie].astype(np.int64)) % 2 == 0).all()


def _scale_per_element(z, group):
    M, K = z.shape
    amax = np.abs(z.reshape(M, K // group, group)).max(axis=2)
    return np.repeat(amax / 127.0, group, axis=1)


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("x_dtype", [0, 1, 2])
def test_prep_ties_no_rotation(torch_cuda, orc, group, x_dtype):
    M, K = 6, 512
    z, tie = _tie_groups(M, K, group, 31 + group + x_dtype)
    x = z.astype(np.float32)   # exact in fp32, fp16 and bf16 (at most 9 significant bits)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, 0, x_dtype)
    ra, rsx, _ = orc.prep_w4a8(x, group, 0)
    _check_codes(a.cpu().numpy(), ra, z, tie, _scale_per_element(z, group))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))


def _hadamard_input(z, group):
    """x with FWHT(x) = z in every group (x = H z / n, Sylvester order)."""
    from scipy.linalg import hadamard
    H = hadamard(group).astype(np.float64)
    M, K = z.shape
    x = (z.reshape(M, K // group, group) @ H.T / group).reshape(M, K)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x), "not exact in fp32"
    return x.astype(np.float32)


@pytest.mark.parametrize("group", [64, 128])
def test_prep_ties_with_rotation(torch_cuda, orc, group):
    M, K = 5, 768
    z, tie = _tie_groups(M, K, group, 47 + group)
    x = _hadamard_input(z, group)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, group, 0)
    ra, rsx, _ = orc.prep_w4a8(x, group, group)
    _check_codes(a.cpu().numpy(), ra, z, tie, _scale_per_element(z, group))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))


@pytest.mark.parametrize("group,had", [(64, 0), (64, 64), (128, 128)])
def test_fused_gemv_prepass_ties(torch_cuda, orc, group, had):
    torch = torch_cuda
    q = gc.lib()
    N, K = 384, 1536
    z, tie = _tie_groups(1, K, group, 53 + group + had)
    x = _hadamard_input(z, group) if had else z.astype(np.float32)
    qb, sw, _ = gc.w4a8_case(54, f"ties/fused/{group}/{had}", N, K, group, had, 1)
    d, packed = gc.pack(gc.W4A8, N, K, group, qb, sw)
    y = gc.guarded((N,), torch.float32, float("nan"))
    a = gc.guarded(K, torch.int8)
    sx = gc.guarded(K // group, torch.float32)
    q.qmm_gemv_fused(d, packed, gc.t(x[0]), 0, had, y, a_out=a, sx_out=sx)
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    _check_codes(a.cpu().numpy()[None, :], ra, z, tie, _scale_per_element(z, group))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx[0].view(np.uint32))
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(y.cpu().numpy()[None, :], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


@pytest.mark.parametrize("rotation", ["identity", "signed_permutation"])
@pytest.mark.parametrize("group", [64, 128])
def test_rotated_prepass_ties(torch_cuda, orc, rotation, group):
    torch = torch_cuda
    q = gc.lib()
    M, K = 3, 512
    rng = np.random.default_rng(61 + group)
    if rotation == "identity":
        R = np.eye(K, dtype=np.float32)
    else:
        perm = rng.permutation(K)
        sign = np.where(rng.integers(0, 2, K) == 1, -1.0, 1.0)
        R = np.zeros((K, K), dtype=np.float32)
        R[np.arange(K), perm] = sign   # z[i] = sign[i] * x[perm[i]]
    z, tie = _tie_groups(M, K, group, 67 + group)
    # x such that R x = z exactly (R orthogonal with entries in {-1, 0, 1})
    x = (R.T.astype(np.float64) @ z.T).T.astype(np.float32)
    a = gc.guarded((M, K), torch.int8)
    sx = gc.guarded((M, K // group), torch.float32)
    q.qmm_prep_act_rotated(M, K, group, gc.t(R), gc.t(x), 0, a=a, sx=sx)
    ra, rsx, _, rz = orc.prep_rotated(R, x, group)
    assert np.array_equal(rz.astype(np.float64), z), "the rotation does not move the ties exactly"
    _check_codes(a.cpu().numpy(), ra, z, tie, _scale_per_element(z, group))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))
    assert q.qmm_device_status() == 0
