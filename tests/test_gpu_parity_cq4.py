"""GPU parity of the codebook 4-bit (CQ4) weights against the CPU oracle.

Bit-exact: packed bytes (chunks and codebook trailer), int32 group partials
of the GEMV and tensor-core kernels. Tolerance for fp32 outputs, as for the
symmetric variant: |d| <= 1e-5 * sum_g |cb_scale sw sx P| + 1e-6. Codebooks
are seeded draws (16 distinct int8 levels), plus the identity levels -8..7
(which must reproduce the symmetric variant) and extreme levels (-128, 127).
"""

import numpy as np
import pytest

from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

W4A8, CQ4 = 0, 2
GEMV, GEMM = 0, 1


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


def _extreme_book():
    return np.array([-128, 127, -128, 127, 0, -1, 1, -127, 127, -128, 64, -64, 5, -5, 127, -128], dtype=np.int8)


def _relabel(idx_bytes, C):
    """(idx2, C2) naming the same levels through other indices."""
    perm = (np.arange(16) * 5 + 11) % 16
    inv = np.argsort(perm)
    i = np.empty((idx_bytes.shape[0], idx_bytes.shape[1] * 2), dtype=np.int64)
    i[:, 0::2], i[:, 1::2] = idx_bytes & 0xF, idx_bytes >> 4
    i2 = inv[i]
    return (i2[:, 0::2] | (i2[:, 1::2] << 4)).astype(np.uint8), C[perm]


# ------------------------------------------------------------------ pack

PACK_CASES = [(1024, 1024, 64), (200, 192, 64), (130, 512, 128), (1, 64, 64), (12288, 1536, 64)]


@pytest.mark.parametrize("N,K,group", PACK_CASES)
def test_pack_bytes(torch_cuda, orc, N, K, group):
    idx, sw, C, cb, _ = gc.cq4_case(1, f"cq4/pack/{N}/{K}", N, K, group, 0, 1)
    _, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    ref = orc.pack_cq4(N, K, group, idx, C, cb, sw)
    assert np.array_equal(packed.cpu().numpy(), ref)


# ------------------------------------------------------------------ GEMV

GEMV_CASES = [
    (1024, 1024, 64, 0, 0.0),
    (200, 192, 64, 64, 0.0),      # ragged rows
    (256, 512, 128, 128, 0.0),
    (128, 64, 64, 0, 0.0),        # one group
    (12288, 1536, 64, 64, 0.01),  # gate_up
    (1536, 6144, 64, 64, 0.01),   # down
]


@pytest.mark.parametrize("book", ["seeded", "identity", "extreme"])
@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES)
def test_gemv_partials_bit_exact(torch_cuda, orc, N, K, group, had, outl, book):
    idx, sw, C, cb, x = gc.cq4_case(6, f"cq4/gemv/{N}/{K}", N, K, group, had, 1, outl)
    if book == "identity":
        C = np.arange(-8, 8, dtype=np.int8)
    elif book == "extreme":
        C = _extreme_book()
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    a, _, _, _, _ = gc.prep_w4a8(x, group, had)
    P = gc.partials(d, packed, 1, GEMV, a)
    assert gc.lib().qmm_last_kernel_id() == 10
    ra, _, _ = orc.prep_w4a8(x, group, had)
    ref = orc.partials_cq4(idx, C, ra, group)
    assert np.array_equal(P.cpu().numpy(), ref)
    if book == "identity":   # the symmetric variant's partials of q = index - 8
        assert np.array_equal(ref, orc.partials_w4a8((idx ^ 0x88).astype(np.uint8), ra, group))


@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES)
@pytest.mark.parametrize("workspace", [True, False])
def test_gemv_output(torch_cuda, orc, N, K, group, had, outl, workspace):
    idx, sw, C, cb, x = gc.cq4_case(7, f"cq4/gemv/{N}/{K}", N, K, group, had, 1, outl)
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, had)
    y1 = gc.gemv(d, packed, a, sx, workspace).cpu().numpy()
    y2 = gc.gemv(d, packed, a, sx, workspace).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "not deterministic"
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(y1[None, :], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES)
@pytest.mark.parametrize("x_dtype", [0, 1])
def test_gemv_fused(torch_cuda, orc, N, K, group, had, outl, x_dtype):
    """One-kernel prepass + CQ4 GEMV: codes and scales bit-exact, y within
    tolerance, deterministic, and unchanged by relabelling the codebook."""
    import torch
    q = gc.lib()
    idx, sw, C, cb, x = gc.cq4_case(12, f"cq4/fused/{N}/{K}", N, K, group, had, 1, outl)
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    xt = torch.from_numpy(x)
    if x_dtype == 1:
        xt = xt.to(torch.float16)
    xval = xt.float().numpy()
    dev = gc.dev()
    y = gc.guarded((N,), torch.float32, float("nan"))
    a = gc.guarded(K, torch.int8)
    sx = gc.guarded(K // group, torch.float32)
    q.qmm_gemv_fused(d, packed, xt.to(dev), x_dtype, had, y, a, sx)
    assert q.qmm_last_kernel_id() == 7
    ra, rsx, _ = orc.prep_w4a8(xval, group, had)
    assert np.array_equal(a.cpu().numpy(), ra[0])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx[0].view(np.uint32))
    Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, group)
    y1 = y.cpu().numpy()
    ok, worst = gc.within_w4a8(y1[None, :], Y, Ym)
    assert ok, f"worst error / bound = {worst}"
    q.qmm_gemv_fused(d, packed, xt.to(dev), x_dtype, had, y)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y1.view(np.uint32)), "not deterministic"
    idx2, C2 = _relabel(idx, C)
    d2, packed2 = gc.pack_cq4(N, K, group, idx2, C2, cb, sw)
    q.qmm_gemv_fused(d2, packed2, xt.to(dev), x_dtype, had, y)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y1.view(np.uint32)), "relabelling changed y"


@pytest.mark.parametrize("Ns,K,group,had", [((2048, 512, 512), 1536, 64, 64), ((200, 100, 384), 512, 64, 0),
                                            ((256, 130), 1024, 128, 128)])
def test_gemv_fused_siblings(torch_cuda, orc, Ns, K, group, had):
    """CQ4 siblings, each with its own codebook and cb_scale, in one launch."""
    import torch
    q = gc.lib()
    dev = gc.dev()
    x = None
    descs, packs, ys, refs = [], [], [], []
    for i, N in enumerate(Ns):
        idx, sw, C, cb, xi = gc.cq4_case(30 + i, f"cq4/siblings/{i}/{N}/{K}", N, K, group, had, 1)
        x = xi if x is None else x
        d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
        descs.append(d)
        packs.append(packed)
        ys.append(gc.guarded((N,), torch.float32, float("nan")))
        refs.append((idx, sw, C, cb))
    xt = gc.t(x[0].astype(np.float32))
    q.qmm_gemv_fused_siblings(descs, packs, xt, 0, had, ys)
    assert q.qmm_last_kernel_id() == 9
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    for (idx, sw, C, cb), y in zip(refs, ys):
        Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, group)
        ok, worst = gc.within_w4a8(y.cpu().numpy()[None, :], Y, Ym)
        assert ok, f"worst error / bound = {worst}"


# ------------------------------------------------------------------ GEMM

GEMM_CASES = [
    (16, 256, 512, 64, 64),
    (17, 200, 192, 64, 0),       # ragged rows and columns
    (65, 384, 1024, 64, 64),
    (130, 128, 256, 128, 128),
    (240, 256, 512, 64, 64),     # two activation tiles
]


@pytest.mark.parametrize("book", ["seeded", "extreme"])
@pytest.mark.parametrize("M,N,K,group,had", GEMM_CASES)
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_gemm_partials_bit_exact(torch_cuda, orc, M, N, K, group, had, operand_in_smem, book):
    q = gc.lib()
    idx, sw, C, cb, x = gc.cq4_case(8, f"cq4/gemm/{M}/{N}/{K}", N, K, group, had, M)
    if book == "extreme":
        C = _extreme_book()
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    _, a16, _, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_weight_operand(operand_in_smem)
    try:
        P = gc.partials(d, packed, M, GEMM, a16)
        assert q.qmm_last_kernel_id() == 11
    finally:
        q.qmm_set_gemm_weight_operand(False)
    ra, _, _ = orc.prep_w4a8(x, group, had)
    assert np.array_equal(P.cpu().numpy(), orc.partials_cq4(idx, C, ra, group))


@pytest.mark.parametrize("M,N,K,group,had", GEMM_CASES + [(1, 256, 256, 64, 64), (4, 300, 1536, 128, 128),
                                                          (8, 1024, 1536, 64, 64), (32, 512, 1536, 128, 128)])
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_gemm_output(torch_cuda, orc, M, N, K, group, had, operand_in_smem):
    """Tensor-core kernel for every M (small-M kernel off), and the small-M
    kernel where it applies; both within tolerance of the oracle."""
    q = gc.lib()
    idx, sw, C, cb, x = gc.cq4_case(9, f"cq4/gemm/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, group)
    q.qmm_set_gemm_weight_operand(operand_in_smem)
    q.qmm_set_gemm_rows_max(0)
    q.qmm_set_gemm_narrow(q.NARROW_OFF)
    try:
        Yg = gc.gemm(d, packed, M, a16, sx, kernel=11).cpu().numpy()
    finally:
        q.qmm_set_gemm_weight_operand(False)
        q.qmm_set_gemm_rows_max(8)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    ok, worst = gc.within_w4a8(Yg, Y, Ym)
    assert ok, f"tensor-core kernel: worst error / bound = {worst}"
    if M <= 32 and not operand_in_smem:
        # the weights-in-N tensor-core kernel (not chosen by default for
        # codebook weights): the same bits
        q.qmm_set_gemm_rows_max(0)
        q.qmm_set_gemm_narrow(q.NARROW_ALWAYS)
        try:
            Yn = gc.gemm(d, packed, M, a16, sx, kernel=13).cpu().numpy()
        finally:
            q.qmm_set_gemm_rows_max(8)
            q.qmm_set_gemm_narrow(q.NARROW_AUTO)
        assert np.array_equal(Yn.view(np.uint32), Yg.view(np.uint32)), "weights-in-N kernel differs"
    if M <= 16 and not operand_in_smem:
        q.qmm_set_gemm_rows_max(16)
        try:
            Yr = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
            Yr2 = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
        finally:
            q.qmm_set_gemm_rows_max(8)
        ok, worst = gc.within_w4a8(Yr, Y, Ym)
        assert ok, f"small-M kernel: worst error / bound = {worst}"
        assert np.array_equal(Yr.view(np.uint32), Yr2.view(np.uint32)), "not deterministic"


@pytest.mark.parametrize("M", [9, 32])
def test_gemm_many_tiles(torch_cuda, orc, M):
    """Narrow tiles over 305 row tiles (several per persistent block)."""
    test_gemm_output(torch_cuda, orc, M, 305 * 128 - 72, 256, 64, 64, False)


@pytest.mark.parametrize("M,K,group", [(4, 384, 128), (16, 256, 64)])
def test_gemm_rows_stream(torch_cuda, orc, M, K, group):
    """640 row tiles: the small-M kernel's streaming form (and the tensor cores)."""
    test_gemm_output(torch_cuda, orc, M, 640 * 128 - 40, K, group, group, False)


def _sample_rows(N, n=48):
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], np.linspace(0, N - 1, n).astype(np.int64)]))
    return rows.astype(np.int32)


@pytest.mark.parametrize("M", [1, 4, 128, 1068])
def test_gemm_prefill_full_size_sampled(torch_cuda, orc, M):
    """The prefill projection K = 1536, N = 12288 with CQ4 weights, at the
    launch configuration the benchmark uses; the oracle checks sampled rows."""
    N, K, group, had = 12288, 1536, 64, 64
    idx, sw, C, cb, x = gc.cq4_case(0, "cq4/prefill", N, K, group, had, M)
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    Yg = gc.gemm(d, packed, M, a16, sx).cpu().numpy()
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    rows = _sample_rows(N)
    Y, Ym = orc.gemm_cq4(idx, C, cb, sw, ra, rsx, group, rows=rows)
    ok, worst = gc.within_w4a8(Yg[:, rows], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


def test_relabelled_codebook_gives_identical_gemm(torch_cuda):
    """Permuting the levels and renaming the indices with them leaves every
    output bit unchanged (the partials are the same integers)."""
    M, N, K, group, had = 64, 384, 1024, 64, 64
    idx, sw, C, cb, x = gc.cq4_case(3, "cq4/relabel", N, K, group, had, M)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    d, packed = gc.pack_cq4(N, K, group, idx, C, cb, sw)
    idx2, C2 = _relabel(idx, C)
    d2, packed2 = gc.pack_cq4(N, K, group, idx2, C2, cb, sw)
    Y1 = gc.gemm(d, packed, M, a16, sx).cpu().numpy()
    Y2 = gc.gemm(d2, packed2, M, a16, sx).cpu().numpy()
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
