"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Bit-exact: packed bytes, int8 codes (and their fp16 image), activation
scales, group sums of the affine prepass, int32 group partials.
Tolerance: W4A8 fp32 outputs |d| <= 1e-5 * sum_g |sw sx P| + 1e-6;
affine outputs |d| <= 2e-3 * sum_k |w x|.
"""

import numpy as np
import pytest

import qmm_synth
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

W4A8, AFFINE = 0, 1
GEMV, GEMM = 0, 1


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


# ------------------------------------------------------------------ pack

PACK_CASES = [
    (W4A8, 1024, 1024, 64),
    (W4A8, 200, 192, 64),      # ragged last row tile
    (W4A8, 130, 512, 128),
    (W4A8, 1, 64, 64),         # one row, one group
    (AFFINE, 129, 256, 64),
    (W4A8, 12288, 1536, 64),   # gate_up
    (W4A8, 1536, 6144, 64),    # down
]


@pytest.mark.parametrize("variant,N,K,group", PACK_CASES)
def test_pack_bytes(torch_cuda, orc, variant, N, K, group):
    lay = qmm_synth.Layer("p", variant, N, K, group, 0)
    qb, s, b = qmm_synth.layer_weights(1, f"pack/{variant}/{N}/{K}/{group}", lay)
    _, packed = gc.pack(variant, N, K, group, qb, s, b)
    ref = orc.pack(variant, N, K, group, qb, s, b)
    assert np.array_equal(packed.cpu().numpy(), ref)


@pytest.mark.parametrize("variant,N,K,group", [(W4A8, 262144, 1536, 128), (AFFINE, 34816, 5120, 64)])
def test_pack_bytes_full_size_sampled(torch_cuda, orc, variant, N, K, group):
    """Full-size weights: the oracle packs row tiles 0, 1, a middle one and the
    last; the GPU blob's chunks of those tiles must match byte for byte."""
    lay = qmm_synth.Layer("p", variant, N, K, group, 0)
    qb, s, b = qmm_synth.layer_weights(0, "full/pack", lay)
    _, packed = gc.pack(variant, N, K, group, qb, s, b)
    blob = packed.cpu().numpy()
    G = K // group
    CB = 64 * group + 256 + (256 if variant == AFFINE else 0)
    T = (N + 127) // 128
    for t0 in (0, 1, T // 2, T - 1):
        rows = slice(128 * t0, min(N, 128 * (t0 + 1)))
        ref = orc.pack(variant, rows.stop - rows.start, K, group, qb[rows], s[rows],
                       None if b is None else b[rows])
        assert np.array_equal(blob[t0 * G * CB:(t0 + 1) * G * CB], ref), t0


def test_pack_control_nibble_order_is_detected(torch_cuda, orc):
    """Control: a blob built with the nibble halves swapped differs from the
    GPU's (the byte comparison is sensitive to the order)."""
    N, K, g = 256, 256, 64
    lay = qmm_synth.Layer("p", W4A8, N, K, g, 0)
    qb, s, _ = qmm_synth.layer_weights(2, "pack/control", lay)
    _, packed = gc.pack(W4A8, N, K, g, qb, s)
    swapped = ((qb & 0xF) << 4) | (qb >> 4)
    assert not np.array_equal(packed.cpu().numpy(), orc.pack(W4A8, N, K, g, swapped, s))


# ------------------------------------------------------------------ W4A8 prep

PREP_CASES = [
    (1, 1536, 64, 64, 0.01),
    (7, 256, 64, 0, 0.0),
    (5, 512, 128, 128, 0.01),
    (65, 1536, 64, 64, 0.0),
    (1068, 1536, 64, 64, 0.0),
    (32, 1536, 128, 128, 0.0),
]


def _prep_input(x, x_dtype):
    """(device-side input tensor on CPU, float32 values the oracle sees)."""
    import torch
    xt = torch.from_numpy(x)
    if x_dtype == 1:
        xt = xt.to(torch.float16)
    elif x_dtype == 2:
        xt = xt.to(torch.bfloat16)
    return xt, xt.float().numpy()


@pytest.mark.parametrize("M,K,group,had,outl", PREP_CASES)
@pytest.mark.parametrize("x_dtype", [0, 1, 2])
def test_prep_w4a8_bit_exact(torch_cuda, orc, M, K, group, had, outl, x_dtype):
    if x_dtype and M > 65:
        pytest.skip("dtype variants on the small shapes only")
    x = qmm_synth.activations_f32(3, f"prep/{M}/{K}", M, K, outlier_frac=outl)
    x[0, :group] = 0.0     # an all-zero group
    xin, xval = _prep_input(x, x_dtype)
    q = gc.lib()
    G = K // group
    dev = gc.dev()
    xt = xin.to(dev)
    a = torch_cuda.empty((M, K), dtype=torch_cuda.int8, device=dev)
    a16 = torch_cuda.empty((M, K), dtype=torch_cuda.float16, device=dev)
    sx = torch_cuda.empty((M, G), dtype=torch_cuda.float32, device=dev)
    asum = torch_cuda.empty((M, G), dtype=torch_cuda.int32, device=dev)
    q.qmm_prep_act(W4A8, M, K, group, had, xt, x_dtype, a=a, a16=a16, sx=sx, asum=asum)
    ra, rsx, rsum = orc.prep_w4a8(xval, group, had)
    assert np.array_equal(a.cpu().numpy(), ra)
    assert np.array_equal(a16.cpu().numpy(), ra.astype(np.float16))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx.view(np.uint32))
    assert np.array_equal(asum.cpu().numpy(), rsum)


def test_prep_control_rotation_is_detected(torch_cuda, orc):
    """Control: codes of the rotated prepass differ from unrotated ones."""
    x = qmm_synth.activations_f32(4, "prep/control", 4, 512)
    a, _, _, _, _ = gc.prep_w4a8(x, 64, 64)
    ra, _, _ = orc.prep_w4a8(x, 64, 0)
    assert not np.array_equal(a.cpu().numpy(), ra)


# ------------------------------------------------------------------ affine prep

@pytest.mark.parametrize("M,K,x_dtype", [(1, 64, 1), (65, 5120, 1), (3, 640, 0), (9, 192, 2), (128, 5120, 1)])
def test_prep_affine_group_sums_bit_exact(torch_cuda, orc, M, K, x_dtype):
    import torch
    q = gc.lib()
    dev = gc.dev()
    x = qmm_synth.normal(5, f"aff/{M}/{K}", M * K).astype(np.float32).reshape(M, K)
    xin, xval = _prep_input(x, x_dtype)
    G = K // 64
    S = gc.guarded((M, G), torch.float32)
    x16 = gc.guarded((M, K), torch.float16) if x_dtype != 1 else None
    q.qmm_prep_act(AFFINE, M, K, 64, 0, xin.to(dev), x_dtype, gsum=S, x16=x16)
    assert q.qmm_last_kernel_id() == 3
    ref = orc.group_sums_affine(xval)
    assert np.array_equal(S.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    if x16 is not None:
        assert np.array_equal(x16.cpu().numpy().view(np.uint16), xval.astype(np.float16).view(np.uint16))


def test_prep_affine_tree_fixture(torch_cuda):
    """The page's summation tree on the GPU, on the hand-worked fixture."""
    import torch
    from tests import oracle_pins
    q = gc.lib()
    cases = oracle_pins.read_cases("group_sum_tree.txt")
    x = np.array([c["chunk"] for c in cases], dtype=np.float32).reshape(len(cases), 64)
    S = gc.guarded((len(cases), 1), torch.float32)
    q.qmm_prep_act(AFFINE, len(cases), 64, 64, 0, torch.from_numpy(x).to(gc.dev()), 0, gsum=S)
    expect = np.array([float(c["expect"]) for c in cases], dtype=np.float32)
    assert np.array_equal(S.cpu().numpy()[:, 0], expect)


# ------------------------------------------------------------------ GEMV

GEMV_CASES = [
    (1024, 1024, 64, 0, 0.0),     # the K = N = 1024 GEMV
    (200, 192, 64, 64, 0.0),      # ragged rows
    (256, 512, 128, 128, 0.0),
    (128, 64, 64, 0, 0.0),        # one group
    (12288, 1536, 64, 64, 0.01),  # gate_up
    (1536, 6144, 64, 64, 0.01),   # down
    (2048, 1536, 64, 64, 0.01),   # q
    (1536, 2048, 64, 64, 0.01),   # o
]


@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES)
def test_gemv_partials_bit_exact(torch_cuda, orc, N, K, group, had, outl):
    qb, sw, x = gc.w4a8_case(6, f"gemv/{N}/{K}", N, K, group, had, 1, outl)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, had)
    P = gc.partials(d, packed, 1, GEMV, a)
    ra, _, _ = orc.prep_w4a8(x, group, had)
    assert np.array_equal(P.cpu().numpy(), orc.partials_w4a8(qb, ra, group))


@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES)
@pytest.mark.parametrize("workspace", [True, False])
def test_gemv_output(torch_cuda, orc, N, K, group, had, outl, workspace):
    qb, sw, x = gc.w4a8_case(7, f"gemv/{N}/{K}", N, K, group, had, 1, outl)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    a, _, sx, _, _ = gc.prep_w4a8(x, group, had)
    y1 = gc.gemv(d, packed, a, sx, workspace).cpu().numpy()
    y2 = gc.gemv(d, packed, a, sx, workspace).cpu().numpy()
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), "not deterministic"
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(y1[None, :], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


@pytest.mark.parametrize("N,K,group,had,outl", GEMV_CASES + [(256, 512, 128, 0, 0.0)])
@pytest.mark.parametrize("x_dtype", [0, 1])
def test_gemv_fused(torch_cuda, orc, N, K, group, had, outl, x_dtype):
    """One-kernel prepass + GEMV: codes and scales bit-exact, y within tolerance."""
    import torch
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(12, f"fused/{N}/{K}", N, K, group, had, 1, outl)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    xin, xval = _prep_input(x, x_dtype)
    dev = gc.dev()
    y = gc.guarded((N,), torch.float32, float("nan"))
    a = gc.guarded(K, torch.int8)
    sx = gc.guarded(K // group, torch.float32)
    q.qmm_gemv_fused(d, packed, xin.to(dev), x_dtype, had, y, a, sx)
    assert q.qmm_last_kernel_id() == 7
    ra, rsx, _ = orc.prep_w4a8(xval, group, had)
    assert np.array_equal(a.cpu().numpy(), ra[0])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx[0].view(np.uint32))
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    y1 = y.cpu().numpy()
    ok, worst = gc.within_w4a8(y1[None, :], Y, Ym)
    assert ok, f"worst error / bound = {worst}"
    q.qmm_gemv_fused(d, packed, xin.to(dev), x_dtype, had, y)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y1.view(np.uint32)), "not deterministic"


SIBLING_CASES = [
    ((2048, 512, 512), 1536, 64, 64),     # q | k | v
    ((6144, 6144), 1536, 64, 64),         # gate | up
    ((200, 100, 384), 512, 64, 0),        # ragged tiles, no rotation
    ((256, 130), 1024, 128, 128),
]


@pytest.mark.parametrize("Ns,K,group,had", SIBLING_CASES)
def test_gemv_fused_siblings(torch_cuda, orc, Ns, K, group, had):
    """Sibling matrices in one launch: shared codes/scales bit-exact, every
    output within tolerance of the oracle, deterministic."""
    import torch
    q = gc.lib()
    dev = gc.dev()
    x = None
    descs, packs, ys, refs = [], [], [], []
    for i, N in enumerate(Ns):
        qb, sw, xi = gc.w4a8_case(20 + i, f"siblings/{i}/{N}/{K}", N, K, group, had, 1)
        x = xi if x is None else x
        d, packed = gc.pack(W4A8, N, K, group, qb, sw)
        descs.append(d)
        packs.append(packed)
        ys.append(gc.guarded((N,), torch.float32, float("nan")))
        refs.append((qb, sw))
    a = gc.guarded(K, torch.int8)
    sx = gc.guarded(K // group, torch.float32)
    xt = gc.t(x[0].astype(np.float32))
    q.qmm_gemv_fused_siblings(descs, packs, xt, 0, had, ys, a, sx)
    assert q.qmm_last_kernel_id() == 9
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    assert np.array_equal(a.cpu().numpy(), ra[0])
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rsx[0].view(np.uint32))
    first = [y.cpu().numpy().copy() for y in ys]
    for (qb, sw), y in zip(refs, first):
        Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
        ok, worst = gc.within_w4a8(y[None, :], Y, Ym)
        assert ok, f"worst error / bound = {worst}"
    q.qmm_gemv_fused_siblings(descs, packs, xt, 0, had, ys)
    for y0, y in zip(first, ys):
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y0.view(np.uint32)), "not deterministic"


def test_pack_then_consume_same_stream(torch_cuda, orc):
    """A blob packed on the stream is complete before the next kernel reads it:
    the consumers stream weights before their dependency wait, so the pack must
    not let them start early. Each consumer runs right after packing into a
    buffer full of stale bytes, with nothing in between."""
    import torch
    q = gc.lib()
    N, K, g = 32768, 1536, 64
    qb, sw, x = gc.w4a8_case(14, "pack_then_consume", N, K, g, g, 64)
    d = q.weight_desc(W4A8, N, K, g)
    size = q.qmm_packed_size(d)
    _, a16, sx, _, _ = gc.prep_w4a8(x, g, g)
    xt = gc.t(x.astype(np.float32))
    qt, st = gc.t(qb), gc.t(sw)
    ra, rsx, _ = orc.prep_w4a8(x, g, g)
    rows = _sample_rows(N)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, g, rows=rows)
    torch.cuda.synchronize()

    def fresh():
        return gc.guarded((size,), torch.uint8, 0xFF)

    # fused GEMV (row 0 of x)
    blob = fresh()
    y = gc.guarded((N,), torch.float32, float("nan"))
    q.qmm_pack_weights(d, qt, st, None, blob)
    q.qmm_gemv_fused(d, blob, xt[0], 0, g, y)
    ok, worst = gc.within_w4a8(y.cpu().numpy()[None, rows], Y[:1], Ym[:1])
    assert ok, f"fused GEMV: worst error / bound = {worst}"
    # GEMM on the CUDA cores (M = 2) and on the tensor cores (M = 64)
    for M, kernel in ((2, 8), (64, 5)):
        blob = fresh()
        Yg = gc.guarded((M, N), torch.float32, float("nan"))
        q.qmm_pack_weights(d, qt, st, None, blob)
        q.qmm_gemm(d, blob, M, a16[:M], sx[:M], Yg)
        assert q.qmm_last_kernel_id() == kernel
        ok, worst = gc.within_w4a8(Yg.cpu().numpy()[:, rows], Y[:M], Ym[:M])
        assert ok, f"GEMM M={M}: worst error / bound = {worst}"


# ------------------------------------------------------------------ GEMM

GEMM_CASES = [
    (1, 256, 256, 64, 64),
    (16, 256, 512, 64, 64),
    (17, 200, 192, 64, 0),       # ragged rows and columns
    (65, 384, 1024, 64, 64),
    (130, 128, 256, 128, 128),
    (240, 256, 512, 64, 64),     # two activation tiles
    (32, 512, 1536, 128, 128),
]


@pytest.mark.parametrize("M,N,K,group,had", GEMM_CASES)
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_gemm_partials_bit_exact(torch_cuda, orc, M, N, K, group, had, operand_in_smem):
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(8, f"gemm/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_weight_operand(operand_in_smem)
    try:
        P = gc.partials(d, packed, M, GEMM, a16)
    finally:
        q.qmm_set_gemm_weight_operand(False)
    ra, _, _ = orc.prep_w4a8(x, group, had)
    assert np.array_equal(P.cpu().numpy(), orc.partials_w4a8(qb, ra, group))


@pytest.mark.parametrize("M,N,K,group,had", GEMM_CASES)
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_gemm_output(torch_cuda, orc, M, N, K, group, had, operand_in_smem):
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(9, f"gemm/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_weight_operand(operand_in_smem)
    q.qmm_set_gemm_narrow(q.NARROW_OFF)   # the general tensor-core kernel (or the small-M one)
    try:
        Yg = gc.gemm(d, packed, M, a16, sx).cpu().numpy()
    finally:
        q.qmm_set_gemm_weight_operand(False)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(Yg, Y, Ym)
    assert ok, f"worst error / bound = {worst}"


# Narrow tiles (at most 32 activation rows) over 305 row tiles, the last one
# ragged: every persistent block runs two or three tiles; every output compared.
WIDE_N = 305 * 128 - 72


@pytest.mark.parametrize("M", [9, 17, 32])
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_gemm_many_tiles(torch_cuda, orc, M, operand_in_smem):
    test_gemm_output(torch_cuda, orc, M, WIDE_N, 256, 64, 64, operand_in_smem)


# M <= 32 above the small-M limit: the tensor-core kernel with the weights in
# the MMA's N slot (256 weight rows per MMA, activations loaded into all four
# lane quadrants). Against the oracle (every output), bit for bit against the
# general tensor-core kernel (same operations in the same order), and a repeat.
# Odd tile counts leave the last pair half empty; 640 tiles run several pairs
# per persistent block.
NARROW_CASES = [
    (1, 200, 256, 64, 64),
    (9, 384, 512, 64, 64),          # 3 tiles: one full pair, one half
    (16, 256, 1536, 128, 128),
    (17, 640 * 128 - 40, 256, 64, 64),
    (32, 1000, 384, 128, 128),
    (32, 130, 1536, 64, 0),
    (12, 640 * 128 - 41, 256, 64, 64),   # N % 4 != 0: scalar stores
]


@pytest.mark.parametrize("M,N,K,group,had", NARROW_CASES)
def test_gemm_narrow_output(torch_cuda, orc, M, N, K, group, had):
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(16, f"narrow/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_rows_max(0)
    q.qmm_set_gemm_narrow(q.NARROW_F16)
    try:
        Yn = gc.gemm(d, packed, M, a16, sx, kernel=13).cpu().numpy()
        Yn2 = gc.gemm(d, packed, M, a16, sx, kernel=13).cpu().numpy()
        q.qmm_set_gemm_narrow(q.NARROW_OFF)
        Yt = gc.gemm(d, packed, M, a16, sx, kernel=5).cpu().numpy()
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    assert np.array_equal(Yn.view(np.uint32), Yn2.view(np.uint32)), "not deterministic"
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(Yn, Y, Ym)
    assert ok, f"worst error / bound = {worst}"
    assert np.array_equal(Yn.view(np.uint32), Yt.view(np.uint32)), "differs from the general tensor-core kernel"


# M <= 16, group 128: the e4m3 form of the weights-in-N kernel (kind::f8f6f4
# MMAs on the nibbles u = q + 8 and the two planes of each activation code).
# Every output against the oracle; bit for bit against the fp16 form and the
# general tensor-core kernel (the partials are the same exact integers and the
# rescale is the same operations); a repeat. Ragged and odd tile counts, N % 4
# != 0 (scalar stores), rows M..15 unused, no rotation, K of 12 and 14 groups
# (the longest it holds) and one group.
E4M3_CASES = [
    (1, 200, 256, 128, 128),
    (9, 384, 512, 128, 128),            # 3 tiles: one full pair, one half
    (16, 256, 1536, 128, 128),
    (16, 640 * 128 - 40, 256, 128, 0),  # 320 pairs over the persistent blocks
    (12, 640 * 128 - 41, 256, 128, 128),
    (5, 1000, 384, 128, 128),
    (16, 300, 1792, 128, 128),
    (3, 130, 128, 128, 128),
]


@pytest.mark.parametrize("M,N,K,group,had", E4M3_CASES)
def test_gemm_narrow_e4m3_output(torch_cuda, orc, M, N, K, group, had):
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(17, f"narrow_e4m3/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_rows_max(0)
    q.qmm_set_gemm_narrow(q.NARROW_ALWAYS)
    try:
        Ye = gc.gemm(d, packed, M, a16, sx, kernel=14).cpu().numpy()
        Ye2 = gc.gemm(d, packed, M, a16, sx, kernel=14).cpu().numpy()
        q.qmm_set_gemm_narrow(q.NARROW_F16)
        Yn = gc.gemm(d, packed, M, a16, sx, kernel=13).cpu().numpy()
        q.qmm_set_gemm_narrow(q.NARROW_OFF)
        Yt = gc.gemm(d, packed, M, a16, sx, kernel=5).cpu().numpy()
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    assert np.array_equal(Ye.view(np.uint32), Ye2.view(np.uint32)), "not deterministic"
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(Ye, Y, Ym)
    assert ok, f"worst error / bound = {worst}"
    assert np.array_equal(Ye.view(np.uint32), Yn.view(np.uint32)), "differs from the fp16 form"
    assert np.array_equal(Ye.view(np.uint32), Yt.view(np.uint32)), "differs from the general tensor-core kernel"


def test_gemm_narrow_e4m3_falls_back_on_long_k(torch_cuda, orc):
    """K = 1920 (15 groups of 128) leaves the e4m3 form's shared memory too
    small for its activation planes: the call runs the fp16 form (kernel 13)
    and is still right."""
    q = gc.lib()
    M, N, K, g = 16, 640 * 128, 1920, 128
    qb, sw, x = gc.w4a8_case(18, "narrow_e4m3/long_k", N, K, g, g, M)
    d, packed = gc.pack(W4A8, N, K, g, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, g, g)
    q.qmm_set_gemm_rows_max(0)
    try:
        Yg = gc.gemm(d, packed, M, a16, sx, kernel=13).cpu().numpy()   # NARROW_AUTO, 640 row tiles
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
    ra, rsx, _ = orc.prep_w4a8(x, g, g)
    rows = _sample_rows(N)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, g, rows=rows)
    ok, worst = gc.within_w4a8(Yg[:, rows], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


def test_gemm_narrow_e4m3_extreme_codes(torch_cuda):
    """Codes at the ends of both ranges: weights q = -8 and 7 (u = 0 and 15),
    activation codes -127, 127, -1, 0, 1, 15, 16, -16, -17 (every hi/lo split
    edge); bit for bit against the general tensor-core kernel."""
    import torch
    q = gc.lib()
    N, K, g, M = 512, 256, 128, 16
    rng = np.random.default_rng(5)
    qv = rng.choice(np.array([-8, 7, 0, -1, 1], np.int8), size=(N, K))
    nib = (qv & 15).astype(np.uint8)
    qbytes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)   # low nibble = even k
    sw = rng.uniform(0.005, 0.02, size=(N, K // g)).astype(np.float16)
    d, packed = gc.pack(W4A8, N, K, g, qbytes, sw.view(np.uint16))
    codes = rng.choice(np.array([-127, 127, -1, 0, 1, 15, 16, -16, -17], np.float16), size=(M, K))
    a16 = gc.t(codes)
    sx = gc.t(rng.uniform(0.5, 2.0, size=(M, K // g)).astype(np.float32))
    q.qmm_set_gemm_narrow(q.NARROW_ALWAYS)
    q.qmm_set_gemm_rows_max(0)
    try:
        Ye = gc.gemm(d, packed, M, a16, sx, kernel=14).cpu().numpy()
        q.qmm_set_gemm_narrow(q.NARROW_OFF)
        Yt = gc.gemm(d, packed, M, a16, sx, kernel=5).cpu().numpy()
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    assert np.array_equal(Ye.view(np.uint32), Yt.view(np.uint32))
    # and against the definition: sum_g sw sx sum_k q a, in fp64
    P = np.einsum("mgk,ngk->mng", codes.astype(np.float64).reshape(M, K // g, g),
                  qv.astype(np.float64).reshape(N, K // g, g))
    ref = np.einsum("mng,ng,mg->mn", P, sw.astype(np.float64), sx.cpu().numpy().astype(np.float64))
    bound = 1e-5 * np.einsum("mng,ng,mg->mn", np.abs(P), sw.astype(np.float64), sx.cpu().numpy().astype(np.float64)) + 1e-6
    assert np.all(np.abs(Ye - ref) <= bound)


def _sample_rows(N, n=48):
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], np.linspace(0, N - 1, n).astype(np.int64)]))
    return rows.astype(np.int32)


@pytest.mark.parametrize("M", [16, 64, 128, 512, 1068])
def test_gemm_prefill_full_size_sampled(torch_cuda, orc, M):
    """K=1536, N=12288, group 64, Hadamard-64: every row m on sampled columns n."""
    N, K, g = 12288, 1536, 64
    qb, sw, x = gc.w4a8_case(0, "prefill_gemm", N, K, g, g, M)
    d, packed = gc.pack(W4A8, N, K, g, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, g, g)
    Yg = gc.gemm(d, packed, M, a16, sx).cpu().numpy()
    assert not np.isnan(Yg).any()
    ra, rsx, _ = orc.prep_w4a8(x, g, g)
    rows = _sample_rows(N)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, g, rows=rows)
    ok, worst = gc.within_w4a8(Yg[:, rows], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


@pytest.fixture(scope="module")
def lm_head(torch_cuda):
    N, K, g = 262144, 1536, 128
    lay = qmm_synth.Layer("lm_head", W4A8, N, K, g, g)
    qb, sw, _ = qmm_synth.layer_weights(0, "lm_head", lay)
    d, packed = gc.pack(W4A8, N, K, g, qb, sw)
    return lay, qb, sw, d, packed


@pytest.mark.parametrize("M", [1, 2, 4, 8, 12, 16, 32])
def test_lm_head_full_size_sampled(lm_head, orc, M):
    lay, qb, sw, d, packed = lm_head
    g = lay.group
    x = qmm_synth.layer_activations(0, f"lm_head/x{M}", lay, M)
    a, a16, sx, _, _ = gc.prep_w4a8(x, g, g)
    Yg = gc.gemm(d, packed, M, a16, sx, kernel=8 if M <= 8 else (14 if M <= 16 else 13)).cpu().numpy()
    ra, rsx, _ = orc.prep_w4a8(x, g, g)
    rows = _sample_rows(lay.N)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, g, rows=rows)
    ok, worst = gc.within_w4a8(Yg[:, rows], Y, Ym)
    assert ok, f"GEMM worst error / bound = {worst}"
    # the same call on the other kernels that serve this M
    q = gc.lib()
    on, off, f16 = q.NARROW_AUTO, q.NARROW_OFF, q.NARROW_F16
    others = [(0, on, 14), (0, f16, 13), (0, off, 5)] if M <= 8 else \
        [(0, off, 5)] + ([(16, on, 8), (0, f16, 13)] if M <= 16 else [])
    for rows_max, narrow, kernel in others:
        q.qmm_set_gemm_rows_max(rows_max)
        q.qmm_set_gemm_narrow(narrow)
        try:
            Yt = gc.gemm(d, packed, M, a16, sx, kernel=kernel).cpu().numpy()
        finally:
            q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
            q.qmm_set_gemm_narrow(q.NARROW_AUTO)
        ok, worst = gc.within_w4a8(Yt[:, rows], Y, Ym)
        assert ok, f"kernel {kernel}: worst error / bound = {worst}"
    if M == 1:
        y = gc.gemv(d, packed, a, sx).cpu().numpy()
        ok, worst = gc.within_w4a8(y[None, rows], Y, Ym)
        assert ok, f"GEMV worst error / bound = {worst}"


# ------------------------------------------------------------------ small-M GEMM (CUDA cores)

ROWS_DEFAULT = 8   # qmm_set_gemm_rows_max's default

ROWS_CASES = [
    (1, 256, 256, 64, 64),
    (2, 200, 192, 64, 0),        # ragged columns, odd group count
    (3, 384, 1024, 64, 64),
    (5, 128, 512, 128, 128),
    (8, 256, 1536, 128, 128),
    (9, 130, 640, 64, 64),
    (16, 512, 1536, 64, 64),
]


@pytest.mark.parametrize("M,N,K,group,had", ROWS_CASES)
def test_gemm_rows_output(torch_cuda, orc, M, N, K, group, had):
    """M <= 16 W4A8 runs on the dp4a kernel: every output against the oracle,
    the same call on the tensor cores, and a repeat (deterministic)."""
    q = gc.lib()
    qb, sw, x = gc.w4a8_case(11, f"rows/{M}/{N}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_rows_max(16)
    try:
        Yr = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
        Yr2 = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
        assert np.array_equal(Yr, Yr2)
        q.qmm_set_gemm_rows_max(0)
        q.qmm_set_gemm_narrow(q.NARROW_OFF)
        Yt = gc.gemm(d, packed, M, a16, sx, kernel=5).cpu().numpy()
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    for name, Yg in (("dp4a", Yr), ("tensor", Yt)):
        ok, worst = gc.within_w4a8(Yg, Y, Ym)
        assert ok, f"{name}: worst error / bound = {worst}"


# At least 512 row tiles run the dp4a kernel's streaming form: resident blocks
# over successive tiles, all of K per block, one ring of stages per half of the
# groups. 640 tiles, the last one ragged; odd group counts split unevenly
# between the halves; every output compared.
STREAM_N = 640 * 128 - 40
STREAM_CASES = [
    (1, 256, 64, 64),
    (3, 192, 64, 0),       # 3 groups: halves of 2 and 1
    (8, 384, 128, 128),    # 3 groups of 128
    (16, 256, 64, 64),
]


@pytest.mark.parametrize("M,K,group,had", STREAM_CASES)
def test_gemm_rows_stream_output(torch_cuda, orc, M, K, group, had):
    q = gc.lib()
    N = STREAM_N
    qb, sw, x = gc.w4a8_case(15, f"rows_stream/{M}/{K}", N, K, group, had, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, had)
    q.qmm_set_gemm_rows_max(16)
    try:
        Yr = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
        Yr2 = gc.gemm(d, packed, M, a16, sx, kernel=8).cpu().numpy()
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)
    assert np.array_equal(Yr.view(np.uint32), Yr2.view(np.uint32)), "not deterministic"
    ra, rsx, _ = orc.prep_w4a8(x, group, had)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(Yr, Y, Ym)
    assert ok, f"worst error / bound = {worst}"


def test_gemm_rows_limit_and_fallback(torch_cuda, orc):
    """The rows limit picks the kernel; a K too long for one cluster of the
    dp4a kernel (193 groups of 64) falls back to the tensor cores: not to the
    weights-in-N kernel (its shared memory holds every group's activation
    scales, which 193 groups overflow) but to the general one."""
    q = gc.lib()
    M, N, K, group = 4, 128, 193 * 64, 64
    qb, sw, x = gc.w4a8_case(12, "rows/fallback", N, K, group, 0, M)
    d, packed = gc.pack(W4A8, N, K, group, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, group, 0)
    Yg = gc.gemm(d, packed, M, a16, sx, kernel=5).cpu().numpy()
    ra, rsx, _ = orc.prep_w4a8(x, group, 0)
    Y, Ym = orc.gemm_w4a8(qb, sw, ra, rsx, group)
    ok, worst = gc.within_w4a8(Yg, Y, Ym)
    assert ok, f"worst error / bound = {worst}"
    qb, sw, x = gc.w4a8_case(13, "rows/limit", 256, 512, 64, 64, 8)
    d, packed = gc.pack(W4A8, 256, 512, 64, qb, sw)
    _, a16, sx, _, _ = gc.prep_w4a8(x, 64, 64)
    gc.gemm(d, packed, ROWS_DEFAULT, a16, sx, kernel=8)     # the library default
    q.qmm_set_gemm_rows_max(4)
    try:
        gc.gemm(d, packed, 4, a16, sx, kernel=8)
        gc.gemm(d, packed, 8, a16, sx, kernel=5)
    finally:
        q.qmm_set_gemm_rows_max(ROWS_DEFAULT)


# ------------------------------------------------------------------ affine GEMM

AFF_CASES = [(1, 128, 64), (33, 256, 256), (65, 200, 320), (128, 384, 1024), (240, 128, 512)]


def _affine_run(M, N, K, seed, name, zero_sums=False):
    import torch
    q = gc.lib()
    lay = qmm_synth.Layer(name, AFFINE, N, K, 64, 0)
    qb, s, b = qmm_synth.layer_weights(seed, name, lay)
    x16 = qmm_synth.layer_activations(seed, name, lay, M)
    d, packed = gc.pack(AFFINE, N, K, 64, qb, s, b)
    xt = gc.t(x16).view(torch.float16)
    S = gc.guarded((M, K // 64), torch.float32)
    q.qmm_prep_act(AFFINE, M, K, 64, 0, xt, 1, gsum=S)
    if zero_sums:
        S.zero_()
    Yg = gc.gemm(d, packed, M, xt, S).cpu().numpy()
    return qb, s, b, x16, Yg


@pytest.mark.parametrize("M,N,K", AFF_CASES)
@pytest.mark.parametrize("operand_in_smem", [False, True])
def test_affine_gemm_output(torch_cuda, orc, M, N, K, operand_in_smem):
    q = gc.lib()
    q.qmm_set_gemm_weight_operand(operand_in_smem)
    try:
        qb, s, b, x16, Yg = _affine_run(M, N, K, 10, f"aff/{M}/{N}/{K}")
    finally:
        q.qmm_set_gemm_weight_operand(False)
    Y, Ym = orc.gemm_affine(qb, s, b, x16)
    ok, worst = gc.within_affine(Yg, Y, Ym)
    assert ok, f"worst error / bound = {worst}"


@pytest.mark.parametrize("M", [9, 32])
def test_affine_gemm_many_tiles(torch_cuda, orc, M):
    test_affine_gemm_output(torch_cuda, orc, M, WIDE_N, 128, False)


def test_affine_control_zero_sums_is_detected(torch_cuda, orc):
    """Control: leaving the prepass's group sums at zero must break the tolerance."""
    qb, s, b, x16, Yg = _affine_run(33, 256, 256, 11, "aff/control", zero_sums=True)
    Y, Ym = orc.gemm_affine(qb, s, b, x16)
    ok, _ = gc.within_affine(Yg, Y, Ym)
    assert not ok


@pytest.mark.parametrize("M", [64, 65, 128])
def test_affine_full_size_sampled(torch_cuda, orc, M):
    """K=5120, N=34816 (fused gate_up): every row m on sampled columns n."""
    N, K = 34816, 5120
    qb, s, b, x16, Yg = _affine_run(M, N, K, 0, "affine_gemm")
    rows = _sample_rows(N)
    Y, Ym = orc.gemm_affine(qb, s, b, x16, rows=rows)
    ok, worst = gc.within_affine(Yg[:, rows], Y, Ym)
    assert ok, f"worst error / bound = {worst}"


def test_device_status_clean(torch_cuda):
    assert gc.lib().qmm_device_status() == 0
