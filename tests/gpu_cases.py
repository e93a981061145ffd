"""Helpers of the GPU parity tests: run one path of the library on cuda:0 and
return numpy results, with the inputs drawn by qmm_synth."""

from __future__ import annotations

import numpy as np

import qmm_synth

W4A8, AFFINE, CQ4 = 0, 1, 2


def lib():
    import bit_group_quantized_qmm_gb300 as q
    return q


def dev():
    import torch
    return torch.device("cuda:0")


def t(a):
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


# Guard regions (the substitute for a memory checker): every output a helper
# allocates sits inside a larger buffer whose GUARD bytes before and after it
# hold a fixed pattern; after each library call the helper asserts that no
# byte of either guard changed, so a kernel writing past the end (or before
# the start) of its output fails the test that ran it.
GUARD = 256                       # bytes on each side (keeps 16-byte alignment)
_PATTERN = (0xA5, 0x3C)           # before, after


def guarded(shape, dtype, fill=None):
    """A device tensor of `shape` inside a buffer with patterned guards."""
    import torch
    shape = tuple(shape) if isinstance(shape, (tuple, list)) else (int(shape),)
    n = 1
    for d_ in shape:
        n *= int(d_)
    itemsize = torch.empty((), dtype=dtype).element_size()
    nbytes = n * itemsize
    raw = torch.empty(GUARD + nbytes + GUARD, dtype=torch.uint8, device=dev())
    raw[:GUARD].fill_(_PATTERN[0])
    raw[GUARD + nbytes:].fill_(_PATTERN[1])
    view = raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
    if fill is not None:
        view.fill_(fill)
    _live.append((raw, nbytes))
    return view


_live = []


def assert_guards_intact():
    """Every guard allocated since the last check still holds its pattern."""
    bad = []
    for raw, nbytes in _live:
        head = raw[:GUARD].cpu().numpy()
        tail = raw[GUARD + nbytes:].cpu().numpy()
        if (head != _PATTERN[0]).any() or (tail != _PATTERN[1]).any():
            bad.append((nbytes, int((head != _PATTERN[0]).sum()), int((tail != _PATTERN[1]).sum())))
    _live.clear()
    assert not bad, f"guard bytes overwritten (output bytes, bytes changed before, after): {bad}"


def pack(variant, N, K, group, q_bytes, scales, biases=None):
    import torch
    q = lib()
    d = q.weight_desc(variant, N, K, group)
    packed = guarded(q.qmm_packed_size(d), torch.uint8)
    q.qmm_pack_weights(d, t(q_bytes), t(scales), None if biases is None else t(biases), packed)
    assert q.qmm_last_kernel_id() == 1
    assert_guards_intact()
    return d, packed


def pack_cq4(N, K, group, idx_bytes, codebook, cb_scale, scales):
    import torch
    q = lib()
    d = q.weight_desc(CQ4, N, K, group)
    packed = guarded(q.qmm_packed_size(d), torch.uint8)
    q.qmm_pack_weights_cq4(d, t(idx_bytes), codebook, cb_scale, t(scales), packed)
    assert q.qmm_last_kernel_id() == 1
    assert_guards_intact()
    return d, packed


def prep_w4a8(x, group, hadamard, x_dtype=0):
    """x: float32 [M][K] numpy (converted to x_dtype on the device)."""
    import torch
    q = lib()
    M, K = x.shape
    G = K // group
    xt = t(x.astype(np.float32))
    if x_dtype == 1:
        xt = xt.to(torch.float16)
    elif x_dtype == 2:
        xt = xt.to(torch.bfloat16)
    a = guarded((M, K), torch.int8)
    a16 = guarded((M, K), torch.float16)
    sx = guarded((M, G), torch.float32)
    asum = guarded((M, G), torch.int32)
    q.qmm_prep_act(W4A8, M, K, group, hadamard, xt, x_dtype, a=a, a16=a16, sx=sx, asum=asum)
    assert q.qmm_last_kernel_id() == 2
    assert_guards_intact()
    return a, a16, sx, asum, xt


def gemv(d, packed, a, sx, workspace=True):
    import torch
    q = lib()
    y = guarded((d.N,), torch.float32, float("nan"))
    ws = None
    if workspace:
        nbytes = q.qmm_gemv_workspace_size(d)
        if nbytes:
            ws = guarded((nbytes,), torch.uint8, 0)
    q.qmm_gemv(d, packed, a, sx, y, ws)
    assert q.qmm_last_kernel_id() == (10 if d.variant == CQ4 else 4)
    assert_guards_intact()
    return y


def gemm(d, packed, M, act16, act_scale, kernel=None):
    """qmm_gemm into a NaN-filled Y; checks which kernel ran (W4A8: the
    tensor-core kernel 5, its weights-in-N form 13 (M <= 32) or 14 (e4m3,
    M <= 16, group 128), or the CUDA-core small-M kernel 8; CQ4: 11, 13 or 8;
    affine: 6)."""
    import torch
    q = lib()
    Y = guarded((M, d.N), torch.float32, float("nan"))
    q.qmm_gemm(d, packed, M, act16, act_scale, Y)
    assert_guards_intact()
    kid = q.qmm_last_kernel_id()
    if kernel is not None:
        assert kid == kernel, kid
    else:
        assert kid in {W4A8: (5, 8, 13, 14), CQ4: (11, 8, 13), AFFINE: (6,)}[d.variant], kid
    return Y


def partials(d, packed, M, path, act):
    import torch
    q = lib()
    G = d.K // d.group
    P = guarded((M, d.N, G), torch.int32, -2**31)
    q.qmm_debug_partials(d, packed, M, path, act, P)
    assert_guards_intact()
    return P


def w4a8_case(seed, name, N, K, group, hadamard, M, outlier_frac=0.0):
    lay = qmm_synth.Layer(name, W4A8, N, K, group, hadamard, outlier_frac=outlier_frac)
    qb, sw, _ = qmm_synth.layer_weights(seed, name, lay)
    x = qmm_synth.layer_activations(seed, name, lay, M)
    return qb, sw, x


def cq4_case(seed, name, N, K, group, hadamard, M, outlier_frac=0.0):
    """(index bytes, sw, codebook, cb_scale, x) of a codebook-4-bit layer."""
    lay = qmm_synth.Layer(name, CQ4, N, K, group, hadamard, outlier_frac=outlier_frac)
    idx, sw, _ = qmm_synth.layer_weights(seed, name, lay)
    C, cb = qmm_synth.layer_codebook(seed, name)
    x = qmm_synth.layer_activations(seed, name, lay, M)
    return idx, sw, C, cb, x


def within_w4a8(y, Y, Ym):
    err = np.abs(np.asarray(y, dtype=np.float64) - Y)
    bound = 1e-5 * Ym + 1e-6
    return bool(np.all(err <= bound)), float((err / bound).max())


def within_affine(y, Y, Ym):
    err = np.abs(np.asarray(y, dtype=np.float64) - Y)
    bound = 2e-3 * Ym
    return bool(np.all(err <= bound)), float((err / np.maximum(bound, 1e-300)).max())
