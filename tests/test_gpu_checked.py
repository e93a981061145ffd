"""The checked library variant on the GPU (the memory-checker substitute's
second half, beside the guard regions of tests/gpu_cases.py).

libqmm_gb300_checked.so is built from the same sources with QMM_CHECKS=1: the
kernels test their internal index ranges (weight chunks inside the blob,
tensor-memory columns inside the allocation, the epilogue's columns inside its
accumulator buffer and scale stage) and record a failure in the device error
word instead of making the access. A child process loads it
(QMM_CHECKED_LIBRARY=1) and runs a set of small calls that reach every kernel
family: pack, both prepasses, the plain and fused GEMVs (and siblings), the
tensor-core GEMM with the weight operand in tensor and in shared memory, its
weights-in-N forms (fp16 and e4m3), the CUDA-core small-M GEMM, the
raw-partials hook, the affine GEMM and codebook weights. Every call must leave the error word at
zero, and every output must equal the product library's, bit for bit (the
checks change no arithmetic).
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_cases(out_path):
    """Run the calls with whichever library the binding loaded; save the
    outputs to `out_path` (npz) and return the device error word after each."""
    import torch

    import qmm_synth
    from tests import gpu_cases as gc

    q = gc.lib()
    torch.cuda.set_device(0)
    status, outs = {}, {}

    def done(name, arr):
        torch.cuda.synchronize()
        status[name] = q.qmm_device_status()
        outs[name] = arr.cpu().numpy().copy()

    # symmetric W4A8, ragged rows and columns, rotation
    N, K, g, M = 200, 512, 64, 17
    qb, sw, x = gc.w4a8_case(91, "checked/w4a8", N, K, g, g, M)
    d, packed = gc.pack(gc.W4A8, N, K, g, qb, sw)
    done("pack", packed)
    a, a16, sx, _, _ = gc.prep_w4a8(x, g, g)
    done("prep_w4a8", a)
    y = gc.gemv(d, packed, a[0:1].reshape(-1), sx[0:1].reshape(-1), workspace=True)
    done("gemv", y)
    y = gc.guarded((N,), torch.float32, float("nan"))
    q.qmm_gemv_fused(d, packed, gc.t(x[0]), 0, g, y)
    done("gemv_fused", y)
    for smem in (False, True):
        q.qmm_set_gemm_weight_operand(smem)
        try:
            Y = gc.gemm(d, packed, M, a16, sx, kernel=5)
            done(f"gemm_{'smem' if smem else 'tmem'}", Y)
            P = gc.partials(d, packed, M, 1, a16)
            done(f"partials_{'smem' if smem else 'tmem'}", P)
        finally:
            q.qmm_set_gemm_weight_operand(False)
    Y = gc.gemm(d, packed, 4, a16[0:4], sx[0:4], kernel=8)   # CUDA-core small-M kernel
    done("gemm_rows", Y)
    q.qmm_set_gemm_narrow(q.NARROW_ALWAYS)
    try:
        Y = gc.gemm(d, packed, 16, a16[0:16], sx[0:16], kernel=13)   # weights in the N slot
        done("gemm_narrow", Y)
    finally:
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    # two activation tiles, group 128
    N2, K2, g2, M2 = 256, 512, 128, 150
    qb2, sw2, x2 = gc.w4a8_case(92, "checked/w4a8/g128", N2, K2, g2, g2, M2)
    d2, packed2 = gc.pack(gc.W4A8, N2, K2, g2, qb2, sw2)
    _, a16b, sxb, _, _ = gc.prep_w4a8(x2, g2, g2)
    Y = gc.gemm(d2, packed2, M2, a16b, sxb, kernel=5)
    done("gemm_g128", Y)
    q.qmm_set_gemm_narrow(q.NARROW_ALWAYS)
    try:
        Y = gc.gemm(d2, packed2, 16, a16b[0:16], sxb[0:16], kernel=14)   # e4m3 operands, weights in N
        done("gemm_narrow_e4m3", Y)
    finally:
        q.qmm_set_gemm_narrow(q.NARROW_AUTO)
    # siblings
    ys = [gc.guarded((n,), torch.float32, float("nan")) for n in (N, N2)]
    qb3, sw3, _ = gc.w4a8_case(93, "checked/sib", N2, K, g, g, 1)
    d3, packed3 = gc.pack(gc.W4A8, N2, K, g, qb3, sw3)
    q.qmm_gemv_fused_siblings([d, d3], [packed, packed3], gc.t(x[0]), 0, g, ys)
    done("siblings_0", ys[0])
    done("siblings_1", ys[1])
    # codebook weights: GEMV and GEMM
    idx, swc, C, cb, xc = gc.cq4_case(94, "checked/cq4", N, K, g, g, M)
    dc, packedc = gc.pack_cq4(N, K, g, idx, C, cb, swc)
    ac, a16c, sxc, _, _ = gc.prep_w4a8(xc, g, g)
    y = gc.gemv(dc, packedc, ac[0:1].reshape(-1), sxc[0:1].reshape(-1), workspace=False)
    done("gemv_cq4", y)
    Y = gc.gemm(dc, packedc, M, a16c, sxc, kernel=11)
    done("gemm_cq4", Y)
    # affine: group sums and the GEMM (an odd row count)
    Na, Ka, Ma = 256, 512, 65
    lay = qmm_synth.Layer("checked/affine", gc.AFFINE, Na, Ka, 64, 0)
    qa, sa, ba = qmm_synth.layer_weights(95, "checked/affine", lay)
    xa = qmm_synth.layer_activations(95, "checked/affine/x", lay, Ma)
    da, packeda = gc.pack(gc.AFFINE, Na, Ka, 64, qa, sa, ba)
    x16 = gc.t(xa.view(np.float16)) if xa.dtype == np.uint16 else gc.t(xa.astype(np.float16))
    S = gc.guarded((Ma, Ka // 64), torch.float32)
    q.qmm_prep_act(gc.AFFINE, Ma, Ka, 64, 0, x16, 1, gsum=S)
    done("prep_affine", S)
    Y = gc.gemm(da, packeda, Ma, x16, S, kernel=6)
    done("gemm_affine", Y)
    gc.assert_guards_intact()
    np.savez(out_path, **outs)
    return status


CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bit_group_quantized_qmm_gb300 as q
assert q.LIB_PATH.endswith("libqmm_gb300_checked.so"), q.LIB_PATH
from tests.test_gpu_checked import run_cases
print(json.dumps(run_cases(sys.argv[2])))
"""


def test_checked_variant_is_clean_and_identical(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300 as q
    lib_checked = os.path.join(os.path.dirname(q.__file__), "libqmm_gb300_checked.so")
    if not os.path.exists(lib_checked):
        pytest.fail("libqmm_gb300_checked.so not built (__graft_entry__.build() builds it)")
    checked_npz = str(tmp_path / "checked.npz")
    env = dict(os.environ, QMM_CHECKED_LIBRARY="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, checked_npz], env=env, capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    status = json.loads(r.stdout.strip().splitlines()[-1])
    assert status and all(v == 0 for v in status.values()), status
    product_npz = str(tmp_path / "product.npz")
    run_cases(product_npz)
    a, b = np.load(checked_npz), np.load(product_npz)
    assert sorted(a.files) == sorted(b.files)
    for name in a.files:
        assert np.array_equal(a[name].view(np.uint8), b[name].view(np.uint8)), name
