"""The C-ABI library on the host (no GPU needed): it builds, loads, exports
every function include/qmm.h declares, and rejects bad arguments before it
touches a device."""

import ctypes
import os
import subprocess

import pytest

import oracle


@pytest.fixture(scope="module")
def q():
    import __graft_entry__
    __graft_entry__._build_module().build()
    import bit_group_quantized_qmm_gb300 as q
    return q


def test_exports_every_declared_symbol(q):
    declared = q.declared_symbols()
    assert len(declared) >= 12
    out = subprocess.run(["nm", "-D", "--defined-only", q.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    for s in declared:
        assert hasattr(q.library(), s)


@pytest.mark.parametrize("variant,N,K,group", [(0, 1024, 1024, 64), (0, 1, 64, 64), (0, 130, 512, 128),
                                               (1, 34816, 5120, 64), (0, 262144, 1536, 128), (1, 129, 192, 64),
                                               (2, 12288, 1536, 64), (2, 130, 256, 128), (2, 1, 64, 64)])
def test_packed_size_matches_oracle(q, variant, N, K, group):
    d = q.weight_desc(variant, N, K, group)
    assert q.qmm_packed_size(d) == oracle.packed_size(variant, N, K, group)


def test_packed_size_rejects(q):
    assert q.qmm_packed_size(q.weight_desc(0, 128, 100, 64)) == 0     # K % group
    assert q.qmm_packed_size(q.weight_desc(1, 128, 256, 128)) == 0    # affine group 128
    assert q.qmm_packed_size(q.weight_desc(0, 0, 256, 64)) == 0
    assert q.qmm_packed_size(q.weight_desc(5, 128, 256, 64)) == 0
    assert q.qmm_packed_size(q.weight_desc(2, 128, 256, 32)) == 0     # CQ4 group 32


def test_host_validation(q):
    L = q.library()
    d = q.weight_desc(0, 256, 256, 64)
    bad = q.weight_desc(0, 256, 250, 64)
    D = ctypes.byref
    INV, SHAPE, DEV, MIS = 1, 2, 3, 4
    A = 1 << 20     # an aligned (never dereferenced) address
    assert L.qmm_pack_weights(D(d), None, A, None, A, None) == INV
    assert L.qmm_pack_weights(D(bad), A, A, None, A, None) == SHAPE
    assert L.qmm_pack_weights(D(d), A + 1, A, None, A, None) == MIS
    assert L.qmm_pack_weights(D(d), A, A, A, A, None) == INV          # biases for W4A8
    assert L.qmm_prep_act(0, 0, 256, 64, 0, A, 0, A, A, A, A, None, None, None) == INV
    assert L.qmm_prep_act(0, 1, 256, 64, 32, A, 0, A, A, A, A, None, None, None) == SHAPE
    assert L.qmm_prep_act(0, 1, 256, 64, 0, A, 7, A, A, A, A, None, None, None) == INV
    assert L.qmm_prep_act(0, 1, 256, 64, 0, A, 0, A, A, None, A, None, None, None) == INV   # sx required
    assert L.qmm_prep_act(1, 1, 256, 64, 0, A, 1, None, None, None, None, None, None, None) == INV  # gsum
    assert L.qmm_prep_act(1, 1, 256, 128, 0, A, 1, None, None, None, None, A, None, None) == SHAPE
    assert L.qmm_gemv(D(q.weight_desc(1, 256, 256, 64)), A, A, A, A, None, 0, None) == SHAPE
    assert L.qmm_gemv(D(d), A, A, A, A + 4, None, 0, None) == MIS
    assert L.qmm_gemm(D(d), A, 0, A, A, A, None) == INV
    assert L.qmm_gemm(D(d), A, 4, A, None, A, None) == INV
    assert L.qmm_debug_partials(D(q.weight_desc(1, 256, 256, 64)), A, 1, 0, A, A, None) == SHAPE
    assert L.qmm_debug_partials(D(d), A, 2, 0, A, A, None) == INV    # GEMV path needs M == 1
    assert L.qmm_debug_partials(D(d), A, 1, 9, A, A, None) == INV
    # sibling GEMVs: count, per-matrix shape agreement, alignment
    descs = (q.qmm_weight_desc * 3)(q.weight_desc(0, 256, 256, 64), q.weight_desc(0, 128, 256, 64),
                                    q.weight_desc(0, 64, 256, 64))
    ptrs = (ctypes.c_void_p * 3)(A, A, A)
    assert L.qmm_gemv_fused_siblings(0, descs, ptrs, A, 0, 64, ptrs, None, None, None) == INV
    assert L.qmm_gemv_fused_siblings(9, descs, ptrs, A, 0, 64, ptrs, None, None, None) == INV
    assert L.qmm_gemv_fused_siblings(3, descs, ptrs, A + 8, 0, 64, ptrs, None, None, None) == MIS
    mixed = (q.qmm_weight_desc * 2)(q.weight_desc(0, 256, 256, 64), q.weight_desc(0, 256, 512, 64))
    assert L.qmm_gemv_fused_siblings(2, mixed, ptrs, A, 0, 64, ptrs, None, None, None) == SHAPE
    grp = (q.qmm_weight_desc * 2)(q.weight_desc(0, 256, 256, 64), q.weight_desc(0, 256, 256, 128))
    assert L.qmm_gemv_fused_siblings(2, grp, ptrs, A, 0, 64, ptrs, None, None, None) == SHAPE
    nulls = (ctypes.c_void_p * 3)(A, None, A)
    assert L.qmm_gemv_fused_siblings(3, descs, nulls, A, 0, 64, ptrs, None, None, None) == INV
    # codebook weights: packed only with their codebook, one variant per sibling launch
    c = q.weight_desc(2, 256, 256, 64)
    book = (ctypes.c_int8 * 16)(*range(-8, 8))
    assert L.qmm_pack_weights(D(c), A, A, None, A, None) == INV
    assert L.qmm_pack_weights_cq4(D(d), A, book, 1.0, A, A, None) == INV          # not a CQ4 desc
    assert L.qmm_pack_weights_cq4(D(c), A, None, 1.0, A, A, None) == INV         # no codebook
    assert L.qmm_pack_weights_cq4(D(c), A, book, float("nan"), A, A, None) == INV
    assert L.qmm_pack_weights_cq4(D(c), A, book, float("inf"), A, A, None) == INV
    assert L.qmm_pack_weights_cq4(D(c), A + 2, book, 1.0, A, A, None) == MIS
    assert L.qmm_pack_weights_cq4(D(q.weight_desc(2, 256, 250, 64)), A, book, 1.0, A, A, None) == SHAPE
    assert L.qmm_gemv(D(c), A, A, A, A + 4, None, 0, None) == MIS
    assert L.qmm_gemv_workspace_size(D(c)) == L.qmm_gemv_workspace_size(D(d))
    mixv = (q.qmm_weight_desc * 2)(q.weight_desc(0, 256, 256, 64), q.weight_desc(2, 256, 256, 64))
    assert L.qmm_gemv_fused_siblings(2, mixv, ptrs, A, 0, 64, ptrs, None, None, None) == SHAPE
    # full-K rotation prepass: shapes, required outputs, dtypes, alignment
    rot = L.qmm_prep_act_rotated
    assert rot(0, 256, 64, A, A, 0, A, A, A, A, None) == INV
    assert rot(1, 256, 64, None, A, 0, A, A, A, A, None) == INV
    assert rot(1, 256, 64, A, A, 0, A, A, None, A, None) == INV       # sx required
    assert rot(1, 256, 64, A, A, 5, A, A, A, A, None) == INV
    assert rot(1, 320, 64, A, A, 0, A, A, A, A, None) == SHAPE        # K % 128
    assert rot(1, 256, 32, A, A, 0, A, A, A, A, None) == SHAPE
    assert rot(1, 256, 64, A + 4, A, 0, A, A, A, A, None) == MIS
    assert rot(1, 256, 64, A, A, 0, A, A + 2, A, A, None) == MIS
    # 4-row panel input: chunk width, K divisible by it, per-variant pointers, alignment
    il4 = L.qmm_pack_weights_interleaved4
    aff = q.weight_desc(1, 256, 256, 64)
    for bad in (0, 4, 24, 256):
        assert il4(D(d), bad, A, A, None, None, 1.0, A, None) == INV
    assert il4(D(q.weight_desc(0, 256, 320, 64)), 128, A, A, None, None, 1.0, A, None) == SHAPE
    assert il4(D(d), 32, None, A, None, None, 1.0, A, None) == INV
    assert il4(D(d), 32, A, A, A, None, 1.0, A, None) == INV          # biases on a symmetric desc
    assert il4(D(aff), 32, A, A, None, None, 1.0, A, None) == INV     # affine needs biases
    assert il4(D(d), 32, A, A, None, book, 1.0, A, None) == INV       # codebook on a W4A8 desc
    assert il4(D(c), 32, A, A, None, None, 1.0, A, None) == INV       # CQ4 needs its codebook
    assert il4(D(c), 32, A, A, None, book, float("nan"), A, None) == INV
    assert il4(D(d), 32, A + 4, A, None, None, 1.0, A, None) == MIS
    assert il4(D(aff), 32, A, A, A + 2, None, 1.0, A, None) == MIS


def test_valid_arguments_reach_the_device_probe(q):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L = q.library()
    d = q.weight_desc(0, 256, 256, 64)
    A = 1 << 20
    assert L.qmm_pack_weights(ctypes.byref(d), A, A, None, A, None) == 3
    assert L.qmm_gemm(ctypes.byref(d), A, 4, A, A, A, None) == 3
    c = q.weight_desc(2, 256, 256, 64)
    book = (ctypes.c_int8 * 16)(*range(-8, 8))
    assert L.qmm_pack_weights_cq4(ctypes.byref(c), A, book, 0.5, A, A, None) == 3
    assert L.qmm_gemm(ctypes.byref(c), A, 4, A, A, A, None) == 3
    assert L.qmm_pack_weights_interleaved4(ctypes.byref(d), 8, A, A, None, None, 1.0, A, None) == 3
    assert L.qmm_prep_act_rotated(1, 1536, 128, A, A, 0, A, A, A, A, None) == 3
    assert L.qmm_pack_weights_interleaved4(ctypes.byref(c), 128, A, A, None, book, 0.5, A, None) == 3


def test_status_strings(q):
    for s in range(8):
        assert q.status_string(s) and q.status_string(s) != "unknown status"
    assert q.status_string(99) == "unknown status"


def test_no_cpu_fallback_in_product_path():
    """The product package never imports the oracle."""
    pkg = os.path.join(os.path.dirname(os.path.dirname(__file__)), "bit_group_quantized_qmm_gb300")
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(root, f)).read()
                assert "oracle" not in text.lower(), f


def test_kernel_ids_match_header(q):
    """The binding's kernel names cover exactly the qmm_kernel_id values the
    header declares, and the narrow-kernel modes match the header's enum."""
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", "include", "qmm.h")).read()
    ids = {int(v) for v in re.findall(r"QMM_KERNEL_\w+\s*=\s*(\d+)", hdr)}
    assert ids == set(q.KERNEL_IDS), (sorted(ids), sorted(q.KERNEL_IDS))
    modes = dict(re.findall(r"(QMM_NARROW_\w+)\s*=\s*(\d+)", hdr))
    assert {int(v) for v in modes.values()} == {q.NARROW_OFF, q.NARROW_AUTO, q.NARROW_ALWAYS, q.NARROW_F16}
    assert int(modes["QMM_NARROW_AUTO"]) == q.NARROW_AUTO


def test_static_scratch_probes_the_device_first(q):
    """qmm_gemv_static_scratch validates its arguments on the host and then
    probes the device before any other CUDA call: without a supported device
    (this host has none) a valid call returns QMM_ERR_UNSUPPORTED_DEVICE, the
    code qmm_gemv gives, not QMM_ERR_CUDA from the scratch set-up."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    L = q.library()
    A = 1 << 20   # aligned, never dereferenced
    d = q.weight_desc(0, 1536, 6144, 64)   # a split-K shape: the scratch path
    assert q.qmm_gemv_workspace_size(d) > 0
    assert L.qmm_gemv_static_scratch(ctypes.byref(d), A, A, A, A, None) == 3
    assert L.qmm_gemv(ctypes.byref(d), A, A, A, A, A, q.qmm_gemv_workspace_size(d), None) == 3
