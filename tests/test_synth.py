"""The seeded input generator (no GPU): determinism, counters, distributions."""

import numpy as np

import qmm_synth


def test_counter_based_and_deterministic():
    a = qmm_synth.draws(0, "x", 1000)
    b = qmm_synth.draws(0, "x", 1000)
    assert np.array_equal(a, b)
    # element i depends only on (seed, stream, i)
    assert np.array_equal(qmm_synth.draws(0, "x", 10, start=500), a[500:510])
    assert np.array_equal(qmm_synth.draws_at(0, "x", np.array([7, 3, 999])), a[[7, 3, 999]])
    assert not np.array_equal(qmm_synth.draws(1, "x", 1000), a)
    assert not np.array_equal(qmm_synth.draws(0, "y", 1000), a)


def test_splitmix64_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state advanced by GAMMA before mixing).
    z = np.array([1, 2, 3], dtype=np.uint64) * qmm_synth.GAMMA
    out = qmm_synth._mix64(z)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_distributions():
    q = qmm_synth.nibble_bytes(0, "q", 256, 1024)
    nib = np.concatenate([(q & 0xF).ravel(), (q >> 4).ravel()])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.9 * counts.mean() and counts.max() < 1.1 * counts.mean()
    s = qmm_synth.uniform_f16(0, "s", (512, 64), 0.005, 0.02).view(np.float16).astype(np.float64)
    assert s.min() >= 0.005 - 1e-5 and s.max() <= 0.02 + 1e-5
    assert abs(s.mean() - 0.0125) < 2e-4
    x = qmm_synth.normal(0, "n", 200000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


def test_outliers():
    K = 1536
    x = qmm_synth.activations_f32(0, "x", 4, K, outlier_frac=0.01)
    for m in range(4):
        out = np.abs(x[m]) == 20.0
        assert out.sum() == round(0.01 * K)


def test_workload_catalogue():
    w = qmm_synth.workloads()
    assert set(w) == {"gemv_k1024_n1024", "gemma_decode", "prefill_gemm", "affine_gemm", "lm_head"}
    assert [l.name for l in w["gemma_decode"].layers] == ["gate_up", "down", "q", "o"]
    assert w["lm_head"].layers[0].group == 128 and w["lm_head"].Ms == [1, 2, 4, 8, 16, 32]


def test_codebook_levels():
    C = qmm_synth.codebook_i8(0, "cb")
    assert C.dtype == np.int8 and C.size == 16
    assert np.all(np.diff(C.astype(np.int64)) > 0)            # distinct, ascending
    assert C.min() >= -127 and C.max() <= 127
    assert np.array_equal(C, qmm_synth.codebook_i8(0, "cb"))
    C2, cb = qmm_synth.layer_codebook(1, "w")
    assert 0.04 <= cb <= 0.08 and float(np.float32(cb)) == cb


def test_orthogonal_draw_is_seeded_and_orthogonal():
    R = qmm_synth.orthogonal_f32(0, "t/orth", 128)
    assert R.dtype == np.float32 and R.shape == (128, 128)
    assert np.array_equal(R, qmm_synth.orthogonal_f32(0, "t/orth", 128))
    assert not np.array_equal(R, qmm_synth.orthogonal_f32(1, "t/orth", 128))
    R64 = R.astype(np.float64)
    assert np.abs(R64 @ R64.T - np.eye(128)).max() < 1e-5
