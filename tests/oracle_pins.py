"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when that oracle disagrees with a library routine, a closed form, a brute-force
computation or a hand-worked fixture. ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on copies with planted
mistakes and requires each mistake to be caught.
"""

from __future__ import annotations

import os

import numpy as np
import scipy.linalg

import qmm_synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
W4A8, AFFINE, CQ4 = 0, 1, 2


# ----------------------------------------------------------------- fixtures

def read_cases(name):
    """Parse a golden file of ``case`` blocks with ``key = value`` lines."""
    cases, cur = [], None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line.split()[1], "chunk": []}
                cases.append(cur)
                continue
            key, _, val = line.partition("=")
            key, val = key.strip(), val.strip()
            if key == "chunk":
                cur["chunk"].append([float(t) for t in val.split()])
            else:
                cur[key] = val
    return cases


def _index_values(spec, n, dtype):
    out = np.zeros(n, dtype=dtype)
    for tok in spec.split():
        i, v = tok.split(":")
        if i == "all":
            out[:] = float(v)
        else:
            out[int(i)] = float(v)
    return out


# ----------------------------------------------------------------- binary16

def pin_f16_to_f64(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.f16_to_f64(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def pin_f64_to_f16(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between neighbouring fp16 values (binary16 spacing 2^-10 at 1)
        1.0 + (np.arange(0, 64) + 0.5) * 2.0 ** -10,
        -(2.0 + (np.arange(0, 64) + 0.5) * 2.0 ** -9),
        (np.arange(0, 64) + 0.5) * 2.0 ** -24,           # subnormal ties
        [0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, 2.0 ** -25, 2.0 ** -26, 6.1e-5],
    ])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = orc.f64_to_f16(vals)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------- Hadamard

def pin_hadamard_matrix(orc):
    """FWHT(e_i) is column i of the Sylvester matrix; H H^T = n I."""
    for n in (2, 4, 8, 16, 32, 64, 128):
        ref = scipy.linalg.hadamard(n)
        H32 = np.stack([orc.fwht_f32(np.eye(n, dtype=np.float32)[i]) for i in range(n)], axis=1)
        H64 = np.stack([orc.fwht_f64(np.eye(n)[i]) for i in range(n)], axis=1)
        assert np.array_equal(H32, ref.astype(np.float32)), n
        assert np.array_equal(H64, ref.astype(np.float64)), n
        assert np.array_equal(H64 @ H64.T, n * np.eye(n)), n


def pin_hadamard_involution_and_error(orc):
    """FWHT(FWHT(v)) = n v (fp64); fp32 transform within its rounding bound."""
    rng = np.random.default_rng(2)
    for n in (64, 128):
        v = rng.standard_normal(n)
        twice = orc.fwht_f64(orc.fwht_f64(v))
        assert np.allclose(twice, n * v, rtol=0, atol=1e-12 * n * np.abs(v).max())
        v32 = v.astype(np.float32)
        exact = scipy.linalg.hadamard(n) @ v32.astype(np.float64)
        got = orc.fwht_f32(v32).astype(np.float64)
        bound = np.log2(n) * 2.0 ** -23 * np.abs(v32).astype(np.float64).sum()
        assert np.all(np.abs(got - exact) <= bound)


def pin_rotation_invariance(orc):
    """(W H^T/sqrt n)(H x/sqrt n) = W x per group, in fp64."""
    rng = np.random.default_rng(3)
    for n, K in ((64, 256), (128, 512)):
        W = rng.standard_normal((8, K))
        x = rng.standard_normal(K)
        Wr = np.concatenate([np.stack([orc.fwht_f64(W[r, g:g + n]) for r in range(8)]) / np.sqrt(n)
                             for g in range(0, K, n)], axis=1)
        xr = np.concatenate([orc.fwht_f64(x[g:g + n]) / np.sqrt(n) for g in range(0, K, n)])
        assert np.allclose(Wr @ xr, W @ x, rtol=0, atol=1e-12 * np.abs(W).sum(axis=1).max() * np.abs(x).max())


# ----------------------------------------------------------------- prep

def pin_quant_fixture(orc):
    for case in read_cases("quant_ties.txt"):
        g = int(case["group"])
        had = int(case["hadamard"])
        x = _index_values(case["x"], g, np.float32)[None, :]
        a, sx, asum = orc.prep_w4a8(x, g, had)
        codes = _index_values(case["codes"], g, np.int64)
        assert np.array_equal(a[0].astype(np.int64), codes), case["name"]
        assert sx[0, 0] == np.float32(float(case["sx"])), case["name"]
        assert asum[0, 0] == codes.sum(), case["name"]


def pin_quant_properties(orc):
    """Amax maps to +-127, codes in range, codes are nearest integers, zero groups."""
    for group, had in ((64, 0), (64, 64), (128, 128)):
        x = qmm_synth.activations_f32(0, f"pin/{group}/{had}", 5, 4 * group, outlier_frac=0.01)
        x[2, group:2 * group] = 0.0                       # one all-zero group
        a, sx, asum = orc.prep_w4a8(x, group, had)
        G = x.shape[1] // group
        c = (1.0 / np.sqrt(group)) if had else 1.0
        assert a.min() >= -127 and a.max() <= 127
        assert np.array_equal(asum, a.reshape(5, G, group).astype(np.int64).sum(-1))
        for m in range(5):
            for g in range(G):
                v = x[m, g * group:(g + 1) * group].astype(np.float64)
                if had:
                    v = scipy.linalg.hadamard(group) @ v
                amax = np.abs(v).max()
                ag = a[m, g * group:(g + 1) * group].astype(np.float64)
                if amax == 0:
                    assert sx[m, g] == 0 and not ag.any()
                    continue
                s = float(sx[m, g]) / c
                assert abs(s - amax / 127) <= 1e-6 * amax / 127
                assert np.abs(ag).max() == 127
                assert ag[np.argmax(np.abs(v))] == np.sign(v[np.argmax(np.abs(v))]) * 127
                # nearest integer to v/s (slack for the fp32 transform and division)
                assert np.all(np.abs(ag * s - v) <= 0.5 * s + 1e-5 * amax)


def pin_rotated_quant_exact(orc):
    """With integer inputs whose transform is exact in fp32, rotating inside the
    prepass equals quantizing the library-transformed input, and sx carries
    the normalisation 1/sqrt(n)."""
    rng = np.random.default_rng(4)
    for n in (64, 128):
        x = rng.integers(-3, 4, size=(3, 2 * n)).astype(np.float32)
        Hx = np.concatenate([x[:, g:g + n] @ scipy.linalg.hadamard(n).T for g in (0, n)], axis=1)
        a_rot, sx_rot, _ = orc.prep_w4a8(x, n, n)
        a_ref, sx_ref, _ = orc.prep_w4a8(Hx.astype(np.float32), n, 0)
        assert np.array_equal(a_rot, a_ref)
        assert np.array_equal(sx_rot, (sx_ref * np.float32(1.0 / np.sqrt(n))).astype(np.float32))


def pin_quantized_rotation_end_to_end(orc):
    """Rotated weights (unquantized) against the rotated, quantized activations
    reproduce W x within the quantization error bound."""
    rng = np.random.default_rng(5)
    for n, K in ((64, 256), (128, 256)):
        W = rng.standard_normal((16, K))
        x = rng.standard_normal((1, K)).astype(np.float32)
        a, sx, _ = orc.prep_w4a8(x, n, n)
        Wr = np.concatenate([np.stack([orc.fwht_f64(W[r, g:g + n]) for r in range(16)]) / np.sqrt(n)
                             for g in range(0, K, n)], axis=1)
        deq = a[0].astype(np.float64) * np.repeat(sx[0].astype(np.float64), n)
        y = Wr @ deq
        ref = W @ x[0].astype(np.float64)
        bound = np.abs(Wr) @ (np.repeat(sx[0].astype(np.float64), n) * 0.5) * (1 + 1e-5) + 1e-9
        assert np.all(np.abs(y - ref) <= bound)


# ----------------------------------------------------------------- weights

def pin_nibble_order(orc):
    fix = {}
    with open(os.path.join(GOLDEN, "nibble_order.txt")) as f:
        for raw in f:
            line = raw.strip()
            if line and not line.startswith("#"):
                k, _, v = line.partition("=")
                fix[k.strip()] = v.split()
    row = np.array([[int(t, 16) for t in fix["bytes"]]], dtype=np.uint8)
    K = 2 * row.shape[1]
    assert np.array_equal(orc.unpack_nibbles(W4A8, row, K)[0], np.array(fix["w4a8"], dtype=np.int8))
    assert np.array_equal(orc.unpack_nibbles(AFFINE, row, K)[0], np.array(fix["affine"], dtype=np.int8))


def _zero_weights(variant, N, K, group):
    G = K // group
    q = np.zeros((N, K), dtype=np.int8)
    s = np.zeros((N, G), dtype=np.uint16)
    b = np.zeros((N, G), dtype=np.uint16) if variant == AFFINE else None
    return q, s, b


def pin_pack_positions(orc):
    with open(os.path.join(GOLDEN, "pack_positions.txt")) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    for ln in lines:
        left, mid, right = [p.split() for p in ln.split("|")]
        if left[0] == "scale":
            variant = W4A8 if left[1] == "w4a8" else AFFINE
            N, K, group = map(int, left[2:5])
            n, g = map(int, mid)
            q, s, b = _zero_weights(variant, N, K, group)
            s[n, g] = 0x1234
            if b is not None:
                b[n, g] = 0x5678
            blob = orc.pack_from_values(variant, N, K, group, q, s, b)
            off = int(right[0])
            assert blob[off] == 0x34 and blob[off + 1] == 0x12, ln
            if right[1] != "-":
                boff = int(right[1])
                assert blob[boff] == 0x78 and blob[boff + 1] == 0x56, ln
            continue
        variant = W4A8 if left[0] == "w4a8" else AFFINE
        N, K, group = map(int, left[1:4])
        n, k = map(int, mid)
        q, s, b = _zero_weights(variant, N, K, group)
        base = orc.pack_from_values(variant, N, K, group, q, s, b)
        v = 5
        q[n, k] = v
        blob = orc.pack_from_values(variant, N, K, group, q, s, b)
        diff = np.nonzero(blob != base)[0]
        off = int(right[0])
        assert list(diff) == [off], (ln, diff)
        u = (v + 8) if variant == W4A8 else v
        nib = (blob[off] >> 4) if right[1] == "hi" else (blob[off] & 0xF)
        assert nib == u, ln


def pin_pack_roundtrip_and_invariance(orc):
    """unpack(pack(q)) == q; packing from nibble bytes and from values given in
    another layout (transposed, K-major) gives identical bytes; padded rows."""
    for variant, N, K, group in ((W4A8, 200, 256, 64), (W4A8, 130, 512, 128), (AFFINE, 129, 192, 64)):
        q_bytes, s, b = qmm_synth.layer_weights(7, f"pin/pack/{variant}/{group}",
                                                qmm_synth.Layer("w", variant, N, K, group, 0))
        blob = orc.pack(variant, N, K, group, q_bytes, s, b)
        assert blob.size == ((N + 127) // 128) * (K // group) * (64 * group + 256 + (256 if variant else 0))
        q, s2, b2 = orc.unpack_blob(variant, N, K, group, blob)
        vals = orc.unpack_nibbles(variant, q_bytes, K)
        assert np.array_equal(q, vals)
        assert np.array_equal(s2, s)
        if variant == AFFINE:
            assert np.array_equal(b2, b)
        # values handed over K-major, transposed back: same bytes
        kmajor = np.ascontiguousarray(vals.T)
        assert np.array_equal(orc.pack_from_values(variant, N, K, group, kmajor.T, s, b), blob)
        # brute-force reading of the nibble bytes agrees with the unpacker
        lo = (q_bytes & 0xF).astype(np.int64)
        hi = (q_bytes >> 4).astype(np.int64)
        raw = np.empty((N, K), dtype=np.int64)
        raw[:, 0::2], raw[:, 1::2] = lo, hi
        if variant == W4A8:
            raw = np.where(raw >= 8, raw - 16, raw)
        assert np.array_equal(vals.astype(np.int64), raw)
        # padded rows of the last tile: q = 0, zero scales
        T, G = (N + 127) // 128, K // group
        Npad = T * 128
        qpad, spad, _ = orc.unpack_blob(variant, Npad, K, group, blob)
        assert not qpad[N:].any() and not spad[N:].any()


def pin_interleaved4_fixture(orc):
    """Hand-worked 4-row panels (tests/golden/interleaved4_panels.txt)."""
    for case in read_cases("interleaved4_panels.txt"):
        N, K, group, ck = (int(case[k]) for k in ("N", "K", "group", "chunk_k"))
        G = K // group
        nblk = (N + 3) // 4
        panels = np.arange(nblk * 2 * K, dtype=np.int64).astype(np.uint8)
        pscales = np.arange(nblk * G * 4, dtype=np.uint16)
        q, s, b = orc.interleaved4_to_rows(N, K, group, ck, panels, pscales, pscales)
        for n in range(N):
            left, _, right = case[f"row{n}"].partition("|")
            assert list(q[n]) == [int(t, 16) for t in left.split()], (case["name"], n)
            assert list(s[n]) == [int(t) for t in right.split()], (case["name"], n)
            assert list(b[n]) == list(s[n])


def pin_interleaved4_layout(orc):
    """4-row panels against a numpy reshape/transpose of the row-major bytes
    (every chunk width, N not a multiple of 4), and the page's statement that
    each 128-wide k range of block nb is the 256-byte sub-panel at
    nb*2K + g*256."""
    rng = np.random.default_rng(11)
    for N, K, group in ((8, 256, 64), (6, 384, 128), (13, 128, 64)):
        G = K // group
        nblk = (N + 3) // 4
        q = rng.integers(0, 256, size=(nblk * 4, K // 2), dtype=np.uint8)
        sc = rng.integers(0, 65536, size=(nblk * 4, G), dtype=np.uint16)
        for ck in (8, 16, 32, 64, 128):
            if K % ck:
                continue
            cb = ck // 2
            panels = q.reshape(nblk, 4, K // ck, cb).transpose(0, 2, 1, 3).reshape(-1)
            psc = sc.reshape(nblk, 4, G).transpose(0, 2, 1).reshape(-1)
            q2, s2, _ = orc.interleaved4_to_rows(N, K, group, ck, panels, psc)
            assert np.array_equal(q2, q[:N]), (N, K, ck)
            assert np.array_equal(s2, sc[:N]), (N, K, ck)
            # rows of the last block beyond N are never read
            if N % 4:
                junk = panels.copy().reshape(nblk, K // ck, 4, cb)
                junk[-1, :, N % 4:, :] ^= 0x5A
                q3, _, _ = orc.interleaved4_to_rows(N, K, group, ck, junk.reshape(-1), psc)
                assert np.array_equal(q3, q[:N])
            if K % 128 == 0 and 128 % ck == 0:
                vng = K // 128
                for nb in range(nblk):
                    for g in range(vng):
                        only = np.zeros_like(panels)
                        at = (nb * vng + g) * 256
                        assert at == nb * 2 * K + g * 256
                        only[at:at + 256] = 0xFF
                        Nf = nblk * 4
                        q4, _, _ = orc.interleaved4_to_rows(Nf, K, group, ck, only, psc)
                        rows, cols = np.nonzero(q4)
                        assert set(rows) == set(range(4 * nb, 4 * nb + 4))
                        assert set(cols) == set(range(64 * g, 64 * g + 64)) and len(rows) == 256


# ----------------------------------------------------------------- full-K rotation

def _rotation_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "rotation_order.txt")) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case "):
                cur = {"name": line.split()[1]}
                cases.append(cur)
                continue
            key, _, val = line.partition("=")
            cur[key.strip()] = [float(t) for t in val.split()]
    out = []
    for c in cases:
        K, group = int(c["K"][0]), int(c["group"][0])
        R = np.array([c[f"R{i}"] for i in range(K)], dtype=np.float64)
        out.append((c["name"], K, group, R, np.array(c["x"]), np.array(c["z"])))
    return out


def pin_rotation_fixture(orc):
    """Hand-worked z = R x: summation order, fused rounding, orientation
    (tests/golden/rotation_order.txt); codes are the pinned quantization of z."""
    for name, K, group, R, x, z in _rotation_cases():
        assert np.array_equal(R.astype(np.float32).astype(np.float64), R), name   # exact fp32 inputs
        a, sx, asum, z2 = orc.prep_rotated(R.astype(np.float32), x.astype(np.float32)[None], group)
        assert np.array_equal(z2[0].astype(np.float64), z), (name, z2[0], z)
        a0, sx0, asum0 = orc.prep_w4a8(z.astype(np.float32)[None], group, 0)
        assert np.array_equal(a, a0) and np.array_equal(sx, sx0) and np.array_equal(asum, asum0), name


def pin_rotation_properties(orc):
    """Random orthogonal R (fp32): z within the fp32 dot-product error bound of
    fp64 R x; identity R = no rotation; a signed permutation moves values
    exactly (orientation R x, not R^T x); rotating both W (W R^T) and x leaves
    W x unchanged within the bound; codes = the pinned quantization of z."""
    u = 2.0 ** -24
    for K, group, M in ((256, 64, 3), (384, 128, 2)):
        R = qmm_synth.orthogonal_f32(0, f"pin/rot/{K}", K)
        R64 = R.astype(np.float64)
        assert np.allclose(R64 @ R64.T, np.eye(K), atol=1e-5)
        x = qmm_synth.activations_f32(0, f"pin/rot/x/{K}", M, K, 0.01)
        x64 = x.astype(np.float64)
        a, sx, asum, z = orc.prep_rotated(R, x, group)
        gam = K * u / (1 - K * u)
        bound = gam * (np.abs(x64) @ np.abs(R64).T)
        assert np.all(np.abs(z - x64 @ R64.T) <= bound)
        a0, sx0, asum0 = orc.prep_w4a8(z, group, 0)
        assert np.array_equal(a, a0) and np.array_equal(sx, sx0) and np.array_equal(asum, asum0)
        # identity: the plain prepass without rotation
        aI, sxI, asumI, zI = orc.prep_rotated(np.eye(K, dtype=np.float32), x, group)
        aP, sxP, asumP = orc.prep_w4a8(x, group, 0)
        assert np.array_equal(zI, x) and np.array_equal(aI, aP) and np.array_equal(sxI, sxP)
        # signed permutation: z[i] = sign[i] * x[perm[i]] exactly
        rng = np.random.default_rng(K)
        perm = rng.permutation(K)
        sign = rng.choice([-1.0, 1.0], size=K)
        Pm = np.zeros((K, K), dtype=np.float32)
        Pm[np.arange(K), perm] = sign
        assert not np.array_equal(Pm, Pm.T)
        _, _, _, zp = orc.prep_rotated(Pm, x, group)
        assert np.array_equal(zp, (x[:, perm] * sign).astype(np.float32))
        # W x == (W R^T)(R x) up to the rotation's rounding
        W = qmm_synth.normal(0, f"pin/rot/W/{K}", 5 * K).reshape(5, K)
        Wr = W @ R64.T
        y0 = x64 @ W.T
        y1 = z.astype(np.float64) @ Wr.T
        tol = bound @ np.abs(Wr).T + 1e-9 * (np.abs(x64) @ np.abs(W).T)
        assert np.all(np.abs(y1 - y0) <= tol)


# ----------------------------------------------------------------- W4A8 GEMM

def _unpack(q_bytes, K, variant):
    lo = (q_bytes & 0xF).astype(np.int64)
    hi = (q_bytes >> 4).astype(np.int64)
    raw = np.empty((q_bytes.shape[0], K), dtype=np.int64)
    raw[:, 0::2], raw[:, 1::2] = lo, hi
    return np.where(raw >= 8, raw - 16, raw) if variant == W4A8 else raw


def pin_partials_brute_force(orc):
    for M, N, K, group in ((3, 5, 128, 64), (2, 4, 256, 128)):
        q_bytes = qmm_synth.nibble_bytes(8, "pin/partials", N, K)
        a = (qmm_synth.draws(8, "pin/a", M * K) % np.uint64(255)).astype(np.int64) - 127
        a = a.reshape(M, K).astype(np.int8)
        P = orc.partials_w4a8(q_bytes, a, group)
        q = _unpack(q_bytes, K, W4A8)
        for m in range(M):
            for n in range(N):
                for g in range(K // group):
                    ref = 0
                    for k in range(g * group, (g + 1) * group):
                        ref += int(q[n, k]) * int(a[m, k])
                    assert P[m, n, g] == ref
        # a == 1 gives the group sums of q
        ones = np.ones((1, K), dtype=np.int8)
        P1 = orc.partials_w4a8(q_bytes, ones, group)
        assert np.array_equal(P1[0], q.reshape(N, K // group, group).sum(-1))
        # bound |P| <= 8 * 127 * group, reached by q = -8, a = -127
        worst = np.full((1, K // 2), 0x88, dtype=np.uint8)
        Pw = orc.partials_w4a8(worst, np.full((1, K), -127, dtype=np.int8), group)
        assert np.all(Pw == 8 * 127 * group)


def pin_gemm_w4a8_dequant(orc):
    """Integer-group formulation == dequantize-then-fp64-matmul (brute force)."""
    for M, N, K, group, had in ((4, 96, 256, 64, 64), (3, 40, 512, 128, 128), (2, 33, 192, 64, 0)):
        lay = qmm_synth.Layer("w", W4A8, N, K, group, had)
        q_bytes, sw, _ = qmm_synth.layer_weights(9, f"pin/gemm/{group}", lay)
        x = qmm_synth.layer_activations(9, f"pin/gemm/{group}", lay, M)
        a, sx, _ = orc.prep_w4a8(x, group, had)
        Y, Ymag = orc.gemm_w4a8(q_bytes, sw, a, sx, group)
        q = _unpack(q_bytes, K, W4A8).astype(np.float64)
        swf = sw.view(np.float16).astype(np.float64)
        Wd = q * np.repeat(swf, group, axis=1)                          # [N][K]
        Ad = a.astype(np.float64) * np.repeat(sx.astype(np.float64), group, axis=1)   # [M][K]
        ref = Ad @ Wd.T
        assert np.all(np.abs(Y - ref) <= 1e-12 * Ymag + 1e-300)
        assert np.all(Ymag >= np.abs(Y) * (1 - 1e-15))
        # sampled rows agree with the full result
        rows = np.array([N - 1, 0, N // 2], dtype=np.int32)
        Yr, Ymr = orc.gemm_w4a8(q_bytes, sw, a, sx, group, rows=rows)
        assert np.array_equal(Yr, Y[:, rows]) and np.array_equal(Ymr, Ymag[:, rows])


# ----------------------------------------------------------------- CQ4

def _cq4_identity(q_bytes):
    """Index bytes that, with C[i] = i - 8, reproduce the symmetric nibbles.

    A two's-complement nibble u stands for q = u - 16*(u >= 8); its index in the
    ascending level set -8..7 is q + 8 = u XOR 8.
    """
    return (q_bytes ^ 0x88).astype(np.uint8), np.arange(-8, 8, dtype=np.int8)


def pin_cq4_identity_codebook_equals_w4a8(orc):
    """The identity codebook with cb_scale 1 is the symmetric variant, bit for bit."""
    for M, N, K, group, had in ((3, 70, 256, 64, 64), (2, 33, 256, 128, 0)):
        lay = qmm_synth.Layer("w", W4A8, N, K, group, had)
        q_bytes, sw, _ = qmm_synth.layer_weights(21, f"pin/cq4id/{group}", lay)
        x = qmm_synth.layer_activations(21, f"pin/cq4id/{group}", lay, M)
        a, sx, _ = orc.prep_w4a8(x, group, had)
        idx, C = _cq4_identity(q_bytes)
        assert np.array_equal(orc.partials_cq4(idx, C, a, group), orc.partials_w4a8(q_bytes, a, group))
        Yc, Ymc = orc.gemm_cq4(idx, C, 1.0, sw, a, sx, group)
        Yw, Ymw = orc.gemm_w4a8(q_bytes, sw, a, sx, group)
        assert np.array_equal(Yc, Yw) and np.array_equal(Ymc, Ymw)
        # the blobs agree before the trailer on whole 128-row tiles (padding
        # rows differ: index 0 there, the symmetric q = 0 stored as 8)
        Nt = N - N % 128 or 128
        q_t, sw_t = np.resize(q_bytes, (Nt, K // 2)), np.resize(sw, (Nt, K // group))
        idx_t, _ = _cq4_identity(q_t)
        bc = orc.pack_cq4(Nt, K, group, idx_t, C, 1.0, sw_t)
        bw = orc.pack(W4A8, Nt, K, group, q_t, sw_t)
        assert bc.size == bw.size + 32 and np.array_equal(bc[:-32], bw)


def pin_cq4_partials_brute_force(orc):
    for M, N, K, group in ((2, 3, 128, 64), (1, 2, 256, 128)):
        idx = qmm_synth.nibble_bytes(22, "pin/cq4p", N, K)
        C = qmm_synth.codebook_i8(22, f"pin/cq4p/cb/{group}")
        a = (qmm_synth.draws(22, "pin/cq4p/a", M * K) % np.uint64(255)).astype(np.int64) - 127
        a = a.reshape(M, K).astype(np.int8)
        P = orc.partials_cq4(idx, C, a, group)
        i = _unpack(idx, K, CQ4)
        for m in range(M):
            for n in range(N):
                for g in range(K // group):
                    ref = 0
                    for k in range(g * group, (g + 1) * group):
                        ref += int(C[i[n, k]]) * int(a[m, k])
                    assert P[m, n, g] == ref
        # bound |P| <= 127 * 127 * group, reached by C = -127 everywhere, a = -127
        worst = np.full(16, -127, dtype=np.int8)
        Pw = orc.partials_cq4(idx[:1], worst, np.full((1, K), -127, dtype=np.int8), group)
        assert np.all(Pw == 127 * 127 * group)


def pin_cq4_dequant_and_invariances(orc):
    """Integer-group form == dequantize-then-fp64-matmul; relabeling and scale laws."""
    for M, N, K, group, had in ((4, 96, 256, 64, 64), (2, 40, 512, 128, 128)):
        lay = qmm_synth.Layer("w", CQ4, N, K, group, had)
        idx, sw, _ = qmm_synth.layer_weights(23, f"pin/cq4/{group}", lay)
        C, cb = qmm_synth.layer_codebook(23, f"pin/cq4/{group}")
        x = qmm_synth.layer_activations(23, f"pin/cq4/{group}", lay, M)
        a, sx, _ = orc.prep_w4a8(x, group, had)
        Y, Ymag = orc.gemm_cq4(idx, C, cb, sw, a, sx, group)
        i = _unpack(idx, K, CQ4)
        swf = sw.view(np.float16).astype(np.float64)
        Wd = float(np.float32(cb)) * C.astype(np.float64)[i] * np.repeat(swf, group, axis=1)
        Ad = a.astype(np.float64) * np.repeat(sx.astype(np.float64), group, axis=1)
        ref = Ad @ Wd.T
        assert np.all(np.abs(Y - ref) <= 1e-12 * Ymag + 1e-300)
        # relabeling: permute the table and the indices with it -> same partials
        perm = (np.arange(16) * 7 + 3) % 16                  # a permutation of 0..15
        inv = np.argsort(perm)
        C2 = C[perm]                                         # C2[j] = C[perm[j]]
        i2 = inv[i]                                          # C2[i2] = C[perm[inv[i]]] = C[i]
        idx2 = (i2[:, 0::2] | (i2[:, 1::2] << 4)).astype(np.uint8)
        assert np.array_equal(orc.partials_cq4(idx2, C2, a, group), orc.partials_cq4(idx, C, a, group))
        # negating the table or doubling cb_scale scales Y exactly
        Yn, _ = orc.gemm_cq4(idx, (-C.astype(np.int16)).astype(np.int8), cb, sw, a, sx, group)
        assert np.array_equal(Yn, -Y)
        Y2, _ = orc.gemm_cq4(idx, C, 2.0 * cb, sw, a, sx, group)
        assert np.array_equal(Y2, 2.0 * Y)
        # sampled rows agree with the full result
        rows = np.array([N - 1, 0, N // 2], dtype=np.int32)
        Yr, Ymr = orc.gemm_cq4(idx, C, cb, sw, a, sx, group, rows=rows)
        assert np.array_equal(Yr, Y[:, rows]) and np.array_equal(Ymr, Ymag[:, rows])


def pin_cq4_blob_trailer_and_roundtrip(orc):
    N, K, group = 130, 192, 64
    idx = qmm_synth.nibble_bytes(24, "pin/cq4b", N, K)
    sw = qmm_synth.uniform_f16(24, "pin/cq4b/s", (N, K // group), 0.005, 0.02)
    C = qmm_synth.codebook_i8(24, "pin/cq4b/cb")
    cb = 0.0625
    blob = orc.pack_cq4(N, K, group, idx, C, cb, sw)
    T, G = (N + 127) // 128, K // group
    assert blob.size == orc.packed_size(CQ4, N, K, group) == T * G * (64 * group + 256) + 32
    tr = blob[-32:]
    assert np.array_equal(tr[:16].view(np.int8), C)
    assert tr[16:20].view("<f4")[0] == np.float32(cb)
    assert not tr[20:].any()
    q, s, _ = orc.unpack_blob(CQ4, N, K, group, blob)
    assert np.array_equal(q, _unpack(idx, K, CQ4)) and np.array_equal(s, sw)
    # the nibbles are stored raw: the symmetric variant reads index i as i - 8
    qs, _, _ = orc.unpack_blob(W4A8, N, K, group, blob)
    assert np.array_equal(qs.astype(np.int64), _unpack(idx, K, CQ4) - 8)
    # padding rows of the last tile hold index 0 and zero scales
    qp, sp, _ = orc.unpack_blob(CQ4, T * 128, K, group, blob)
    assert not qp[N:].any() and not sp[N:].any()


# ----------------------------------------------------------------- affine

def pin_group_sum_tree_fixture(orc):
    for case in read_cases("group_sum_tree.txt"):
        x = np.array(case["chunk"], dtype=np.float32).reshape(1, 64)
        S = orc.group_sums_affine(x)
        assert S[0, 0] == np.float32(float(case["expect"])), case["name"]


def pin_group_sums_close_to_exact(orc):
    x16 = qmm_synth.activations_f16(10, "pin/gs", 6, 5 * 64)
    xf = x16.view(np.float16).astype(np.float32)
    S = orc.group_sums_affine(xf)
    exact = xf.astype(np.float64).reshape(6, 5, 64).sum(-1)
    bound = 7 * 2.0 ** -24 * np.abs(xf).astype(np.float64).reshape(6, 5, 64).sum(-1)
    assert np.all(np.abs(S - exact) <= bound)


def pin_affine_dequant_and_bias(orc):
    M, N, K, group = 3, 40, 256, 64
    G = K // group
    lay = qmm_synth.Layer("w", AFFINE, N, K, group, 0)
    q_bytes, s, b = qmm_synth.layer_weights(11, "pin/aff", lay)
    x16 = qmm_synth.layer_activations(11, "pin/aff", lay, M)
    xf = x16.view(np.float16).astype(np.float64)
    Y, Ymag = orc.gemm_affine(q_bytes, s, b, x16)
    q = _unpack(q_bytes, K, AFFINE).astype(np.float64)
    sf = s.view(np.float16).astype(np.float64)
    bf = b.view(np.float16).astype(np.float64)
    Wd = q * np.repeat(sf, group, axis=1) + np.repeat(bf, group, axis=1)
    ref = xf @ Wd.T
    assert np.allclose(Y, ref, rtol=0, atol=1e-12 * Ymag.max())
    assert np.allclose(Ymag, np.abs(xf) @ np.abs(Wd).T, rtol=1e-12, atol=0)
    # q == 0: only the bias term, b * (group sums of x)
    zero = np.zeros_like(q_bytes)
    Y0, _ = orc.gemm_affine(zero, s, b, x16)
    gsum = xf.reshape(M, G, group).sum(-1)
    assert np.allclose(Y0, gsum @ bf.T, rtol=0, atol=1e-12 * np.abs(gsum).max() * np.abs(bf).sum(1).max())
    # s == 0, b == 1: row sums of x
    one = np.full_like(b, 0x3C00)
    Y1, _ = orc.gemm_affine(q_bytes, np.zeros_like(s), one, x16)
    assert np.allclose(Y1, np.repeat(xf.sum(1, keepdims=True), N, axis=1), rtol=0, atol=1e-12 * np.abs(xf).sum())


ALL_PINS = [
    pin_f16_to_f64, pin_f64_to_f16,
    pin_hadamard_matrix, pin_hadamard_involution_and_error, pin_rotation_invariance,
    pin_quant_fixture, pin_quant_properties, pin_rotated_quant_exact, pin_quantized_rotation_end_to_end,
    pin_nibble_order, pin_pack_positions, pin_pack_roundtrip_and_invariance,
    pin_partials_brute_force, pin_gemm_w4a8_dequant,
    pin_group_sum_tree_fixture, pin_group_sums_close_to_exact, pin_affine_dequant_and_bias,
    pin_cq4_identity_codebook_equals_w4a8, pin_cq4_partials_brute_force, pin_cq4_dequant_and_invariances,
    pin_cq4_blob_trailer_and_roundtrip,
    pin_interleaved4_fixture, pin_interleaved4_layout,
    pin_rotation_fixture, pin_rotation_properties,
]
