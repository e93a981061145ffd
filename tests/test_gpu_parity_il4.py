"""GPU parity of weight packing from 4-row panels (INTERLEAVED_4ROW input).

The panels are built on the host from seeded row-major weights by a numpy
reshape; the expected blob is the oracle's pack of the oracle's decoding of
those panels. Bit-exact: every byte of the blob. The GPU blob must also equal
the one qmm_pack_weights / qmm_pack_weights_cq4 builds from the row-major
weights (cactus PR #697: the cache is byte-identical for both input layouts).
Rows of the last 4-row block beyond N hold junk that must never be read.
"""

import numpy as np
import pytest

import qmm_synth
from tests import gpu_cases as gc

pytestmark = pytest.mark.gpu

W4A8, AFFINE, CQ4 = 0, 1, 2
CHUNKS = (8, 16, 32, 64, 128)


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bit_group_quantized_qmm_gb300  # noqa: F401  (fails loudly when the library is missing)
    return torch


def _panels(rows, ck, junk_seed=5):
    """[N][W] row-major bytes or scales -> 4-row panel order; the missing rows
    of the last block are junk."""
    N, W = rows.shape
    nblk = (N + 3) // 4
    full = np.random.default_rng(junk_seed).integers(0, 1 << (8 * rows.itemsize), size=(nblk * 4, W),
                                                      dtype=np.uint64).astype(rows.dtype)
    full[:N] = rows
    if ck is None:   # scales: [nblk][G][4]
        return np.ascontiguousarray(full.reshape(nblk, 4, W).transpose(0, 2, 1).reshape(-1))
    cb = ck // 2
    return np.ascontiguousarray(full.reshape(nblk, 4, W // cb, cb).transpose(0, 2, 1, 3).reshape(-1))


def _weights(variant, N, K, group, tag):
    if variant == CQ4:
        idx, sw, C, cb, _ = gc.cq4_case(3, f"il4/{tag}", N, K, group, 0, 1)
        return idx, sw, None, C, cb
    lay = qmm_synth.Layer("p", variant, N, K, group, 0)
    qb, s, b = qmm_synth.layer_weights(3, f"il4/{tag}", lay)
    return qb, s, b, None, 1.0


def _pack_il4(variant, N, K, group, ck, qb, s, b, C, cb):
    import torch
    q = gc.lib()
    d = q.weight_desc(variant, N, K, group)
    packed = gc.guarded((q.qmm_packed_size(d),), torch.uint8, 0xA5)
    q.qmm_pack_weights_interleaved4(d, ck, gc.t(_panels(qb, ck)), gc.t(_panels(s, None)),
                                    None if b is None else gc.t(_panels(b, None)), packed, codebook=C,
                                    cb_scale=cb)
    assert q.qmm_last_kernel_id() == 1
    return packed.cpu().numpy()


def _pack_rows(variant, N, K, group, qb, s, b, C, cb):
    if variant == CQ4:
        return gc.pack_cq4(N, K, group, qb, C, cb, s)[1].cpu().numpy()
    return gc.pack(variant, N, K, group, qb, s, b)[1].cpu().numpy()


CASES = [
    (W4A8, 130, 384, 64),     # N % 4 == 2: half-used last block; two row tiles
    (W4A8, 263, 256, 128),    # N % 4 == 3
    (AFFINE, 129, 256, 64),   # N % 4 == 1, biases in panel order
    (CQ4, 130, 384, 64),
    (CQ4, 132, 512, 128),
    (W4A8, 4, 128, 64),       # one block
]


@pytest.mark.parametrize("variant,N,K,group", CASES)
def test_pack_interleaved4_bytes(torch_cuda, orc, variant, N, K, group):
    qb, s, b, C, cb = _weights(variant, N, K, group, f"{variant}/{N}/{K}/{group}")
    rows_blob = _pack_rows(variant, N, K, group, qb, s, b, C, cb)
    for ck in CHUNKS:
        if K % ck:
            continue
        blob = _pack_il4(variant, N, K, group, ck, qb, s, b, C, cb)
        # expected: the oracle decodes the same panels, then packs
        q2, s2, b2 = orc.interleaved4_to_rows(N, K, group, ck, _panels(qb, ck), _panels(s, None),
                                              None if b is None else _panels(b, None))
        if variant == CQ4:
            ref = orc.pack_cq4(N, K, group, q2, C, cb, s2)
        else:
            ref = orc.pack(variant, N, K, group, q2, s2, b2)
        assert np.array_equal(blob, ref), ck
        assert np.array_equal(blob, rows_blob), ck


def test_pack_interleaved4_full_size_sampled(torch_cuda, orc):
    """lm_head-sized weights (K=1536, N=262144, group 128) from panels of
    32-wide chunks: the whole blob equals the row-major pack, and the oracle
    reproduces row tiles 0, a middle one and the last byte for byte."""
    N, K, group, ck = 262144, 1536, 128, 32
    qb, s, b, C, cb = _weights(W4A8, N, K, group, "full")
    blob = _pack_il4(W4A8, N, K, group, ck, qb, s, b, C, cb)
    assert np.array_equal(blob, _pack_rows(W4A8, N, K, group, qb, s, b, C, cb))
    G, CB, T = K // group, 64 * group + 256, (N + 127) // 128
    for t0 in (0, T // 2, T - 1):
        rows = slice(128 * t0, 128 * (t0 + 1))
        q2, s2, _ = orc.interleaved4_to_rows(128, K, group, ck, _panels(qb[rows], ck), _panels(s[rows], None))
        ref = orc.pack(W4A8, 128, K, group, q2, s2)
        assert np.array_equal(blob[t0 * G * CB:(t0 + 1) * G * CB], ref), t0


def test_pack_interleaved4_control_layout_is_detected(torch_cuda):
    """Control: panels read with the wrong chunk width give a different blob."""
    N, K, group = 128, 256, 64
    qb, s, b, C, cb = _weights(W4A8, N, K, group, "control")
    import torch
    q = gc.lib()
    d = q.weight_desc(W4A8, N, K, group)
    packed = gc.guarded(q.qmm_packed_size(d), torch.uint8)
    q.qmm_pack_weights_interleaved4(d, 16, gc.t(_panels(qb, 32)), gc.t(_panels(s, None)), None, packed)
    assert not np.array_equal(packed.cpu().numpy(), _pack_rows(W4A8, N, K, group, qb, s, b, C, cb))
