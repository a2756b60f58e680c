"""Pins for the oracle's river construction (int4 round-to-nearest, fp16 scale
and zero, canonical packing).  CPU only."""
import numpy as np
import pytest
import torch

import oracle
import synth
from ongrid import ongrid_matrix, pack_canonical, unpack_canonical, ongrid_weights

FP16, BF16 = 0, 1


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("act", [FP16, BF16])
def test_rtn_ongrid_round_trip(act):
    rng = np.random.default_rng(11)
    bits, q, s, z = ongrid_matrix(rng, 6, 128, 64, act)
    for n in range(6):
        for gi in range(2):
            qq, ss, zz, rc = oracle.rtn_group(bits[n, gi * 64:(gi + 1) * 64], act)
            assert rc == 0
            assert ss == s[n, gi] and zz == z[n, gi]
            assert np.array_equal(qq, q[n, gi * 64:(gi + 1) * 64])


def test_rtn_error_bound_and_range():
    rng = np.random.default_rng(12)
    for _ in range(200):
        w = rng.normal(0, 0.02, 64).astype(np.float16)
        q, s, z, rc = oracle.rtn_group(w.view(np.uint16), FP16)
        assert rc == 0 and q.min() >= 0 and q.max() <= 15
        sv, zv = f16(s), f16(z)
        assert zv == int(zv) and 0 <= zv <= 15
        what = (q.astype(np.float64) - zv) * sv
        wv = w.astype(np.float64)
        # mixed-sign group: every weight is within half a step (plus the fp16
        # rounding of the scale, which shifts the grid by at most 15 * ulp(s))
        assert np.all(np.abs(wv - what) <= sv / 2 + 15 * abs(sv - (wv.max() - wv.min()) / 15) + 1e-12)


def test_rtn_ties_round_half_even():
    s = 2.0 ** -7
    z = 4
    # group holds the grid ends (q = 0 and 15) plus two midpoints
    vals = np.array([(0 - z) * s, (15 - z) * s, 2.5 * s, 3.5 * s, -1.5 * s] + [0.0] * 59)
    q, ss, zz, rc = oracle.rtn_group(vals.astype(np.float16).view(np.uint16), FP16)
    assert rc == 0 and f16(ss) == s and f16(zz) == z
    assert q[2] == 2 + z and q[3] == 4 + z and q[4] == -2 + z
    # odd zero point: the tie rounds w / s to even before z is added
    z = 5
    vals = np.array([(0 - z) * s, (15 - z) * s, 2.5 * s, 3.5 * s] + [0.0] * 60)
    q, ss, zz, rc = oracle.rtn_group(vals.astype(np.float16).view(np.uint16), FP16)
    assert rc == 0 and f16(zz) == z
    assert q[2] == 2 + z and q[3] == 4 + z


def test_rtn_degenerate_and_clamps():
    # all equal: scale 0 -> s = 1, z = 0, q = clamp(rint(w))
    q, s, z, rc = oracle.rtn_group(np.full(64, np.float16(3.0)).view(np.uint16), FP16)
    assert rc == 0 and s == 0x3C00 and z == 0 and np.all(q == 3)
    q, s, z, rc = oracle.rtn_group(np.full(64, np.float16(-0.25)).view(np.uint16), FP16)
    assert rc == 0 and s == 0x3C00 and z == 0 and np.all(q == 0)
    # all positive: z clamps to 0
    w = np.linspace(1.0, 2.5, 64).astype(np.float16)
    q, s, z, rc = oracle.rtn_group(w.view(np.uint16), FP16)
    assert rc == 0 and z == 0 and q.max() == 15
    # all negative: z clamps to 15, values below the grid clamp to q = 0
    q, s, z, rc = oracle.rtn_group((-w).view(np.uint16), FP16)
    assert rc == 0 and f16(z) == 15 and q.min() == 0
    # scale overflows fp16: error
    wb = torch.tensor([-1e6, 1e6] + [0.0] * 62).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert oracle.rtn_group(wb, BF16)[3] == oracle.RV_EINVAL


def test_pack_unpack_bijection():
    # every nibble value at every position of a word
    q = np.zeros((16, 64), dtype=np.uint8)
    for r in range(16):
        q[r] = (np.arange(64) + r) % 16
    p = pack_canonical(q)
    assert np.array_equal(unpack_canonical(p), q)
    assert len({int(x) for x in p.reshape(-1)}) > 8


def test_export_matches_constructed_grid_with_ragged_group():
    shape = synth.TINY  # ffn 688 = 10 * 64 + 48: the down projection ends in a ragged group
    ws, truth = ongrid_weights(shape, 64, seed=3)
    m = oracle.Model(shape, ws, 1, 8)
    assert m.quantize_river(64) == 0
    for (layer, name), (q, s, z) in truth.items():
        proj = synth.LAYER_TENSORS.index(name)
        proj = {1: 0, 2: 1, 3: 2, 4: 3, 6: 4, 7: 5, 8: 6}[proj]
        pq, ps, pz = m.export_river(layer, proj)
        assert np.array_equal(pq, pack_canonical(q)), (layer, name)
        assert np.array_equal(ps, s) and np.array_equal(pz, z), (layer, name)
    m.close()


def test_quantize_rejects_bad_args():
    m = oracle.Model(synth.TINY, synth.make_weights(synth.TINY), 1, 8)
    assert m.quantize_river(12) == oracle.RV_EINVAL  # not a multiple of 8
    assert m.quantize_river(64, 0) == oracle.RV_EINVAL  # entry below 1
    assert m.quantize_river(64, 5) == oracle.RV_EINVAL  # entry above L
    m.close()
