"""Seeded input generator: determinism, distribution and the forced-exit mix."""
import numpy as np

import synth


def test_weights_deterministic_and_distributed():
    a = synth.normal_act16(1234, 7, 200000, synth.BF16)
    b = synth.normal_act16(1234, 7, 200000, synth.BF16)
    c = synth.normal_act16(1234, 8, 200000, synth.BF16)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    v = synth.act16_to_f32(a, synth.BF16).astype(np.float64)
    assert abs(v.mean()) < 3e-4 and abs(v.std() - 0.02) < 3e-4
    # fraction within one standard deviation of a normal
    assert abs(np.mean(np.abs(v) < 0.02) - 0.6827) < 0.01


def test_thread_count_does_not_change_values():
    import ctypes
    lib = synth._load()
    x = np.empty(300000, dtype=np.uint16)
    y = np.empty(300000, dtype=np.uint16)
    lib.synth_normal_act16(5, 3, 0.02, x.size, 0, x.ctypes.data, 1)
    lib.synth_normal_act16(5, 3, 0.02, y.size, 0, y.ctypes.data, 7)
    assert np.array_equal(x, y)


def test_prompt_ids_uniform_in_range():
    p = synth.make_prompt(1024, 4, 5000)
    assert p.min() >= 0 and p.max() < 1024
    counts = np.bincount(p.reshape(-1), minlength=1024)
    assert counts.min() > 0 and counts.max() < 3 * counts.mean()


def test_forced_exit_mixture():
    L = 32
    e = np.concatenate([synth.forced_exits(s, 64, L) for s in range(400)])
    assert e.min() >= 1 and e.max() <= L
    assert abs(np.mean(e <= 5) - 0.55) < 0.01
    # uniform inside each branch
    lo = np.bincount(e[e <= 5], minlength=6)[1:]
    assert lo.min() > 0.9 * lo.mean()
    assert abs(e.mean() - (0.55 * 3 + 0.45 * (6 + L) / 2)) < 0.2
    assert np.array_equal(synth.forced_exits(3, 8, L), synth.forced_exits(3, 8, L))


def test_param_counts():
    assert synth.LLAMA_8B.param_count() == 8_030_261_248
    assert synth.LLAMA_1B.param_count() == 1_235_814_400
