"""Backbone offloading in the oracle (paperlayer.ai section 4, Backbone
Offloading): only backbone layers 1..cap stay, so every exit is capped at
cap.  The cap is pinned against the uncapped rule and the forced-exit path:

- cap = L changes nothing (bit for bit);
- from the same cache state, the capped exit is min(uncapped exit, cap),
  and the hidden states up to that layer are the uncapped ones bit for bit;
- a capped step equals the forced-exit step at the capped exits, bit for
  bit (the cap is the forced rule applied at layer cap);
- prefill: the sequence exit is min(uncapped e_seq, cap);
- out-of-range caps, forced and fixed exits above the cap are errors."""
import numpy as np
import pytest

import oracle
import synth

RV_OK, RV_EINVAL, RV_ESTATE = 0, -1, -5


@pytest.fixture(scope="module")
def tiny():
    shape = synth.TINY
    return shape, synth.make_weights(shape)


def fresh(shape, w, cap=None):
    m = oracle.Model(shape, w, 2, 48)
    assert m.quantize_river(64, 1) == 0
    if cap is not None:
        assert m.set_exit_cap(cap) == RV_OK
    return m


def test_cap_L_changes_nothing(tiny):
    shape, w = tiny
    L = shape.n_layers
    a, b = fresh(shape, w), fresh(shape, w, L)
    prompt = synth.make_prompt(shape.vocab, 2, 12, seed=5)
    pa, pb = a.prefill(prompt, 0.2, debug=True), b.prefill(prompt, 0.2, debug=True)
    assert np.array_equal(pa["exit_layer"], pb["exit_layer"])
    assert np.array_equal(pa["logits"], pb["logits"])
    tok = pa["next_ids"]
    for tau in (0.1, 0.5, 2.0):
        oa, ob = a.decode_step(tok, tau, debug=True), b.decode_step(tok, tau, debug=True)
        assert np.array_equal(oa["exit_layer"], ob["exit_layer"])
        assert np.array_equal(oa["hidden"], ob["hidden"])
        tok = oa["next_ids"]
    a.close()
    b.close()


@pytest.mark.parametrize("cap", [1, 2, 3])
def test_capped_exit_is_min_of_uncapped_and_cap(tiny, cap):
    shape, w = tiny
    L = shape.n_layers
    a, b = fresh(shape, w), fresh(shape, w, cap)
    prompt = synth.make_prompt(shape.vocab, 2, 12, seed=6)
    a.prefill(prompt, 0.9, fixed_exit=1)
    b.prefill(prompt, 0.9, fixed_exit=1)
    kv, lens = a.get_kv(), a.lens()
    tok = np.array([3, 77], dtype=np.int32)
    seen = set()
    for tau in (-1.0, 0.0, 0.2, 0.5, 0.8, 2.0):
        a.set_kv(kv, lens)
        b.set_kv(kv, lens)
        oa = a.decode_step(tok, tau, debug=True)
        ob = b.decode_step(tok, tau, debug=True)
        assert oa["rc"] == 0 and ob["rc"] == 0
        want = np.minimum(oa["exit_layer"], cap)
        assert np.array_equal(ob["exit_layer"], want), (tau, oa["exit_layer"], ob["exit_layer"])
        seen.update(int(e) for e in oa["exit_layer"])
        for r in range(2):
            e = int(want[r])
            assert np.array_equal(oa["hidden"][: e + 1, r], ob["hidden"][: e + 1, r])
        # the cap is the forced rule at the capped exits
        b.set_kv(kv, lens)
        of = b.decode_step(tok, tau, forced=want, debug=True)
        assert np.array_equal(of["hidden"], ob["hidden"]) and np.array_equal(of["logits"], ob["logits"])
    assert len(seen) > 1  # the tau sweep exercises several exit layers
    a.close()
    b.close()


def test_capped_prefill(tiny):
    shape, w = tiny
    L = shape.n_layers
    prompt = synth.make_prompt(shape.vocab, 2, 12, seed=7)
    for tau in (-1.0, 0.3, 2.0):
        a, b = fresh(shape, w), fresh(shape, w, 2)
        ea = a.prefill(prompt, tau)["exit_layer"]
        eb = b.prefill(prompt, tau)["exit_layer"]
        assert np.array_equal(eb, np.minimum(ea, 2)), (tau, ea, eb)
        a.close()
        b.close()


def test_cap_errors(tiny):
    shape, w = tiny
    L = shape.n_layers
    m = oracle.Model(shape, w, 1, 16)
    assert m.set_exit_cap(2) == RV_ESTATE  # no river yet
    assert m.quantize_river(64, 1) == 0
    assert m.set_exit_cap(0) == RV_EINVAL
    assert m.set_exit_cap(L + 1) == RV_EINVAL
    assert m.set_exit_cap(2) == RV_OK
    prompt = synth.make_prompt(shape.vocab, 1, 8, seed=8)
    with pytest.raises(RuntimeError):
        m.prefill(prompt, 0.9, fixed_exit=3)
    m.prefill(prompt, 0.9, fixed_exit=2)
    assert m.decode_step([5], 0.9, forced=np.array([3], dtype=np.int32))["rc"] == RV_EINVAL
    assert m.decode_step([5], 0.9, forced=np.array([2], dtype=np.int32))["rc"] == RV_OK
    m.close()
