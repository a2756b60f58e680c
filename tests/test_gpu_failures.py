"""Failure handling without a GPU fault: a bounded device wait that runs out,
and a device allocation that fails.

1. The persistent decode kernel bounds every wait (grid barriers, weight-ring
   stages, route hand-offs).  With the wait limit set to a microsecond the
   waits run out on purpose: the step must come back with RV_ETIMEOUT, leave
   the cached positions where they were, and the next step (default limit)
   must compute what the other engine computes for the same token.
2. A device allocation made to fail (test hook) must surface as RV_ENOMEM
   from the call that made it, with nothing leaked on the device, and the
   library must keep working afterwards."""
import numpy as np
import pytest

import synth
import token_level_early_gb300 as rv
from gpu_util import rel_l2

pytestmark = pytest.mark.gpu
TINY = synth.TINY


def test_bounded_wait_times_out_cleanly():
    w = synth.make_weights(TINY)
    prompt = synth.make_prompt(TINY.vocab, 1, 12, seed=3)
    gm = rv.Model(TINY, w, 1, 32)
    twin = rv.Model(TINY, w, 1, 32)
    for m in (gm, twin):
        m.quantize_river(64, 1)
        m.set_debug(True)
        m.prefill(prompt, 2.0, fixed_exit=TINY.n_layers)
    gm.set_engine(rv.ENGINE_PERSISTENT)
    lens0 = gm.dump(rv.DUMP_LENS).copy()

    gm.set_option(rv.OPT_WAIT_LIMIT_US, 1)
    with pytest.raises(rv.RVError) as e:
        gm.decode_step([7], 0.9, np.array([2], dtype=np.int32))
    assert e.value.code == rv.RV_ETIMEOUT, e.value
    assert np.array_equal(gm.dump(rv.DUMP_LENS), lens0)  # the step did not happen

    gm.set_option(rv.OPT_WAIT_LIMIT_US, 0)
    for step, tok in enumerate((7, 9, 11)):
        f = np.array([(2, 0, TINY.n_layers)[step]], dtype=np.int32)
        n1, e1 = gm.decode_step([tok], 0.9, f)
        n2, e2 = twin.decode_step([tok], 0.9, f)
        assert int(e1[0]) == int(e2[0]) == int(f[0])
        l1, l2 = gm.dump(rv.DUMP_LOGITS)[0], twin.dump(rv.DUMP_LOGITS)[0]
        assert np.abs(l1 - l2).max() <= 5e-2
        h1, h2 = gm.dump(rv.DUMP_HIDDEN)[:, 0], twin.dump(rv.DUMP_HIDDEN)[:, 0]
        for l in range(h1.shape[0]):
            assert rel_l2(h1[l], h2[l]) <= 1e-2
    lens = gm.dump(rv.DUMP_LENS)
    assert int(lens[0]) == int(lens0[0]) + 3
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, 0, :, : int(lens[0])] == 0x7FFF).any()
    assert (kv[:, :, 0, :, int(lens[0]):] == 0x7FFF).all()
    gm.close()
    twin.close()


def test_injected_allocation_failure_returns_enomem_without_leak():
    import torch

    w = synth.make_weights(TINY)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for after in (0, 3, 9, 25):
            rv.debug_fail_alloc(after)
            with pytest.raises(rv.RVError) as e:
                rv.Model(TINY, w, 1, 64)
            assert e.value.code == rv.RV_ENOMEM, (after, e.value)
        rv.debug_fail_alloc(-1)
        free1 = torch.cuda.mem_get_info()[0]
        assert abs(free1 - free0) <= 8 << 20, (free0, free1)

        # a failed river build leaves the model usable: build again and decode
        gm = rv.Model(TINY, w, 1, 64)
        rv.debug_fail_alloc(5)
        with pytest.raises(rv.RVError) as e:
            gm.quantize_river(64, 1)
        assert e.value.code == rv.RV_ENOMEM
        rv.debug_fail_alloc(-1)
        gm.quantize_river(64, 1)
        nxt, ex = gm.decode_step([5], 0.9)
        assert 0 <= int(nxt[0]) < TINY.vocab and 1 <= int(ex[0]) <= TINY.n_layers
        gm.close()
    finally:
        rv.debug_fail_alloc(-1)
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) <= 8 << 20
