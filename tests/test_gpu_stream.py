"""The persistent decode engine on the tiny decoder, step by step against the
CPU oracle: every step of a tau-rule and a forced-exit run is compared layer
by layer and free-running (hidden states, s(l), logits, exit layers, ids and
the new K/V slots), including the all-river (e = 0) and full-backbone
(e = L) modes and a change of engine in the middle of a sequence."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import sampled_step

pytestmark = pytest.mark.gpu
TINY = synth.TINY


@pytest.mark.parametrize("mode", ["tau", "forced", "edges"])
def test_stream_tiny_every_step(mode):
    w = synth.make_weights(TINY)
    L = TINY.n_layers
    T = 32 + 24
    gm = rv.Model(TINY, w, 1, T)
    om = oracle.Model(TINY, w, 1, T)
    gm.quantize_river(64, 1)
    om.quantize_river(64, 1)
    gm.set_debug(True)
    gm.set_engine(rv.ENGINE_PERSISTENT)
    prompt = synth.make_prompt(TINY.vocab, 1, 32)
    g_next, g_exit = gm.prefill(prompt, 0.9)
    om.prefill(prompt, 0.9, tf_exit=g_exit, tf_ids=g_next)
    tok = [int(g_next[0])]
    for step in range(24):
        forced = None
        tau = (0.9, 0.3, 0.6)[step % 3]
        if mode == "forced":
            forced = synth.forced_exits(step, 1, L)
        elif mode == "edges":
            forced = np.array([(0, L, 1, L - 1)[step % 4]], dtype=np.int32)
        if step == 12:  # the chain continues the same sequence, then back
            gm.set_engine(rv.ENGINE_CHAIN)
        if step == 16:
            gm.set_engine(rv.ENGINE_PERSISTENT)
        nxt, ex = sampled_step(gm, om, tok, tau, forced, 1, L, TINY.act_dtype, 1, f"stream-tiny:{mode}:{step}")
        if forced is not None:
            assert int(ex[0]) == int(forced[0])
        tok = [int(nxt[0])]
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, 0, :, :T] == 0x7FFF).any()
    gm.close()
    om.close()
