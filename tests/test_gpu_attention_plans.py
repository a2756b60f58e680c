"""Decode attention across its two launch plans.

Short contexts run the clustered kernel: each warp of a split holds at most
one 32-position tile, i.e. up to 16 x 4 x 32 = 2048 positions with clusters
of 16 splits.  Longer contexts run about one block per SM per row, whose
splits merge through global memory.  A decode that starts just below that
bound and runs past it must match the oracle layer by layer at every step, on
both sides of the switch.  The long plan's splits outnumber the tiles here,
so some splits have no tile of their own and the last one holds only the
position being decoded; the last tile is ragged at most steps."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import check_layerwise

pytestmark = pytest.mark.gpu

T0 = 2040   # prompt length: decode positions 2040 .. 2055 straddle 2048
STEPS = 16


@pytest.mark.parametrize("name", ["tiny", "llama1b"])
def test_decode_across_attention_plans(name):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    L = shape.n_layers
    w = synth.make_weights(shape)
    T = T0 + STEPS + 8
    gm = rv.Model(shape, w, 1, T)
    gm.quantize_river(wl.group, 1)
    gm.set_debug(True)
    ot = oracle.Model(shape, w, 1, T)
    ot.quantize_river(wl.group, 1)
    prompt = synth.make_prompt(shape.vocab, 1, T0, seed=17)
    nxt, _ = gm.prefill(prompt, wl.prefill_tau)
    tok = int(nxt[0])
    for step in range(STEPS):
        kv_pre = gm.dump(rv.DUMP_KV)
        lens_pre = gm.dump(rv.DUMP_LENS).copy()
        forced = np.array([(0, L, 2, L // 2)[step % 4]], dtype=np.int32)
        g_next, g_exit = gm.decode_step([tok], 0.9, forced)
        check_layerwise(gm, ot, kv_pre, lens_pre, g_next, g_exit, 1, L, shape.act_dtype, None, forced, 1,
                        tag=f"plans:{name}:{int(lens_pre[0])}")
        tok = int(g_next[0])
    assert int(gm.dump(rv.DUMP_LENS)[0]) == T0 + STEPS
    gm.close()
    ot.close()
