"""GPU parity with backbone offloading (paperlayer.ai section 4, Backbone
Offloading): after rv_offload_backbone(k) only backbone layers 1..k stay on
the device and every exit is capped at k.  Checked against the oracle with
the same cap, layer by layer, on both decode engines and in prefill; the
resident parameter bytes follow the shape."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import log, sampled_step

pytestmark = pytest.mark.gpu


def resident_bytes(shape, keep):
    """16-bit parameters left on the device: embedding, LM head, final norm,
    every layer's two norms, backbone matrices of layers 1..keep."""
    d, F, L = shape.d_model, shape.ffn, shape.n_layers
    qkv = (shape.n_heads + 2 * shape.n_kv_heads) * shape.head_dim
    qd = shape.n_heads * shape.head_dim
    t = 2 * (shape.vocab * d * (1 if shape.tied_embed else 2) + d)
    t += L * 2 * 2 * d
    t += keep * 2 * (qkv * d + d * qd + 2 * F * d + d * F)
    return t


@pytest.mark.parametrize("name,keep", [("tiny", 2), ("llama1b", 3)])
def test_offloaded_backbone_decode(name, keep):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    L = shape.n_layers
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 1, 96)
    om = oracle.Model(shape, w, 1, 96)
    gm.quantize_river(wl.group, 1)
    om.quantize_river(wl.group, 1)
    full_bb, river_b = gm.param_bytes(0), gm.param_bytes(1)
    assert full_bb == resident_bytes(shape, L)
    gm.set_debug(True)
    prompt = synth.make_prompt(shape.vocab, 1, 32, seed=11)
    g_next, g_exit = gm.prefill(prompt, 0.9, fixed_exit=keep)
    om.prefill(prompt, 0.9, fixed_exit=keep, tf_ids=g_next)

    gm.offload_backbone(keep)
    assert om.set_exit_cap(keep) == 0
    assert gm.param_bytes(0) == resident_bytes(shape, keep) < full_bb
    assert gm.param_bytes(1) == river_b
    log({"tag": f"offload:{name}", "keep": keep, "resident_bytes": gm.param_bytes(0), "full_bytes": full_bb,
         "river_bytes": river_b})

    tok = [int(g_next[0])]
    exits = []
    for step in range(6):
        if step == 3:
            gm.set_engine(rv.ENGINE_PERSISTENT)
        tau = (0.9, 0.2, 2.0)[step % 3]
        nxt, ex = sampled_step(gm, om, tok, tau, None, 1, L, shape.act_dtype, 1, f"offload:{name}:{step}", cap=keep)
        assert int(ex[0]) <= keep
        exits.append(int(ex[0]))
        tok = [int(nxt[0])]
    gm.set_engine(rv.ENGINE_CHAIN)
    assert keep in exits  # tau 2.0 never exits on its own: the cap sends the row into the river

    # forced and fixed exits above the cap are rejected; the freed layers cannot come back
    with pytest.raises(rv.RVError):
        gm.decode_step(tok, 0.9, np.array([keep + 1], dtype=np.int32))
    with pytest.raises(rv.RVError):
        gm.offload_backbone(keep + 1)
    kv = gm.dump(rv.DUMP_KV)
    lens = gm.dump(rv.DUMP_LENS)
    assert not (kv[:, :, 0, :, : int(lens[0])] == 0x7FFF).any()  # every layer's slot filled
    gm.close()
    om.close()


def test_offloaded_prefill_rows():
    """Prefill after offloading: the rows path caps the sequence exit and never
    touches the freed matrices (tau 2.0: no exit on its own)."""
    shape = synth.TINY
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 2, 64)
    om = oracle.Model(shape, w, 2, 64)
    gm.quantize_river(64, 1)
    om.quantize_river(64, 1)
    gm.offload_backbone(2)
    om.set_exit_cap(2)
    prompt = synth.make_prompt(shape.vocab, 2, 24, seed=12)
    g_next, g_exit = gm.prefill(prompt, 2.0)
    o = om.prefill(prompt, 2.0, tf_exit=g_exit, tf_ids=g_next)
    assert np.array_equal(g_exit, [2, 2]) and np.array_equal(o["exit_layer"], g_exit)
    assert np.array_equal(o["next_ids"], g_next)
    with pytest.raises(rv.RVError):
        gm.prefill(prompt, 0.9, fixed_exit=3)
    gm.close()
    om.close()
