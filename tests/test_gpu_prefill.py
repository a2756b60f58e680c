"""Prefill with the sequence-level exit against the oracle's own prefill, at
prompt lengths the oracle can replay (the 1B shape at 128 tokens, the 8B
shape at 32):

- per layer, the GPU's minimum over the prompt of s_t(l) (the quantity the
  sequence exit tests against tau) must match the oracle's, and the exit
  layer must be the oracle's (the oracle is teacher-forced only inside the
  tie band |s - tau| <= 1e-3);
- layer by layer at the last position (the stated tolerances): the oracle's
  layer l, fed the GPU's hidden state after layer l - 1 and the GPU's cache
  of the other positions, must give the GPU's hidden state within relative
  L2 1e-2, and the oracle's LM head on the GPU's final state its logits
  within 5e-2 (ids equal unless the top two are within 1e-2);
- free running (the oracle's whole prefill): logged, and held to drift
  bounds, since two correct 16-bit pipelines drift apart by rounding noise
  layer after layer (measured: 1B/128 tokens hidden 1.1e-2, logits 0.046;
  8B/32 tokens hidden 2.8e-2, logits 0.153).

A cosine moves by at most twice the relative error of its two vectors
(first order), so |delta s_min| <= 2 x 1e-2 follows from the per-layer
hidden tolerance."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import DRIFT_HIDDEN, TIE_LOGIT, TIE_S, TOL_HIDDEN, TOL_LOGIT, check_ids, log, rel_l2

# free-running logits after a whole prefill: the decode tests' 0.15 bound,
# raised to the 8B prefill's measured drift (0.153 at 32 tokens) with margin
PREFILL_DRIFT_LOGIT = 0.2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T0", [("llama1b", 128), ("llama8b", 32)])
def test_prefill_sequence_exit_against_oracle(name, T0):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    L = shape.n_layers
    w = synth.make_weights(shape)
    prompt = synth.make_prompt(shape.vocab, 1, T0, seed=13)
    gm = rv.Model(shape, w, 1, T0 + 4)
    gm.quantize_river(wl.group, 1)
    gm.set_debug(True)
    g_next, g_exit = gm.prefill(prompt, wl.prefill_tau)
    s_gpu = gm.dump(rv.DUMP_S)[:, 0].astype(np.float64)
    h_gpu = gm.dump(rv.DUMP_HIDDEN)[:, 0].astype(np.float64)
    l_gpu = gm.dump(rv.DUMP_LOGITS)[0].astype(np.float64)
    kv = gm.dump(rv.DUMP_KV)
    gm.close()

    om = oracle.Model(shape, w, 1, T0 + 4)
    om.quantize_river(wl.group, 1)
    o = om.prefill(prompt, wl.prefill_tau, tf_exit=g_exit, tf_ids=g_next, debug=True)
    om.close()

    e = int(g_exit[0])
    assert int(o["exit_layer"][0]) == e
    worst_s = 0.0
    for l in range(1, L + 1):
        sg, so = s_gpu[l - 1], o["smin"][l - 1, 0]
        if l <= e and l <= L - 1:  # layers whose s_min the rule looked at
            assert np.isfinite(sg) and np.isfinite(so), (l, sg, so)
            worst_s = max(worst_s, abs(sg - so))
            assert abs(sg - so) <= 2 * TOL_HIDDEN, (l, sg, so)
            # the rule: no exit before e, exit at e (ties may go either way)
            if l < e:
                assert sg <= wl.prefill_tau or abs(sg - wl.prefill_tau) <= TIE_S
    if e < L:
        assert s_gpu[e - 1] > wl.prefill_tau or abs(s_gpu[e - 1] - wl.prefill_tau) <= TIE_S
    # layer by layer at the last position, from the GPU's own state
    ol = oracle.Model(shape, w, 1, T0 + 4)
    ol.quantize_river(wl.group, 1)
    ol.set_kv(kv, np.array([T0 - 1], dtype=np.int32))
    worst_l = 0.0
    for l in range(1, L + 1):
        out = ol.layer_forward(l, h_gpu[l - 1][None], [1 if l > e else 0])
        r = rel_l2(h_gpu[l], out[0])
        worst_l = max(worst_l, r)
        assert r <= TOL_HIDDEN, (l, r)
    hl, _ = ol.head(h_gpu[L][None])
    ol.close()
    err_l = float(np.abs(l_gpu - hl[0]).max())
    assert err_l <= TOL_LOGIT, err_l
    check_ids(g_next, hl, TIE_LOGIT)

    # free running
    rels = [rel_l2(h_gpu[l], o["hidden_last"][l, 0]) for l in range(L + 1)]
    err = float(np.abs(l_gpu - o["logits"][0]).max())
    log({"tag": f"prefill:{name}:{T0}", "exit": e, "smin_worst_abs": worst_s, "layer_worst_rel": worst_l,
         "head_logit_err": err_l, "free_hidden_rel": rels, "free_logit_err": err})
    assert max(rels) <= DRIFT_HIDDEN, rels
    assert err <= PREFILL_DRIFT_LOGIT, err
    check_ids(g_next, o["logits"], max(TIE_LOGIT, 2 * err))
