"""Fidelity of River vs the full backbone (the pages' next-token match rate
and KL(backbone || river), paperlayer.ai section 5), measured on the GPU and
checked against the same measurement on two oracle models fed the same
token stream (the GPU backbone's greedy ids) and teacher-forced to the GPU
river model's exit decisions."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import log

pytestmark = pytest.mark.gpu


def kl(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    la = a - a.max()
    lb = b - b.max()
    la -= np.log(np.exp(la).sum())
    lb -= np.log(np.exp(lb).sum())
    return float(np.sum(np.exp(la) * (la - lb)))


def test_fidelity_matches_oracle():
    shape = synth.TINY
    L = shape.n_layers
    w = synth.make_weights(shape)
    prompt = synth.make_prompt(shape.vocab, 1, 16, seed=21)
    tau, steps = 0.3, 12   # low tau: the river model exits early and often
    gb, gr = rv.Model(shape, w, 1, 40), rv.Model(shape, w, 1, 40)
    ob, orr = oracle.Model(shape, w, 1, 40), oracle.Model(shape, w, 1, 40)
    for m in (gr, gb):
        m.quantize_river(64, 1)
        m.set_debug(True)
    for m in (orr, ob):
        m.quantize_river(64, 1)
    nb, _ = gb.prefill(prompt, tau, fixed_exit=L)
    nr, er = gr.prefill(prompt, tau)
    ob.prefill(prompt, tau, fixed_exit=L, tf_ids=nb)
    orr.prefill(prompt, tau, tf_exit=er, tf_ids=nr)
    full = np.array([L], dtype=np.int32)
    tok = int(nb[0])
    g_kl, o_kl, g_match, o_match, exits = [], [], 0, 0, []
    for _ in range(steps):
        ib, _ = gb.decode_step([tok], tau, full)
        lb = gb.dump(rv.DUMP_LOGITS)[0].astype(np.float64)
        ir, ex = gr.decode_step([tok], tau)
        lr = gr.dump(rv.DUMP_LOGITS)[0].astype(np.float64)
        o1 = ob.decode_step([tok], tau, forced=full, tf_ids=ib, debug=True)
        o2 = orr.decode_step([tok], tau, tf_exit=ex, tf_ids=ir, debug=True)
        assert o1["rc"] == 0 and o2["rc"] == 0
        assert int(o2["exit_layer"][0]) == int(ex[0])
        g_kl.append(kl(lb, lr))
        o_kl.append(kl(o1["logits"][0], o2["logits"][0]))
        g_match += int(ib[0] == ir[0])
        o_match += int(o1["next_ids"][0] == o2["next_ids"][0])
        exits.append(int(ex[0]))
        tok = int(ib[0])
    for a, b in zip(g_kl, o_kl):
        assert abs(a - b) <= 0.1 * b + 1e-4, (a, b)
    assert abs(g_match - o_match) <= 1
    assert min(exits) < L  # the river path is exercised
    log({"tag": "fidelity:tiny", "tau": tau, "gpu_match": g_match / steps, "oracle_match": o_match / steps,
         "gpu_kl_mean": float(np.mean(g_kl)), "oracle_kl_mean": float(np.mean(o_kl)), "exits": exits})
    for m in (gb, gr, ob, orr):
        m.close()
