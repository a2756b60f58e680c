"""GPU parity for the long-context workload: Llama-3.1-8B shape, batch 1, a
65536-token prompt prefilled with the sequence exit fixed at layer 20, then
256 greedy decode steps with tau 0.90.

The oracle cannot replay a 64K prefill, so every check starts from the GPU's
own cache (teacher forcing):
- prefill: a sampled prompt position p is recomputed by the oracle as a
  decode of token p over the GPU's K/V of positions < p, with the exit forced
  to 20; the K/V the GPU wrote at p must match in every layer (and at the
  last position the logits and the greedy id);
- decode: sampled steps run through the same layer-by-layer and free-running
  comparisons as the other full-size workloads.
The KV cache holds L x 2 x Hkv x hd x max_seq 16-bit values and building the
river adds nothing to it (the river writes the same slots)."""
import time

import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import TIE_LOGIT, DRIFT_LOGIT, check_ids, kv_values, log, rel_l2, sampled_step

pytestmark = pytest.mark.gpu


def check_prefill_position(gm, om, kv, prompt, p, fixed_exit, act, want_logits=None, g_next=None):
    """Oracle decode of prompt[p] at position p over the GPU's cache of
    positions < p; compares the K/V slot p of every layer."""
    lens = np.zeros(om.max_batch, dtype=np.int32)
    lens[0] = p
    om.set_kv(kv, lens)
    o = om.decode_step(prompt[:, p], 2.0, forced=np.array([fixed_exit], dtype=np.int32),
                       tf_ids=g_next, debug=want_logits is not None)
    assert o["rc"] == 0
    ok = om.get_kv()
    worst = 0.0
    for l in range(kv.shape[0]):
        a = kv_values(kv[l, :, 0, :, p], act)
        r = kv_values(ok[l, :, 0, :, p], act)
        e = rel_l2(a, r)
        worst = max(worst, e)
        assert e <= 3e-2, (p, l + 1, e)
    rec = {"tag": f"long64k:prefill:{p}", "kv_worst_rel": worst}
    if want_logits is not None:
        err = float(np.abs(want_logits - o["logits"]).max())
        assert err <= DRIFT_LOGIT
        check_ids(g_next, o["logits"], max(TIE_LOGIT, 2 * err))
        rec["logit_err"] = err
    log(rec)
    return worst


def test_long64k_prefill_and_decode():
    wl = synth.WORKLOADS["long64k"]
    shape = wl.shape
    L = shape.n_layers
    T0, steps = wl.prompt_len, wl.steps
    T = T0 + steps
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 1, T)
    kv_before = gm.kv_bytes()
    gm.quantize_river(wl.group, 1)
    # the one cache: L x 2 x Hkv x hd x T 16-bit values; the river allocates none
    assert gm.kv_bytes() == kv_before == L * 2 * shape.n_kv_heads * shape.head_dim * 2 * T
    gm.set_debug(True)
    prompt = synth.make_prompt(shape.vocab, 1, T0)

    t0 = time.time()
    g_next, g_exit = gm.prefill(prompt, wl.prefill_tau, fixed_exit=wl.fixed_prefill_exit)
    prefill_s = time.time() - t0
    assert int(g_exit[0]) == wl.fixed_prefill_exit
    logits = gm.dump(rv.DUMP_LOGITS)[:1].copy()
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, 0, :, :T0] == 0x7FFF).any()   # every layer's slot filled, backbone or river
    assert (kv[:, :, 0, :, T0:] == 0x7FFF).all()

    om = oracle.Model(shape, w, 1, T)
    om.quantize_river(wl.group, 1)
    for p in (4097, 40000):
        check_prefill_position(gm, om, kv, prompt, p, wl.fixed_prefill_exit, shape.act_dtype)
    check_prefill_position(gm, om, kv, prompt, T0 - 1, wl.fixed_prefill_exit, shape.act_dtype, logits, g_next)
    del kv

    tau = wl.taus[0]
    tok = [int(g_next[0])]
    exits = []
    for step in range(steps):
        if step in (0, steps - 1):
            nxt, ex = sampled_step(gm, om, tok, tau, None, 1, L, shape.act_dtype, 1, f"long64k:tau:{step}")
        else:
            nxt, ex = gm.decode_step(tok, tau)
        exits.append(int(ex[0]))
        tok = [int(nxt[0])]
    assert gm.dump(rv.DUMP_LENS)[0] == T
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, 0, :, :T] == 0x7FFF).any()
    log({"tag": "long64k:summary", "kv_bytes": int(kv_before), "prefill_s": prefill_s,
         "mean_exit_layer": float(np.mean(exits)), "exit_hist": np.bincount(exits, minlength=L + 1).tolist()})
    gm.close()
    om.close()
