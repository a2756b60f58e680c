"""GPU parity at the full workload sizes (Llama-3.2-1B and Llama-3.1-8B
shapes, batch 1, and the batch-64 mixed-exit workload).  The oracle is too slow
to replay a whole workload, so each check starts from the GPU's own state:
before a sampled step the GPU's KV cache is copied into the oracle, both run
the same step, and the outputs are compared layer by layer and free-running
(per-layer hidden states, s(l), logits, exit layers, greedy ids, the new KV
slots).  The prefill's last position is checked the same way: a decode step
of the last prompt token over the GPU's cache of the others, with the
prefill's sequence exit layer forced."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import kv_values, rel_l2, sampled_step, check_ids, TIE_LOGIT, DRIFT_LOGIT

pytestmark = pytest.mark.gpu


def check_prefill_last_position(gm, om, prompt, g_next, g_exit, act):
    """Prefill's last position = decode of the last token over the cache of
    the others, with the sequence's exit layer forced."""
    B, T0 = prompt.shape
    kv = gm.dump(rv.DUMP_KV)
    logits = gm.dump(rv.DUMP_LOGITS)[:B].copy()
    lens = np.zeros(om.max_batch, dtype=np.int32)
    lens[:B] = T0 - 1
    om.set_kv(kv, lens)
    o = om.decode_step(prompt[:, -1], 2.0, forced=g_exit, tf_ids=g_next, debug=True)
    assert o["rc"] == 0
    err = np.abs(logits - o["logits"]).max()
    assert err <= DRIFT_LOGIT
    check_ids(g_next, o["logits"], max(TIE_LOGIT, 2 * err))
    ok = om.get_kv()
    for b in range(B):
        for l in range(kv.shape[0]):
            a = kv_values(kv[l, :, b, :, T0 - 1], act)
            r = kv_values(ok[l, :, b, :, T0 - 1], act)
            assert rel_l2(a, r) <= 3e-2


def run_single(name, sample_steps, mode, tau=None, engine=rv.ENGINE_CHAIN, steps=None):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    w = synth.make_weights(shape)
    n_steps = wl.steps if steps is None else steps
    T = wl.prompt_len + n_steps
    gm = rv.Model(shape, w, 1, T)
    om = oracle.Model(shape, w, 1, T)
    gm.quantize_river(wl.group, 1)
    om.quantize_river(wl.group, 1)
    # river bit-exact on the first and last layer
    for layer in (1, shape.n_layers):
        for proj in range(7):
            g = gm.export_river(layer, proj)
            o = om.export_river(layer, proj)
            for a, b in zip(g, o):
                assert np.array_equal(a, b), (layer, proj)
    gm.set_debug(True)
    gm.set_engine(engine)
    prompt = synth.make_prompt(shape.vocab, 1, wl.prompt_len)
    g_next, g_exit = gm.prefill(prompt, wl.prefill_tau)
    s_min = gm.dump(rv.DUMP_S)[:, 0]
    # the sequence exit is the first layer >= entry whose min similarity > tau
    exp = next((l for l in range(1, shape.n_layers) if s_min[l - 1] > wl.prefill_tau), shape.n_layers)
    assert g_exit[0] == exp, (g_exit, s_min)
    check_prefill_last_position(gm, om, prompt, g_next, g_exit, shape.act_dtype)
    tau = wl.taus[0] if tau is None else tau
    tok = [int(g_next[0])]
    exits = []
    for step in range(n_steps):
        forced = synth.forced_exits(step, 1, shape.n_layers) if mode == "forced" else None
        if step in sample_steps:
            nxt, ex = sampled_step(gm, om, tok, tau, forced, 1, shape.n_layers, shape.act_dtype, 1,
                                   f"{name}:{mode}:{tau}:{engine}:{step}")
        else:
            nxt, ex = gm.decode_step(tok, tau, forced)
        if forced is not None:
            assert ex[0] == forced[0]
        exits.append(int(ex[0]))
        tok = [int(nxt[0])]
    lens = gm.dump(rv.DUMP_LENS)
    assert lens[0] == T
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, 0, :, :T] == 0x7FFF).any()  # every layer's slot filled, whatever the path
    gm.close()
    om.close()
    return exits


@pytest.mark.parametrize("tau", synth.WORKLOADS["llama1b"].taus)
def test_llama1b_tau_rule_workload(tau):
    """The 1B workload's tau sweep: 0.85, 0.90 and 0.95."""
    exits = run_single("llama1b", {0, 1, 2, 17, 128, 255}, "tau", tau)
    assert len(exits) == 256


def test_llama1b_forced_exit_workload():
    exits = run_single("llama1b", {0, 3, 64, 200}, "forced")
    assert min(exits) >= 1


def test_llama8b_tau_rule_workload():
    run_single("llama8b", {0, 1, 100, 511}, "tau")


def test_llama8b_forced_exit_workload():
    run_single("llama8b", {0, 5, 300}, "forced")


def test_batch64_mixed_exits():
    """Config: 64 rows, 256-token prompts, per-row per-step forced exit layers:
    every layer of a step mixes bf16 backbone rows and int4 river rows that
    write the same cache."""
    wl = synth.WORKLOADS["batch64"]
    shape, B = wl.shape, wl.batch
    w = synth.make_weights(shape)
    T = wl.prompt_len + wl.steps
    gm = rv.Model(shape, w, B, T)
    om = oracle.Model(shape, w, B, T)
    gm.quantize_river(wl.group, 1)
    om.quantize_river(wl.group, 1)
    gm.set_debug(True)
    prompts = synth.make_prompt(shape.vocab, B, wl.prompt_len)
    g_next, g_exit = gm.prefill(prompts, wl.prefill_tau)
    s_min = gm.dump(rv.DUMP_S)[:, :B]
    for b in range(B):
        exp = next((l for l in range(1, shape.n_layers) if s_min[l - 1, b] > wl.prefill_tau), shape.n_layers)
        assert g_exit[b] == exp
    toks = g_next.copy()
    for step in range(wl.steps):
        forced = synth.forced_exits(step, B, shape.n_layers)
        if step in (0, 127):
            nxt, ex = sampled_step(gm, om, toks, 0.9, forced, B, shape.n_layers, shape.act_dtype, 1,
                                   f"batch64:{step}")
        else:
            nxt, ex = gm.decode_step(toks, 0.9, forced)
        assert np.array_equal(ex, forced)
        toks = nxt
    kv = gm.dump(rv.DUMP_KV)
    assert not (kv[:, :, :B, :, :T] == 0x7FFF).any()
    gm.close()
    om.close()


# The persistent decode engine (one cooperative launch per step, weights
# streamed through a shared-memory ring by a producer warp) on the same
# workloads, checked against the oracle the same way.

def test_stream_llama1b_tau_rule_workload():
    exits = run_single("llama1b", {0, 1, 2, 100, 255}, "tau", 0.90, rv.ENGINE_PERSISTENT)
    assert len(exits) == 256


def test_stream_llama1b_forced_exit_workload():
    exits = run_single("llama1b", {0, 3, 64}, "forced", None, rv.ENGINE_PERSISTENT, steps=128)
    assert min(exits) >= 1


def test_stream_llama8b_tau_rule_workload():
    run_single("llama8b", {0, 1, 100, 511}, "tau", None, rv.ENGINE_PERSISTENT)


def test_stream_llama8b_forced_exit_workload():
    run_single("llama8b", {0, 5, 300}, "forced", None, rv.ENGINE_PERSISTENT, steps=320)
