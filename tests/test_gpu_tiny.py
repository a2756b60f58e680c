"""GPU parity on the tiny decoder (4 layers, d 256, fp16): the whole workload
(32-token prompt, 32 greedy decode steps, tau 0.90) and edge cases, through
the C ABI, against the CPU oracle element by element."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import check_free, check_layerwise, rel_l2, kv_values
from ongrid import ongrid_weights

pytestmark = pytest.mark.gpu
TINY = synth.TINY
WL = synth.WORKLOADS["tiny"]


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(TINY)


def pair(weights, B=1, T=96, group=64, entry=1):
    gm = rv.Model(TINY, weights, B, T)
    om = oracle.Model(TINY, weights, B, T)
    gm.quantize_river(group, entry)
    om.quantize_river(group, entry)
    gm.set_debug(True)
    return gm, om


def layer_oracle(weights, B, T, group=64, entry=1):
    ot = oracle.Model(TINY, weights, B, T)
    ot.quantize_river(group, entry)
    return ot


def step_both(gm, om, ot, toks, tau, forced, B, entry=1):
    """GPU step; free-running oracle om; layer-by-layer oracle ot."""
    kv_pre = gm.dump(rv.DUMP_KV)
    lens_pre = gm.dump(rv.DUMP_LENS).copy()
    g_next, g_exit = gm.decode_step(toks, tau, forced)
    o = om.decode_step(toks, tau, forced=forced, tf_exit=g_exit, tf_ids=g_next, debug=True)
    assert o["rc"] == 0
    check_free(gm, o, g_next, g_exit, B, TINY.n_layers)
    check_layerwise(gm, ot, kv_pre, lens_pre, g_next, g_exit, B, TINY.n_layers, TINY.act_dtype, tau, forced, entry)
    return g_next, g_exit


def check_kv(g_kv, o_kv, lens, act, tol=1e-2):
    """Slot pattern bit-exact (sentinel), values within the drift tolerance."""
    assert np.array_equal(g_kv == 0x7FFF, o_kv == 0x7FFF), "KV slot pattern differs"
    for b, n in enumerate(lens):
        gv = kv_values(g_kv[:, :, b, :, :n], act)
        ov = kv_values(o_kv[:, :, b, :, :n], act)
        for l in range(gv.shape[0]):
            assert rel_l2(gv[l], ov[l]) <= tol, (b, l)


def test_river_bit_exact(weights):
    gm, om = pair(weights)
    for layer in range(1, TINY.n_layers + 1):
        for proj in range(7):
            gq, gs, gz = gm.export_river(layer, proj)
            oq, os_, oz = om.export_river(layer, proj)
            assert np.array_equal(gq, oq), (layer, proj)
            assert np.array_equal(gs, os_), (layer, proj)
            assert np.array_equal(gz, oz), (layer, proj)
    gm.close()


def test_tiny_workload_parity(weights):
    """Config: 32-token prompt, 32 greedy decode steps, tau = 0.90."""
    gm, om = pair(weights, T=WL.prompt_len + WL.steps)
    ot = layer_oracle(weights, 1, WL.prompt_len + WL.steps)
    prompt = synth.make_prompt(TINY.vocab, 1, WL.prompt_len)
    tau = WL.taus[0]
    g_next, g_exit = gm.prefill(prompt, tau)
    o = om.prefill(prompt, tau, tf_exit=g_exit, tf_ids=g_next, debug=True)
    assert o["exit_layer"][0] == g_exit[0] and o["next_ids"][0] == g_next[0]
    assert np.abs(gm.dump(rv.DUMP_LOGITS)[0] - o["logits"][0]).max() <= 5e-2
    tok = int(g_next[0])
    exits = []
    for step in range(WL.steps):
        g_next, g_exit = step_both(gm, om, ot, [tok], tau, None, 1)
        exits.append(int(g_exit[0]))
        tok = int(g_next[0])
    check_kv(gm.dump(rv.DUMP_KV), om.get_kv(), [WL.prompt_len + WL.steps], TINY.act_dtype)
    assert list(gm.dump(rv.DUMP_LENS)) == [WL.prompt_len + WL.steps]
    gm.close()


def test_tiny_forced_exits_every_layer(weights):
    gm, om = pair(weights, T=40)
    ot = layer_oracle(weights, 1, 40)
    prompt = synth.make_prompt(TINY.vocab, 1, 8, seed=3)
    g_next, _ = gm.prefill(prompt, 0.9, fixed_exit=2)
    o = om.prefill(prompt, 0.9, fixed_exit=2, tf_ids=g_next)
    assert o["next_ids"][0] == g_next[0]
    tok = 5
    for step in range(15):
        f = np.array([step % (TINY.n_layers + 1)], dtype=np.int32)
        g_next, g_exit = step_both(gm, om, ot, [tok], 0.9, f, 1)
        assert g_exit[0] == f[0]
        tok = int(g_next[0])
    check_kv(gm.dump(rv.DUMP_KV), om.get_kv(), [23], TINY.act_dtype)
    gm.close()


def test_tiny_batched_rows_mixed_paths(weights):
    """B = 3 rows exit at different layers in the same step (general path)."""
    B = 3
    gm, om = pair(weights, B=B, T=40)
    ot = layer_oracle(weights, B, 40)
    prompts = synth.make_prompt(TINY.vocab, B, 6, seed=4)
    g_next, g_exit = gm.prefill(prompts, 0.9, fixed_exit=1)
    o = om.prefill(prompts, 0.9, fixed_exit=1, tf_ids=g_next)
    assert np.array_equal(o["next_ids"], g_next) and np.array_equal(o["exit_layer"], g_exit)
    toks = list(g_next)
    for step in range(8):
        f = np.array([(step + 2 * b) % (TINY.n_layers + 1) for b in range(B)], dtype=np.int32)
        g_next, g_exit = step_both(gm, om, ot, toks, 0.9, f, B)
        toks = list(g_next)
    # tau rule on the batched path
    for step in range(4):
        g_next, g_exit = step_both(gm, om, ot, toks, 0.5, None, B)
        toks = list(g_next)
    check_kv(gm.dump(rv.DUMP_KV), om.get_kv(), [18] * B, TINY.act_dtype)
    gm.close()


@pytest.mark.parametrize("group", [32, 256])
def test_tiny_batched_rows_other_groups(weights, group):
    """Batched river rows on the tensor pipe with group sizes the workloads do
    not use: 32 (sixteen groups per 512-code chunk) and 256 (one group per
    chunk of the 256-wide rows; the 688-wide down projection ends in a ragged
    group).  Forced exits mix both paths in every step; every step is checked
    layer by layer against the oracle."""
    B = 3
    gm, om = pair(weights, B=B, T=32, group=group)
    ot = layer_oracle(weights, B, 32, group=group)
    prompts = synth.make_prompt(TINY.vocab, B, 5, seed=8)
    g_next, g_exit = gm.prefill(prompts, 0.9, fixed_exit=2)
    o = om.prefill(prompts, 0.9, fixed_exit=2, tf_ids=g_next)
    assert np.array_equal(o["next_ids"], g_next)
    toks = list(g_next)
    for step in range(6):
        f = np.array([(step + b) % (TINY.n_layers + 1) for b in range(B)], dtype=np.int32)
        g_next, g_exit = step_both(gm, om, ot, toks, 0.9, f, B)
        toks = list(g_next)
    gm.close()


def test_tiny_prefill_tau_rule_batched(weights):
    B = 2
    gm, om = pair(weights, B=B, T=24)
    prompts = synth.make_prompt(TINY.vocab, B, 12, seed=5)
    for tau in (0.0, 0.3, 0.6, 0.9, 2.0):
        gm.kv_reset()
        om.kv_reset()
        g_next, g_exit = gm.prefill(prompts, tau)
        o = om.prefill(prompts, tau, tf_exit=g_exit, tf_ids=g_next, debug=True)
        assert np.array_equal(o["exit_layer"], g_exit), (tau, o["exit_layer"], g_exit)
        assert np.array_equal(o["next_ids"], g_next)
        assert np.abs(gm.dump(rv.DUMP_LOGITS)[:B] - o["logits"]).max() <= 5e-2
        hid = gm.dump(rv.DUMP_HIDDEN)[:, :B]
        for l in range(TINY.n_layers + 1):
            for b in range(B):
                assert rel_l2(hid[l, b], o["hidden_last"][l, b]) <= 1e-2
        check_kv(gm.dump(rv.DUMP_KV), om.get_kv(), [12] * B, TINY.act_dtype)
    gm.close()


def test_ongrid_river_matches_backbone_on_gpu():
    """On-grid weights: the int4 river equals the backbone, so the all-river
    and all-backbone GPU paths give the same logits up to fp32 rounding.  The
    two paths sum the same products in different orders (the int4 path folds
    the zero point per run), so a 16-bit activation occasionally rounds the
    other way (fp16 half-ulp 2^-11 relative), which moves the logits by about
    1e-3; a wrong weight (one int4 step is 1/15 of a group's range) moves them
    by orders of magnitude more.  Bound: 5e-3."""
    ws, _ = ongrid_weights(TINY, 64, seed=4)
    gm = rv.Model(TINY, ws, 1, 16)
    gm.quantize_river(64)
    gm.set_debug(True)
    prompt = synth.make_prompt(TINY.vocab, 1, 10, seed=11)
    out = []
    for e in (0, TINY.n_layers):
        gm.kv_reset()
        gm.prefill(prompt, 2.0, fixed_exit=e)
        gm.decode_step([5], 2.0, np.array([e], dtype=np.int32))
        out.append(gm.dump(rv.DUMP_LOGITS)[0].copy())
    assert np.abs(out[0] - out[1]).max() < 5e-3
    gm.close()


def test_capacity_and_errors(weights):
    gm = rv.Model(TINY, weights, 1, 4)
    with pytest.raises(rv.RVError) as e:
        gm.decode_step([1], 0.9)  # tau rule before the river exists
    assert e.value.code == rv.RV_ESTATE
    gm.quantize_river(64)
    with pytest.raises(rv.RVError) as e:
        gm.decode_step([TINY.vocab], 0.9)
    assert e.value.code == rv.RV_EINVAL
    with pytest.raises(rv.RVError) as e:
        gm.decode_step([1], 0.9, np.array([TINY.n_layers + 1], dtype=np.int32))
    assert e.value.code == rv.RV_EINVAL
    for _ in range(4):
        gm.decode_step([1], 0.9)
    kv = gm.dump(rv.DUMP_KV)
    with pytest.raises(rv.RVError) as e:
        gm.decode_step([1], 0.9)
    assert e.value.code == rv.RV_ECAPACITY
    assert np.array_equal(kv, gm.dump(rv.DUMP_KV))
    gm.kv_reset()
    assert (gm.dump(rv.DUMP_KV) == 0x7FFF).all()
    gm.decode_step([1], 0.9)
    with pytest.raises(rv.RVError) as e:
        gm.quantize_river(48)
    assert e.value.code == rv.RV_EINVAL
    gm.close()


def test_device_pointer_variant(weights):
    import torch

    gm, om = pair(weights, T=16)
    gm2 = rv.Model(TINY, weights, 1, 16)
    gm2.quantize_river(64)
    toks = [3, 9, 27, 81]
    d_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_next = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_exit = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_forced = torch.tensor([2], dtype=torch.int32, device="cuda")
    for t in toks:
        d_tok.fill_(t)
        torch.cuda.synchronize()
        gm2.decode_step_dev(d_tok.data_ptr(), 1, 0.9, d_forced.data_ptr(), d_next.data_ptr(), d_exit.data_ptr())
        gm2.sync_status()
        h_next, h_exit = gm.decode_step([t], 0.9, np.array([2], dtype=np.int32))
        assert int(d_next.item()) == h_next[0] and int(d_exit.item()) == h_exit[0] == 2
    d_forced.fill_(99)
    torch.cuda.synchronize()
    gm2.decode_step_dev(d_tok.data_ptr(), 1, 0.9, d_forced.data_ptr(), d_next.data_ptr(), d_exit.data_ptr())
    with pytest.raises(rv.RVError):
        gm2.sync_status()
    gm.close()
    gm2.close()


@pytest.mark.parametrize("name", ["tiny", "llama1b"])
def test_decode_engines_agree(name):
    """The persistent kernel and the per-kernel chain compute the same step
    (attention split counts differ, so agreement is within tolerance)."""
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    w = synth.make_weights(shape) if name != "tiny" else synth.make_weights(TINY)
    prompt = synth.make_prompt(shape.vocab, 1, 16, seed=8)
    out = []
    for engine in (rv.ENGINE_PERSISTENT, rv.ENGINE_CHAIN):
        gm = rv.Model(shape, w, 1, 40)
        gm.quantize_river(wl.group, 1)
        gm.set_engine(engine)
        gm.set_debug(True)
        gm.prefill(prompt, 2.0, fixed_exit=shape.n_layers)
        rec = []
        tok = 7
        for step in range(6):
            f = np.array([(0, 2, shape.n_layers, 1, 3, 0)[step]], dtype=np.int32)
            nxt, ex = gm.decode_step([tok], 0.9, f)
            rec.append((int(nxt[0]), int(ex[0]), gm.dump(rv.DUMP_LOGITS)[0].copy(),
                        gm.dump(rv.DUMP_HIDDEN)[:, 0].copy()))
            tok = 5 + step
        out.append(rec)
        gm.close()
    for (n1, e1, l1, h1), (n2, e2, l2, h2) in zip(*out):
        assert e1 == e2
        assert np.abs(l1 - l2).max() <= 5e-2
        for l in range(h1.shape[0]):
            assert rel_l2(h1[l], h2[l]) <= 1e-2
        if n1 != n2:
            srt = np.sort(l2)[::-1]
            assert srt[0] - srt[1] < 1e-2
