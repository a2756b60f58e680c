"""Model-level pins for the oracle: a textbook Llama forward built from torch
library routines (float64), the KV-share invariant, prefill/decode
consistency, batch independence, the exit rules and the river special case.
CPU only; tiny decoder shapes."""
import dataclasses
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from ongrid import ongrid_weights

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TINY = synth.TINY


def r16(x: torch.Tensor) -> torch.Tensor:
    """Round float64 values to fp16 (numpy's direct double->half conversion)."""
    return torch.from_numpy(x.detach().numpy().astype(np.float16).astype(np.float64))


def dec(bits):
    return torch.from_numpy(np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64))


def torch_llama(shape, ws, tokens):
    """Textbook Llama forward over one sequence, float64, with the 16-bit
    rounding points of the method (inputs of every matrix product, K/V)."""
    L, d, H, Hkv, hd = shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim
    T = len(tokens)
    E = dec(ws[0])
    head = E if shape.tied_embed else dec(ws[2])
    h = E[torch.as_tensor(tokens, dtype=torch.long)]
    pos = torch.arange(T, dtype=torch.float64)
    inv = shape.rope_theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = pos[:, None] * inv[None]
    cos = torch.cat([torch.cos(ang)] * 2, -1)
    sin = torch.cat([torch.sin(ang)] * 2, -1)

    def rot(x):  # x [heads, T, hd]
        x1, x2 = x[..., : hd // 2], x[..., hd // 2:]
        return x * cos + torch.cat([-x2, x1], -1) * sin

    hidden = [h[-1].clone()]
    for l in range(L):
        w = [None if a is None else dec(a) for a in ws[3 + 9 * l: 12 + 9 * l]]
        ga, Wq, Wk, Wv, Wo, gm, Wg, Wu, Wd = w
        x = r16(F.rms_norm(h, (d,), ga, eps=shape.rms_eps))
        q = (x @ Wq.T).view(T, H, hd).transpose(0, 1)
        k = (x @ Wk.T).view(T, Hkv, hd).transpose(0, 1)
        v = (x @ Wv.T).view(T, Hkv, hd).transpose(0, 1)
        q, k, v = r16(rot(q)), r16(rot(k)), r16(v)
        o = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, enable_gqa=True)[0]
        o = r16(o.transpose(0, 1).reshape(T, H * hd))
        h = h + o @ Wo.T
        x = r16(F.rms_norm(h, (d,), gm, eps=shape.rms_eps))
        a = r16(F.silu(x @ Wg.T) * (x @ Wu.T))
        h = h + a @ Wd.T
        hidden.append(h[-1].clone())
    y = r16(F.rms_norm(h[-1], (d,), dec(ws[1]), eps=shape.rms_eps))
    return torch.stack(hidden).numpy(), (y @ head.T).numpy()


def random_gamma_weights(shape, seed):
    ws = synth.make_weights(shape, seed=seed)
    rng = np.random.default_rng(seed)
    for i, w in enumerate(ws):
        if w is not None and w.ndim == 1:
            ws[i] = rng.uniform(0.5, 1.5, w.shape).astype(np.float16).view(np.uint16)
    return ws


@pytest.fixture(scope="module")
def tiny_weights():
    return random_gamma_weights(TINY, 5)


def test_param_bytes_golden():
    """paperlayer.ai appendix A.3 and aitrends.kr: Llama 3.1 8B parameter memory 14.96 GB."""
    txt = open(os.path.join(ROOT, "tests", "golden", "param_memory_8b.txt")).read()
    vals = dict(line.split("=", 1) for line in txt.splitlines() if "=" in line and not line.startswith("#"))
    assert synth.LLAMA_8B.param_bytes() == int(vals["param_bytes"])
    assert f"{synth.LLAMA_8B.param_bytes() / 2 ** 30:.2f}" == vals["gib_rounded"].strip()


def test_backbone_prefill_matches_textbook_llama(tiny_weights):
    prompt = synth.make_prompt(TINY.vocab, 1, 20, seed=9)
    hid_ref, logits_ref = torch_llama(TINY, tiny_weights, prompt[0])
    m = oracle.Model(TINY, tiny_weights, 1, 32)
    out = m.prefill(prompt, tau=2.0, fixed_exit=TINY.n_layers, debug=True)
    assert out["exit_layer"][0] == TINY.n_layers
    np.testing.assert_allclose(out["hidden_last"][:, 0], hid_ref, rtol=0, atol=2e-4 * np.abs(hid_ref).max())
    np.testing.assert_allclose(out["logits"][0], logits_ref, rtol=0, atol=1e-3)
    assert out["next_ids"][0] == int(np.argmax(logits_ref))
    m.close()


def test_backbone_decode_matches_textbook_llama(tiny_weights):
    prompt = synth.make_prompt(TINY.vocab, 1, 12, seed=10)
    m = oracle.Model(TINY, tiny_weights, 1, 32)
    m.prefill(prompt, tau=2.0, fixed_exit=TINY.n_layers)
    toks = list(prompt[0])
    nxt = 77
    for _ in range(3):
        out = m.decode_step([nxt], tau=2.0, forced=[TINY.n_layers], debug=True)
        toks.append(nxt)
        hid_ref, logits_ref = torch_llama(TINY, tiny_weights, toks)
        np.testing.assert_allclose(out["hidden"][:, 0], hid_ref, rtol=0, atol=2e-4 * np.abs(hid_ref).max())
        np.testing.assert_allclose(out["logits"][0], logits_ref, rtol=0, atol=1e-3)
        nxt = int(out["next_ids"][0])
        assert out["exit_layer"][0] == TINY.n_layers
    assert m.lens()[0] == 15
    m.close()


def test_ongrid_river_equals_backbone():
    """With weights on the int4 grid the river copy is the backbone exactly,
    so all-river (exit 0) and all-backbone (exit L) decode agree bit for bit."""
    ws, _ = ongrid_weights(TINY, 64, seed=4)
    prompt = synth.make_prompt(TINY.vocab, 1, 10, seed=11)
    m = oracle.Model(TINY, ws, 1, 16)
    assert m.quantize_river(64) == 0
    res = []
    for e in (0, TINY.n_layers, 2):
        m.kv_reset()
        m.prefill(prompt, tau=2.0, fixed_exit=e)
        res.append((m.decode_step([5], 2.0, forced=[e], debug=True), m.get_kv()))
    for out, kv in res[1:]:
        assert np.array_equal(out["logits"], res[0][0]["logits"])
        assert np.array_equal(kv, res[0][1])
    m.close()


def test_river_differs_from_backbone_on_random_weights(tiny_weights):
    prompt = synth.make_prompt(TINY.vocab, 1, 10, seed=12)
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64)
    m.prefill(prompt, tau=2.0, fixed_exit=TINY.n_layers)
    a = m.decode_step([5], 2.0, forced=[TINY.n_layers], debug=True)["logits"]
    m.kv_reset()
    m.prefill(prompt, tau=2.0, fixed_exit=TINY.n_layers)
    b = m.decode_step([5], 2.0, forced=[0], debug=True)["logits"]
    diff = np.abs(a - b).max()
    assert 1e-4 < diff < 0.5 * np.abs(a).max()
    m.close()


def kv_check(m, shape, B):
    kv = m.get_kv()
    lens = m.lens()
    for b in range(B):
        filled = kv[:, :, b, :, : lens[b], :]
        empty = kv[:, :, b, :, lens[b]:, :]
        assert not np.any(filled == oracle.KV_SENTINEL), f"row {b}: missing KV below len"
        assert np.all(empty == oracle.KV_SENTINEL), f"row {b}: KV written beyond len"


def test_kv_share_invariant_every_layer_filled(tiny_weights):
    """KV Share: whichever path a token takes, every layer 1..L holds its K/V."""
    B = 3
    m = oracle.Model(TINY, tiny_weights, B, 24)
    m.quantize_river(64)
    prompt = synth.make_prompt(TINY.vocab, B, 6, seed=13)
    m.prefill(prompt, tau=2.0, fixed_exit=1)
    kv_check(m, TINY, B)
    toks = [1, 2, 3]
    for step in range(8):
        forced = [(step + b) % (TINY.n_layers + 1) for b in range(B)]
        out = m.decode_step(toks, 2.0, forced=forced)
        assert list(out["exit_layer"]) == forced
        toks = list(out["next_ids"])
        kv_check(m, TINY, B)
    assert list(m.lens()) == [14, 14, 14]
    m.close()


def test_prefill_then_decode_equals_longer_prefill(tiny_weights):
    m = oracle.Model(TINY, tiny_weights, 1, 32)
    m.quantize_river(64)
    prompt = synth.make_prompt(TINY.vocab, 1, 9, seed=14)
    for e in (0, 2, TINY.n_layers):
        m.kv_reset()
        m.prefill(prompt, tau=2.0, fixed_exit=e)
        d = m.decode_step([int(prompt[0, -1]) ^ 5], 2.0, forced=[e], debug=True)
        kv_a = m.get_kv()
        m.kv_reset()
        longer = np.concatenate([prompt, [[int(prompt[0, -1]) ^ 5]]], axis=1).astype(np.int32)
        p = m.prefill(longer, tau=2.0, fixed_exit=e, debug=True)
        assert np.array_equal(p["logits"], d["logits"])
        assert p["next_ids"][0] == d["next_ids"][0]
        assert np.array_equal(m.get_kv(), kv_a)
    m.close()


def test_batch_rows_are_independent(tiny_weights):
    B = 3
    prompts = synth.make_prompt(TINY.vocab, B, 7, seed=15)
    forced = [0, 2, 4]
    mb = oracle.Model(TINY, tiny_weights, B, 16)
    mb.quantize_river(64)
    mb.prefill(prompts, 2.0, fixed_exit=1)
    ob = mb.decode_step([3, 4, 5], 2.0, forced=forced, debug=True)
    for b in range(B):
        m1 = oracle.Model(TINY, tiny_weights, 1, 16)
        m1.quantize_river(64)
        m1.prefill(prompts[b:b + 1], 2.0, fixed_exit=1)
        o1 = m1.decode_step([3 + b], 2.0, forced=[forced[b]], debug=True)
        assert np.array_equal(o1["logits"][0], ob["logits"][b])
        assert o1["next_ids"][0] == ob["next_ids"][b]
        m1.close()
    mb.close()


def test_tau_rule_extremes(tiny_weights):
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64, entry_layer=1)
    out = m.decode_step([7], tau=2.0)  # s <= 1 < tau: never exits
    assert out["exit_layer"][0] == TINY.n_layers
    out = m.decode_step([7], tau=-2.0)  # s >= -1 > tau: exits at the entry layer
    assert out["exit_layer"][0] == 1
    m.quantize_river(64, entry_layer=3)
    out = m.decode_step([7], tau=-2.0)
    assert out["exit_layer"][0] == 3
    m.quantize_river(64, entry_layer=TINY.n_layers)  # no layer in [entry, L-1]
    out = m.decode_step([7], tau=-2.0)
    assert out["exit_layer"][0] == TINY.n_layers
    m.close()


def test_tau_rule_exits_at_first_layer_above_tau(tiny_weights):
    """Token-level rule: exit after the first layer l >= entry with s(l) > tau,
    strictly greater (aitrends.kr, state transition similarity)."""
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64)
    s = m.decode_step([9], 2.0, forced=[TINY.n_layers], debug=True)["s"][:, 0]
    for l in range(1, TINY.n_layers):
        # tau just below s(l) and above every earlier s: exit at l
        if all(s[j] < s[l - 1] for j in range(l - 1)):
            m.kv_reset()
            out = m.decode_step([9], float(s[l - 1]) - 1e-9)
            assert out["exit_layer"][0] == l
            m.kv_reset()
            out = m.decode_step([9], float(s[l - 1]))  # equal is not greater
            assert out["exit_layer"][0] != l
    m.close()


def test_sequence_exit_is_set_by_latest_token(tiny_weights):
    """Prefill rule: one exit layer for the sequence, the first l where every
    token's s(l) exceeds tau (paperlayer.ai section 3, Sequence-level Exit).
    Per-token similarities come from token-level decode steps on the backbone."""
    L = TINY.n_layers
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64)
    toks = [11, 600]
    m.kv_reset()
    s_tok = []
    for t in toks:
        s_tok.append(m.decode_step([t], 2.0, forced=[L], debug=True)["s"][:, 0])
    s_tok = np.array(s_tok)  # [token, layer]
    smin = s_tok.min(0)
    checked = 0
    for tau in np.unique(np.concatenate([s_tok.reshape(-1) - 1e-7, s_tok.reshape(-1) + 1e-7])):
        exp = next((l for l in range(1, L) if smin[l - 1] > tau), L)
        m.kv_reset()
        got = m.prefill(np.array([toks], dtype=np.int32), float(tau))["exit_layer"][0]
        assert got == exp, (tau, s_tok)
        checked += 1
    assert checked >= 4
    # tau equal to the minimum at a layer: equal is not greater, no exit there
    for l in range(1, L):
        m.kv_reset()
        got = m.prefill(np.array([toks], dtype=np.int32), float(smin[l - 1]))["exit_layer"][0]
        assert got != l or any(smin[j] > smin[l - 1] for j in range(l - 1))
    # a one-token prompt: the sequence rule reduces to the token rule
    for tau in s_tok[0] - 1e-7:
        m.kv_reset()
        e_pre = m.prefill(np.array([[toks[0]]], dtype=np.int32), float(tau))["exit_layer"][0]
        m.kv_reset()
        e_dec = m.decode_step([toks[0]], float(tau))["exit_layer"][0]
        assert e_pre == e_dec
    m.close()


def test_greedy_id_is_argmax_of_logits(tiny_weights):
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64)
    out = m.decode_step([3], 0.5, debug=True)
    assert out["next_ids"][0] == int(np.argmax(out["logits"][0]))
    m.close()


def test_errors_and_capacity(tiny_weights):
    m = oracle.Model(TINY, tiny_weights, 1, 3)
    assert m.decode_step([1], 0.9)["rc"] == oracle.RV_ESTATE  # tau rule needs the river
    assert m.decode_step([TINY.vocab], 2.0, forced=[TINY.n_layers])["rc"] == oracle.RV_EINVAL
    m.quantize_river(64)
    for _ in range(3):
        assert m.decode_step([1], 0.9)["rc"] == 0
    before = m.get_kv()
    assert m.decode_step([1], 0.9)["rc"] == oracle.RV_ECAPACITY
    assert np.array_equal(before, m.get_kv()) and m.lens()[0] == 3
    m.close()


def test_teacher_forcing_on_ties(tiny_weights):
    m = oracle.Model(TINY, tiny_weights, 1, 16)
    m.quantize_river(64)
    s = m.decode_step([9], 2.0, forced=[TINY.n_layers], debug=True)["s"][:, 0]
    tau = float(s[1]) - 5e-4  # within the 1e-3 tie band of s(2)
    m.kv_reset()
    free = m.decode_step([9], tau)
    m.kv_reset()
    other = 3 if free["exit_layer"][0] != 3 else 1
    tf = m.decode_step([9], tau, tf_exit=[other])
    # the oracle follows the given decision only inside the band
    assert tf["exit_layer"][0] in (other, free["exit_layer"][0])
    assert tf["n_forced"][0] >= (1 if tf["exit_layer"][0] != free["exit_layer"][0] else 0)
    m.close()


def test_layer_forward_and_head_compose_to_decode_step(tiny_weights):
    """Chaining the single-layer entry point over layers 1..L from the same
    cache state reproduces a decode step exactly, and the head reproduces its
    logits and greedy id."""
    B = 2
    m = oracle.Model(TINY, tiny_weights, B, 16)
    m.quantize_river(64)
    m.prefill(synth.make_prompt(TINY.vocab, B, 5, seed=21), 2.0, fixed_exit=1)
    kv, lens = m.get_kv(), m.lens()
    forced = [0, 2]
    ref = m.decode_step([7, 8], 2.0, forced=forced, debug=True)
    m.set_kv(kv, lens)
    h = ref["hidden"][0].copy()
    for l in range(1, TINY.n_layers + 1):
        river = [1 if forced[b] < l else 0 for b in range(B)]
        h = m.layer_forward(l, h, river)
        assert np.array_equal(h, ref["hidden"][l])
    logits, ids = m.head(h)
    assert np.array_equal(logits, ref["logits"]) and np.array_equal(ids, ref["next_ids"])
    assert list(m.lens()) == list(lens)  # positions not advanced
    m.close()


def test_thread_count_does_not_change_results():
    """The oracle's row loops split rows over host threads; every row is
    computed by one thread in a fixed order, so 1 and 4 threads agree bit
    for bit (the CPU-baseline timing relies on it)."""
    shape = synth.TINY
    w = synth.make_weights(shape)
    outs = []
    for nt in (1, 4):
        m = oracle.Model(shape, w, 2, 24, nthreads=4)
        assert m.set_threads(nt) == 0
        assert m.quantize_river(64, 1) == 0
        p = m.prefill(synth.make_prompt(shape.vocab, 2, 10, seed=9), 0.5, debug=True)
        d = m.decode_step(p["next_ids"], 0.5, debug=True)
        outs.append((p["logits"], d["logits"], d["hidden"], d["exit_layer"], m.get_kv()))
        assert m.set_threads(0) != 0
        m.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
