"""Helpers for the GPU parity tests.

Two comparisons per checked decode step, both against the CPU oracle:

1. Layer by layer (the per-layer tolerance of the decode path): the oracle's
   layer l takes the GPU's h(l-1) and the GPU's KV cache and must reproduce
   the GPU's h(l) within relative L2 1e-2 (observed far below), on the path
   the GPU took; its new K/V slot likewise.  The oracle's LM head takes the
   GPU's h(L): logits within max-abs 5e-2 and greedy ids equal unless the
   oracle's top-2 gap is below 1e-2.  The GPU's s(l) must equal the cosine of
   its own dumped h(l-1), h(l), and its exit layer must follow its s(l) and
   tau (a decision inside |s - tau| <= 1e-3 may go either way).

2. Free running: the oracle runs the whole step from the same cache state,
   teacher-forced to the GPU's exit decisions (|s - tau| <= 1e-3) and ids (its
   own top-2 gap < 1e-2).  Intermediate 16-bit rounding makes two correct
   implementations drift apart by bf16 noise per layer: the first fp32-vs-fp64
   difference flips a few roundings, which moves later values by whole bf16
   steps.  The drift is reported and bounded by DRIFT_HIDDEN / DRIFT_LOGIT,
   and a GPU id that differs from the oracle's must lie within the observed
   logit error band of the oracle's maximum.
"""
import json
import os

import numpy as np

import token_level_early_gb300 as rv

TOL_HIDDEN = 1e-2
TOL_LOGIT = 5e-2
TIE_S = 1e-3
TIE_LOGIT = 1e-2
DRIFT_HIDDEN = 3e-2
DRIFT_LOGIT = 1.5e-1

_LOG = os.environ.get("RV_PARITY_LOG")


def log(rec):
    if _LOG:
        with open(_LOG, "a") as f:
            f.write(json.dumps(rec) + "\n")


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def cos64(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(a @ b / max(np.linalg.norm(a) * np.linalg.norm(b), 1e-8))


def kv_values(kv_bits, act):
    if act == 1:
        return (kv_bits.astype(np.uint32) << 16).view(np.float32)
    return kv_bits.view(np.float16).astype(np.float32)


def check_ids(g_next, ol, band):
    for b in range(len(g_next)):
        o_id = int(np.argmax(ol[b]))
        if o_id == int(g_next[b]):
            continue
        gap = ol[b][o_id] - np.partition(ol[b], -2)[-2]
        assert gap < band or ol[b][o_id] - ol[b][g_next[b]] <= band, \
            f"row {b}: id {g_next[b]} (oracle logit {ol[b][g_next[b]]:.5f}) vs oracle {o_id} ({ol[b][o_id]:.5f})"


def check_decisions(s_gpu, g_exit, tau, forced, entry, L, cap=None):
    """The GPU's exit layer follows its own s(l): first l in [entry, L-1]
    with s(l) > tau (decisions within the tie band may go either way); with
    backbone offloading (cap < L) a row still in the backbone exits at cap."""
    cap = L if cap is None else cap
    for b in range(len(g_exit)):
        e = int(g_exit[b])
        assert e <= cap, (b, e, cap)
        if forced is not None:
            assert e == min(int(forced[b]), cap)
            continue
        for l in range(1, e + 1):
            s = float(s_gpu[l - 1, b])
            assert np.isfinite(s), (b, l)
            if entry <= l <= L - 1 and l < e:
                assert s <= tau or abs(s - tau) <= TIE_S, (b, l, s, tau)
        if e < L and e < cap:
            s = float(s_gpu[e - 1, b])
            assert s > tau or abs(s - tau) <= TIE_S, (b, e, s, tau)
        for l in range(e + 1, L + 1):
            assert not np.isfinite(s_gpu[l - 1, b])  # river layers do not evaluate s


def check_layerwise(gm, om, kv_pre, lens_pre, g_next, g_exit, B, L, act, tau=None, forced=None, entry=1,
                    tag="", cap=None):
    """Layer-by-layer comparison from the GPU's own inputs (see module doc)."""
    hid = gm.dump(rv.DUMP_HIDDEN)[:, :B].astype(np.float64)
    s_gpu = gm.dump(rv.DUMP_S)[:, :B]
    logits = gm.dump(rv.DUMP_LOGITS)[:B].astype(np.float64)
    kv_post = gm.dump(rv.DUMP_KV)
    om.set_kv(kv_pre, lens_pre)
    worst = 0.0
    for l in range(1, L + 1):
        river = [1 if int(g_exit[b]) < l else 0 for b in range(B)]
        out = om.layer_forward(l, hid[l - 1], river)
        for b in range(B):
            r = rel_l2(hid[l, b], out[b])
            worst = max(worst, r)
            assert r <= TOL_HIDDEN, f"{tag} layer {l} row {b}: rel L2 {r}"
            if not river[b]:
                assert abs(float(s_gpu[l - 1, b]) - cos64(hid[l - 1, b], hid[l, b])) <= 1e-5
    o_kv = om.get_kv()
    kv_worst = 0.0
    for b in range(B):
        p = int(lens_pre[b])
        g = kv_post[:, :, b, :, p]
        o = o_kv[:, :, b, :, p]
        assert not (g == 0x7FFF).any(), "GPU left a KV slot of this step empty"
        for l in range(g.shape[0]):
            r = rel_l2(kv_values(g[l], act), kv_values(o[l], act))
            kv_worst = max(kv_worst, r)
            assert r <= TOL_HIDDEN, f"{tag} KV layer {l + 1} row {b}: rel L2 {r}"
        if p + 1 < kv_post.shape[4]:
            assert (kv_post[:, :, b, :, p + 1] == 0x7FFF).all(), "GPU wrote beyond the step's slot"
        assert np.array_equal(kv_post[:, :, b, :, :p], kv_pre[:, :, b, :, :p]), "GPU rewrote earlier slots"
    ol, _ = om.head(hid[L])
    err = float(np.abs(logits - ol).max())
    assert err <= TOL_LOGIT, f"{tag} head logits max-abs {err}"
    check_ids(g_next, ol, TIE_LOGIT)
    if tau is not None or forced is not None:
        check_decisions(s_gpu, g_exit, tau, forced, entry, L, cap)
    rec = {"tag": tag, "layer_worst_rel": worst, "kv_worst_rel": kv_worst, "head_logit_err": err}
    log(rec)
    return rec


def check_free(gm, o, g_next, g_exit, B, L, tag=""):
    """Free-running comparison (oracle ran the whole step; see module doc)."""
    assert np.array_equal(o["exit_layer"], g_exit), (o["exit_layer"], g_exit)
    logits = gm.dump(rv.DUMP_LOGITS)[:B].astype(np.float64)
    ol = o["logits"]
    err = float(np.abs(logits - ol).max())
    hid = gm.dump(rv.DUMP_HIDDEN)[:, :B]
    rels = [max(rel_l2(hid[l, b], o["hidden"][l, b]) for b in range(B)) for l in range(L + 1)]
    rec = {"tag": tag, "free_hidden_rel": rels, "free_logit_err": err}
    log(rec)
    assert max(rels) <= DRIFT_HIDDEN, f"{tag} free-running drift {max(rels)}"
    assert err <= DRIFT_LOGIT, f"{tag} free-running logits {err}"
    check_ids(g_next, ol, max(TIE_LOGIT, 2 * err))
    return rec


def sampled_step(gm, om, toks, tau, forced, B, L, act, entry=1, tag="", cap=None):
    """Run one GPU decode step and check it both ways from the GPU's state."""
    kv_pre = gm.dump(rv.DUMP_KV)
    lens_pre = gm.dump(rv.DUMP_LENS).copy()
    g_next, g_exit = gm.decode_step(toks, tau, forced)
    om.set_kv(kv_pre, lens_pre)
    o = om.decode_step(toks, tau, forced=forced, tf_exit=g_exit, tf_ids=g_next, debug=True)
    assert o["rc"] == 0
    check_free(gm, o, g_next, g_exit, B, L, tag)
    check_layerwise(gm, om, kv_pre, lens_pre, g_next, g_exit, B, L, act, tau, forced, entry, tag, cap)
    return g_next, g_exit
