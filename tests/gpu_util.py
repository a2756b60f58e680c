"""Helpers for the GPU parity tests: run a step on both sides and compare.

Tolerances (stated for the decode path): per-layer hidden states within
relative L2 error 1e-2, logits within max-abs 5e-2, exit layers and greedy ids
exact.  The oracle is teacher-forced to the GPU's exit decision where
|s - tau| <= 1e-3 and to the GPU's id where its own top-2 logit gap is below
1e-2; a forced id must still be within 1e-2 + 5e-2 of the oracle's maximum.
"""
import numpy as np

import token_level_early_gb300 as rv

TOL_HIDDEN = 1e-2
TOL_LOGIT = 5e-2
TOL_S = 2e-3


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def check_decode(gm, g_next, g_exit, o, B, L, check_hidden=True):
    """Compare one decode step (GPU debug dumps vs oracle debug outputs)."""
    assert np.array_equal(o["exit_layer"], g_exit), (o["exit_layer"], g_exit)
    logits = gm.dump(rv.DUMP_LOGITS)[:B].astype(np.float64)
    ol = o["logits"]
    err = np.abs(logits - ol).max()
    assert err <= TOL_LOGIT, f"logits max-abs {err}"
    for b in range(B):
        if o["next_ids"][b] != g_next[b]:
            raise AssertionError(f"row {b}: id {g_next[b]} vs oracle {o['next_ids'][b]}")
        # a teacher-forced id must be a near-maximum of the oracle's logits
        assert ol[b].max() - ol[b][g_next[b]] <= 1e-2 + TOL_LOGIT
    if check_hidden:
        hid = gm.dump(rv.DUMP_HIDDEN)[:, :B]
        for l in range(L + 1):
            for b in range(B):
                r = rel_l2(hid[l, b], o["hidden"][l, b])
                assert r <= TOL_HIDDEN, f"layer {l} row {b}: rel L2 {r}"
        s = gm.dump(rv.DUMP_S)[:, :B]
        os_ = o["s"]
        both = np.isfinite(s) & np.isfinite(os_)
        assert np.array_equal(np.isfinite(s), np.isfinite(os_)), (s, os_)
        if both.any():
            assert np.abs(s[both] - os_[both]).max() <= TOL_S
    return float(err)


def kv_values(kv_bits, act):
    if act == 1:
        return (kv_bits.astype(np.uint32) << 16).view(np.float32)
    return kv_bits.view(np.float16).astype(np.float32)


def check_kv(g_kv, o_kv, lens, act, tol=TOL_HIDDEN):
    """Slot indexing bit-exact (sentinel pattern), values within tolerance."""
    g_empty = g_kv == 0x7FFF
    o_empty = o_kv == 0x7FFF
    assert np.array_equal(g_empty, o_empty), "KV slot pattern differs"
    for b, n in enumerate(lens):
        gv = kv_values(g_kv[:, :, b, :, :n], act)
        ov = kv_values(o_kv[:, :, b, :, :n], act)
        for l in range(gv.shape[0]):
            r = rel_l2(gv[l], ov[l])
            assert r <= tol, f"row {b} layer {l + 1}: KV rel L2 {r}"
