"""CPU oracle for the River-LLM decode path (ctypes binding of rv_oracle.c).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg load this package; the product path never does, and this
package imports nothing from the CUDA library.

Parity status of each oracle function is pinned by tests/test_oracle_*.py
against closed forms, invariants, brute force and textbook library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "librvoracle.so")
_SRC = os.path.join(_HERE, "rv_oracle.c")
_lib = None

RV_OK, RV_EINVAL, RV_ENOMEM, RV_ECUDA, RV_ECAPACITY, RV_ESTATE = 0, -1, -2, -3, -4, -5
KV_SENTINEL = 0x7FFF


def build(verbose: bool = False) -> str:
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", _LIB_PATH, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return _LIB_PATH


class OraConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("tied_embed", ctypes.c_int), ("act_dtype", ctypes.c_int),
                ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double),
                ("max_batch", ctypes.c_int), ("max_seq", ctypes.c_int)]


def lib():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        build()
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    sig = {
        "ora_create": ([ctypes.POINTER(OraConfig), vp, i32, ctypes.POINTER(vp)], i32),
        "ora_free": ([vp], None),
        "ora_quantize_river": ([vp, i32, i32], i32),
        "ora_set_exit_cap": ([vp, i32], i32),
        "ora_set_threads": ([vp, i32], i32),
        "ora_set_quantizer": ([vp, i32], i32),
        "ora_export_river": ([vp, i32, i32, vp, vp, vp], i32),
        "ora_prefill": ([vp, vp, i32, i32, dbl, i32, vp, vp, vp, vp, vp, vp, vp, vp], i32),
        "ora_decode_step": ([vp, vp, i32, dbl, vp, vp, vp, vp, vp, vp, vp, vp, vp], i32),
        "ora_kv_reset": ([vp, vp, i32], i32),
        "ora_layer_forward": ([vp, i32, i32, vp, vp, vp], i32),
        "ora_head": ([vp, i32, vp, vp, vp], i32),
        "ora_get_kv": ([vp, vp, ctypes.c_size_t], i32),
        "ora_set_kv": ([vp, vp, ctypes.c_size_t, vp], i32),
        "ora_get_lens": ([vp, vp], i32),
        "ora_kv_bytes": ([vp], ctypes.c_size_t),
        "ora_act16_round": ([dbl, i32], dbl),
        "ora_act16_encode": ([dbl, i32], ctypes.c_uint16),
        "ora_act16_decode": ([ctypes.c_uint16, i32], dbl),
        "ora_cosine": ([vp, vp, i32], dbl),
        "ora_rmsnorm": ([vp, vp, i32, dbl, i32, vp], None),
        "ora_rope": ([vp, i32, i32, dbl], None),
        "ora_attention": ([vp, vp, vp, i32, i32, i32, vp], None),
        "ora_argmax": ([vp, i32], i32),
        "ora_rtn_group": ([vp, i32, i32, vp, vp, vp], i32),
        "ora_hqq_group": ([vp, i32, i32, vp, vp, vp], i32),
        "ora_hqq_pow_pm1": ([ctypes.c_float], ctypes.c_float),
        "ora_silu": ([dbl], dbl),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------- primitives

def act16_round(x: float, act: int) -> float:
    return lib().ora_act16_round(float(x), act)


def act16_encode(x: float, act: int) -> int:
    return int(lib().ora_act16_encode(float(x), act))


def act16_decode(bits: int, act: int) -> float:
    return lib().ora_act16_decode(int(bits), act)


def cosine(a, b) -> float:
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    return lib().ora_cosine(_p(a), _p(b), a.size)


def rmsnorm(h, gamma_bits, eps: float, act: int) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.float64)
    g = np.ascontiguousarray(gamma_bits, dtype=np.uint16)
    out = np.empty_like(h)
    lib().ora_rmsnorm(_p(h), _p(g), h.size, eps, act, _p(out))
    return out


def rope(v, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64)
    lib().ora_rope(_p(v), v.size, pos, theta)
    return v


def attention(q, K_bits, V_bits, act: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K_bits, dtype=np.uint16)
    V = np.ascontiguousarray(V_bits, dtype=np.uint16)
    out = np.empty(q.size, dtype=np.float64)
    lib().ora_attention(_p(q), _p(K), _p(V), K.shape[0], q.size, act, _p(out))
    return out


def argmax(v) -> int:
    v = np.ascontiguousarray(v, dtype=np.float64)
    return lib().ora_argmax(_p(v), v.size)


def silu(g: float) -> float:
    return lib().ora_silu(float(g))


def rtn_group(w_bits, act: int):
    """Quantize one group: returns (q uint8[n], s fp16 bits, z fp16 bits, rc)."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    q = np.zeros(w.size, dtype=np.uint8)
    s = ctypes.c_uint16(0)
    z = ctypes.c_uint16(0)
    rc = lib().ora_rtn_group(_p(w), w.size, act, _p(q), ctypes.addressof(s), ctypes.addressof(z))
    return q, s.value, z.value, rc


def hqq_pow_pm1(a: float) -> float:
    return float(lib().ora_hqq_pow_pm1(ctypes.c_float(a)))


def hqq_group(w_bits, act: int):
    """HQQ for one group: returns (q uint8[n], s fp16 bits, z fp16 bits, rc)."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    q = np.zeros(w.size, dtype=np.uint8)
    s = ctypes.c_uint16(0)
    z = ctypes.c_uint16(0)
    rc = lib().ora_hqq_group(_p(w), w.size, act, _p(q), ctypes.addressof(s), ctypes.addressof(z))
    return q, s.value, z.value, rc


# ---------------------------------------------------------------- model

def _cfg(shape, max_batch: int, max_seq: int) -> OraConfig:
    return OraConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim,
                     shape.ffn, shape.vocab, shape.tied_embed, shape.act_dtype, shape.rms_eps,
                     shape.rope_theta, max_batch, max_seq)


PROJ_NAMES = ("q", "k", "v", "o", "gate", "up", "down")


class Model:
    """Oracle model over referenced 16-bit weight arrays (kept alive here)."""

    def __init__(self, shape, weights: Sequence[Optional[np.ndarray]], max_batch: int, max_seq: int,
                 nthreads: Optional[int] = None):
        self.shape = shape
        self.max_batch, self.max_seq = max_batch, max_seq
        self._weights = [None if w is None else np.ascontiguousarray(w, dtype=np.uint16) for w in weights]
        ptrs = (ctypes.c_void_p * len(self._weights))(*[_p(w) for w in self._weights])
        self._ptrs = ptrs
        self.nthreads = nthreads or (os.cpu_count() or 1)
        self._cfg = _cfg(shape, max_batch, max_seq)
        h = ctypes.c_void_p()
        rc = lib().ora_create(ctypes.byref(self._cfg), ptrs, self.nthreads, ctypes.byref(h))
        if rc != RV_OK:
            raise RuntimeError(f"ora_create failed: {rc}")
        self._h = h
        self.group = None

    def close(self):
        if getattr(self, "_h", None):
            lib().ora_free(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def proj_dims(self, proj: int):
        s = self.shape
        d, qd, kvd = s.d_model, s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
        return [(qd, d), (kvd, d), (kvd, d), (d, qd), (s.ffn, d), (s.ffn, d), (d, s.ffn)][proj]

    def set_quantizer(self, method: int) -> int:
        """River quantizer for the next quantize_river: 0 RTN, 1 HQQ."""
        return int(lib().ora_set_quantizer(self._h, int(method)))

    def set_exit_cap(self, cap: int) -> int:
        """Backbone offloading: keep backbone layers 1..cap; exits are capped at cap."""
        return int(lib().ora_set_exit_cap(self._h, int(cap)))

    def set_threads(self, nthreads: int) -> int:
        """Host threads for the row loops (results do not depend on it)."""
        rc = int(lib().ora_set_threads(self._h, int(nthreads)))
        if rc == RV_OK:
            self.nthreads = int(nthreads)
        return rc

    def quantize_river(self, group: int, entry_layer: int = 1) -> int:
        rc = lib().ora_quantize_river(self._h, group, entry_layer)
        if rc == RV_OK:
            self.group = group
        return rc

    def export_river(self, layer: int, proj: int):
        N, K = self.proj_dims(proj)
        G = -(-K // self.group)
        q = np.zeros((N, K // 8), dtype=np.uint32)
        s = np.zeros((N, G), dtype=np.uint16)
        z = np.zeros((N, G), dtype=np.uint16)
        rc = lib().ora_export_river(self._h, layer, proj, _p(q), _p(s), _p(z))
        if rc != RV_OK:
            raise RuntimeError(f"ora_export_river failed: {rc}")
        return q, s, z

    def prefill(self, tokens: np.ndarray, tau: float, fixed_exit: int = -1, tf_exit=None, tf_ids=None,
                debug: bool = False):
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        B, T0 = tokens.shape
        L, d, V = self.shape.n_layers, self.shape.d_model, self.shape.vocab
        nxt = np.zeros(B, dtype=np.int32)
        ex = np.zeros(B, dtype=np.int32)
        nf = np.zeros(2, dtype=np.int32)
        tfe = None if tf_exit is None else np.ascontiguousarray(tf_exit, dtype=np.int32)
        tfi = None if tf_ids is None else np.ascontiguousarray(tf_ids, dtype=np.int32)
        smin = np.full((L, B), np.nan) if debug else None
        hid = np.zeros((L + 1, B, d)) if debug else None
        lg = np.zeros((B, V)) if debug else None
        rc = lib().ora_prefill(self._h, _p(tokens), B, T0, float(tau), fixed_exit, _p(tfe), _p(tfi), _p(nxt),
                               _p(ex), _p(smin), _p(hid), _p(lg), _p(nf))
        if rc != RV_OK:
            raise RuntimeError(f"ora_prefill failed: {rc}")
        out = {"next_ids": nxt, "exit_layer": ex, "n_forced": nf}
        if debug:
            out.update(smin=smin, hidden_last=hid, logits=lg)
        return out

    def decode_step(self, tokens, tau: float, forced=None, tf_exit=None, tf_ids=None, debug: bool = False):
        tokens = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        B = tokens.size
        L, d, V = self.shape.n_layers, self.shape.d_model, self.shape.vocab
        nxt = np.zeros(B, dtype=np.int32)
        ex = np.zeros(B, dtype=np.int32)
        nf = np.zeros(2, dtype=np.int32)
        fo = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
        tfe = None if tf_exit is None else np.ascontiguousarray(tf_exit, dtype=np.int32)
        tfi = None if tf_ids is None else np.ascontiguousarray(tf_ids, dtype=np.int32)
        hid = np.zeros((L + 1, B, d)) if debug else None
        ss = np.full((L, B), np.nan) if debug else None
        lg = np.zeros((B, V)) if debug else None
        rc = lib().ora_decode_step(self._h, _p(tokens), B, float(tau), _p(fo), _p(tfe), _p(tfi), _p(nxt), _p(ex),
                                   _p(hid), _p(ss), _p(lg), _p(nf))
        if rc != RV_OK:
            return {"rc": rc}
        out = {"rc": rc, "next_ids": nxt, "exit_layer": ex, "n_forced": nf}
        if debug:
            out.update(hidden=hid, s=ss, logits=lg)
        return out

    def layer_forward(self, layer: int, h_in, river) -> np.ndarray:
        """Layer `layer` (1-based) for rows 0..B-1 at their current positions."""
        h = np.ascontiguousarray(h_in, dtype=np.float64)
        B = h.shape[0]
        rv = np.ascontiguousarray(river, dtype=np.int32).reshape(-1)
        out = np.zeros_like(h)
        rc = lib().ora_layer_forward(self._h, layer, B, _p(rv), _p(h), _p(out))
        if rc != RV_OK:
            raise RuntimeError(f"ora_layer_forward failed: {rc}")
        return out

    def head(self, h):
        h = np.ascontiguousarray(h, dtype=np.float64)
        B = h.shape[0]
        logits = np.zeros((B, self.shape.vocab))
        ids = np.zeros(B, dtype=np.int32)
        rc = lib().ora_head(self._h, B, _p(h), _p(logits), _p(ids))
        if rc != RV_OK:
            raise RuntimeError(f"ora_head failed: {rc}")
        return logits, ids

    def kv_bytes(self) -> int:
        return int(lib().ora_kv_bytes(self._h))

    def kv_shape(self):
        s = self.shape
        return (s.n_layers, 2, self.max_batch, s.n_kv_heads, self.max_seq, s.head_dim)

    def get_kv(self) -> np.ndarray:
        a = np.empty(self.kv_shape(), dtype=np.uint16)
        rc = lib().ora_get_kv(self._h, _p(a), a.nbytes)
        assert rc == RV_OK
        return a

    def set_kv(self, kv: np.ndarray, lens) -> None:
        kv = np.ascontiguousarray(kv, dtype=np.uint16)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        rc = lib().ora_set_kv(self._h, _p(kv), kv.nbytes, _p(lens))
        if rc != RV_OK:
            raise RuntimeError(f"ora_set_kv failed: {rc}")

    def lens(self) -> np.ndarray:
        a = np.zeros(self.max_batch, dtype=np.int32)
        lib().ora_get_lens(self._h, _p(a))
        return a

    def kv_reset(self, rows=None) -> int:
        if rows is None:
            return lib().ora_kv_reset(self._h, None, 0)
        r = np.ascontiguousarray(rows, dtype=np.int32)
        return lib().ora_kv_reset(self._h, _p(r), r.size)
