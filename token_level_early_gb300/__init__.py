"""River-LLM token-level early-exit decode on GB300 (sm_103a).

Thin ctypes binding of librv.so (C ABI in include/rv.h).  Every step of the
decode path runs in the library's CUDA kernels; this module only marshals
arguments and raises RVError on a non-zero status.  There is no CPU fallback:
loading fails loudly when librv.so is missing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import concurrent.futures as _fut
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
LIB_PATH = os.path.join(_HERE, "librv.so")
_CSRC = os.path.join(_HERE, "csrc")
_BUILD = os.path.join(_ROOT, "_build")
SOURCES = ["api.cu", "decode_b1.cu", "attention.cu", "general.cu", "quant.cu", "noalloc.cu", "stream.cu", "gemm_tc.cu", "rows_mma.cu"]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"

RV_OK, RV_EINVAL, RV_ENOMEM, RV_ECUDA, RV_ECAPACITY, RV_ESTATE, RV_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
PROJ_Q, PROJ_K, PROJ_V, PROJ_O, PROJ_GATE, PROJ_UP, PROJ_DOWN = range(7)
DUMP_HIDDEN, DUMP_S, DUMP_LOGITS, DUMP_KV, DUMP_LENS = range(5)
EXPORTED = ("rv_last_error", "rv_load_model", "rv_quantize_river", "rv_export_river", "rv_prefill",
            "rv_decode_step", "rv_decode_step_dev", "rv_sync_status", "rv_kv_reset", "rv_set_debug",
            "rv_debug_dump", "rv_kv_bytes", "rv_param_bytes", "rv_free_model", "rv_time_kernel", "rv_greedy_head_noalloc", "rv_offload_backbone",
            "rv_set_option", "rv_debug_fail_alloc", "rv_decode_attention_plan")
OPT_DECODE_ENGINE, ENGINE_CHAIN, ENGINE_PERSISTENT = 0, 0, 1
OPT_QUANTIZER, QUANT_RTN, QUANT_HQQ = 1, 0, 1
OPT_WAIT_LIMIT_US = 2
TIME_GATEUP, TIME_O, TIME_LMHEAD, TIME_ATTN = 0, 1, 2, 3


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def build(verbose: bool = False) -> str:
    """Compile librv.so for sm_103a (one translation unit per source, in parallel)."""
    os.makedirs(_BUILD, exist_ok=True)
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-O3",
             "--expt-relaxed-constexpr"]
    hdrs = [os.path.join(_CSRC, h) for h in os.listdir(_CSRC) if h.endswith(".cuh")]
    hdrs.append(os.path.join(_ROOT, "include", "rv.h"))
    newest_hdr = max(os.path.getmtime(h) for h in hdrs)

    def one(src):
        s = os.path.join(_CSRC, src)
        o = os.path.join(_BUILD, src.replace(".cu", ".o"))
        if os.path.exists(o) and os.path.getmtime(o) >= max(os.path.getmtime(s), newest_hdr):
            return o
        cmd = [nvcc(), *flags, "-c", s, "-o", o]
        if verbose:
            print(" ".join(cmd))
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return o

    with _fut.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    cmd = [nvcc(), ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64", *objs,
           "-o", LIB_PATH]
    if verbose:
        print(" ".join(cmd))
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    return LIB_PATH


class RVConfig(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("tied_embed", ctypes.c_int), ("act_dtype", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("max_batch", ctypes.c_int), ("max_seq", ctypes.c_int)]


class RVError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"rv error {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """Load librv.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (token_level_early_gb300.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "rv_last_error": ([], ctypes.c_char_p),
        "rv_load_model": ([ctypes.POINTER(RVConfig), vp, vp, ctypes.POINTER(vp)], i32),
        "rv_quantize_river": ([vp, i32, i32], i32),
        "rv_export_river": ([vp, i32, i32, vp, vp, vp], i32),
        "rv_prefill": ([vp, vp, i32, i32, f32, i32, vp, vp], i32),
        "rv_decode_step": ([vp, vp, i32, f32, vp, vp, vp], i32),
        "rv_decode_step_dev": ([vp, vp, i32, f32, vp, vp, vp], i32),
        "rv_sync_status": ([vp], i32),
        "rv_kv_reset": ([vp, vp, i32], i32),
        "rv_set_debug": ([vp, i32], i32),
        "rv_debug_dump": ([vp, i32, vp, sz], i32),
        "rv_kv_bytes": ([vp], sz),
        "rv_param_bytes": ([vp, i32], sz),
        "rv_offload_backbone": ([vp, i32], i32),
        "rv_free_model": ([vp], None),
        "rv_time_kernel": ([vp, i32, i32, i32, i32, ctypes.POINTER(ctypes.c_float),
                            ctypes.POINTER(ctypes.c_double)], i32),
        "rv_greedy_head_noalloc": ([vp, vp, vp, i32, i32, i32, f32, vp, vp, vp], i32),
        "rv_set_option": ([vp, i32, i32], i32),
        "rv_debug_fail_alloc": ([i32], i32),
        "rv_decode_attention_plan": ([i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def _check(rc: int):
    if rc != RV_OK:
        raise RVError(rc, lib().rv_last_error().decode(errors="replace"))


def _p(a):
    return None if a is None else a.ctypes.data


def greedy_head_noalloc(d_lm_head: int, d_final_norm: int, d_h: int, vocab: int, d_model: int, act_dtype: int,
                        rms_eps: float, d_next_id: int, d_logits: Optional[int] = None, stream: Optional[int] = None):
    """rv_greedy_head_noalloc on device pointers (see include/rv.h)."""
    _check(lib().rv_greedy_head_noalloc(d_lm_head, d_final_norm, d_h, vocab, d_model, act_dtype, float(rms_eps),
                                        d_next_id, d_logits, stream))


def decode_attention_plan(batch: int, n_kv_heads: int, n_sm: int, max_cluster: int, max_splits: int,
                          context: int):
    """rv_decode_attention_plan (host arithmetic, no GPU needed): returns
    (plan, splits), plan 0 = cluster plan, 1 = global-merge plan."""
    sp = ctypes.c_int(0)
    rc = lib().rv_decode_attention_plan(batch, n_kv_heads, n_sm, max_cluster, max_splits, context, ctypes.byref(sp))
    if rc < 0:
        _check(rc)
    return rc, sp.value


def debug_fail_alloc(after: int) -> None:
    """Test hook: the device allocation after the next `after` ones fails
    (once); after < 0 turns it off (rv_debug_fail_alloc)."""
    _check(lib().rv_debug_fail_alloc(int(after)))


def config_of(shape, max_batch: int, max_seq: int) -> RVConfig:
    return RVConfig(shape.n_layers, shape.d_model, shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                    shape.vocab, shape.tied_embed, shape.act_dtype, shape.rms_eps, shape.rope_theta, max_batch,
                    max_seq)


class Model:
    """A backbone on the GPU with its river and KV cache (owns an rv_model)."""

    def __init__(self, shape, weights: Sequence[Optional[np.ndarray]], max_batch: int, max_seq: int,
                 stream: Optional[int] = None):
        self.shape = shape
        self.max_batch, self.max_seq = max_batch, max_seq
        ws = [None if w is None else np.ascontiguousarray(w, dtype=np.uint16) for w in weights]
        ptrs = (ctypes.c_void_p * len(ws))(*[_p(w) for w in ws])
        self._cfg = config_of(shape, max_batch, max_seq)
        h = ctypes.c_void_p()
        _check(lib().rv_load_model(ctypes.byref(self._cfg), ptrs, stream, ctypes.byref(h)))
        self._h = h
        self.group = None

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            lib().rv_free_model(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def proj_dims(self, proj: int):
        s = self.shape
        d, qd, kvd = s.d_model, s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
        return [(qd, d), (kvd, d), (kvd, d), (d, qd), (s.ffn, d), (s.ffn, d), (d, s.ffn)][proj]

    def quantize_river(self, group: int, entry_layer: int = 1):
        _check(lib().rv_quantize_river(self._h, group, entry_layer))
        self.group = group

    def export_river(self, layer: int, proj: int):
        N, K = self.proj_dims(proj)
        G = -(-K // self.group)
        q = np.zeros((N, K // 8), dtype=np.uint32)
        s = np.zeros((N, G), dtype=np.uint16)
        z = np.zeros((N, G), dtype=np.uint16)
        _check(lib().rv_export_river(self._h, layer, proj, _p(q), _p(s), _p(z)))
        return q, s, z

    def prefill(self, tokens: np.ndarray, tau: float, fixed_exit: int = -1):
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        B, T0 = t.shape
        nxt = np.zeros(B, dtype=np.int32)
        ex = np.zeros(B, dtype=np.int32)
        _check(lib().rv_prefill(self._h, _p(t), B, T0, float(tau), int(fixed_exit), _p(nxt), _p(ex)))
        return nxt, ex

    def decode_step(self, tokens, tau: float, forced=None):
        t = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
        B = t.size
        f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32).reshape(-1)
        nxt = np.zeros(B, dtype=np.int32)
        ex = np.zeros(B, dtype=np.int32)
        _check(lib().rv_decode_step(self._h, _p(t), B, float(tau), _p(f), _p(nxt), _p(ex)))
        return nxt, ex

    def decode_step_dev(self, d_tokens: int, B: int, tau: float, d_forced: Optional[int], d_next: int,
                        d_exit: int):
        _check(lib().rv_decode_step_dev(self._h, d_tokens, B, float(tau), d_forced, d_next, d_exit))

    def sync_status(self):
        _check(lib().rv_sync_status(self._h))

    def kv_reset(self, rows=None):
        if rows is None:
            _check(lib().rv_kv_reset(self._h, None, 0))
        else:
            r = np.ascontiguousarray(rows, dtype=np.int32)
            _check(lib().rv_kv_reset(self._h, _p(r), r.size))

    def set_option(self, option: int, value: int):
        _check(lib().rv_set_option(self._h, option, value))

    def set_engine(self, engine: int):
        self.set_option(OPT_DECODE_ENGINE, engine)

    def set_quantizer(self, method: int):
        """River quantizer of the next quantize_river: QUANT_RTN or QUANT_HQQ."""
        self.set_option(OPT_QUANTIZER, method)

    def set_debug(self, enable: bool):
        _check(lib().rv_set_debug(self._h, 1 if enable else 0))

    def dump(self, what: int) -> np.ndarray:
        s, B = self.shape, self.max_batch
        if what == DUMP_HIDDEN:
            a = np.zeros((s.n_layers + 1, B, s.d_model), dtype=np.float32)
        elif what == DUMP_S:
            a = np.zeros((s.n_layers, B), dtype=np.float32)
        elif what == DUMP_LOGITS:
            a = np.zeros((B, s.vocab), dtype=np.float32)
        elif what == DUMP_KV:
            a = np.zeros((s.n_layers, 2, B, s.n_kv_heads, self.max_seq, s.head_dim), dtype=np.uint16)
        elif what == DUMP_LENS:
            a = np.zeros(B, dtype=np.int32)
        else:
            raise ValueError(what)
        _check(lib().rv_debug_dump(self._h, what, _p(a), a.nbytes))
        return a

    def time_kernel(self, kind: int, layer: int, river: bool, iters: int):
        """Mean device ms per launch and algorithmic bytes per launch of one GEMV kernel."""
        ms = ctypes.c_float(0)
        by = ctypes.c_double(0)
        _check(lib().rv_time_kernel(self._h, kind, layer, 1 if river else 0, iters, ctypes.byref(ms),
                                    ctypes.byref(by)))
        return float(ms.value), float(by.value)

    def kv_bytes(self) -> int:
        return int(lib().rv_kv_bytes(self._h))

    def offload_backbone(self, keep_layers: int) -> None:
        """Free backbone layers keep_layers+1..L on the device; exits are capped at keep_layers."""
        _check(lib().rv_offload_backbone(self._h, int(keep_layers)))

    def param_bytes(self, which: int) -> int:
        return int(lib().rv_param_bytes(self._h, which))
