"""Seeded synthetic inputs: model shapes, weights, prompts and forced exits.

This module draws numbers and nothing else.  It holds none of the River-LLM
arithmetic; the oracle and the CUDA library both receive what it returns as
plain input arrays (16-bit weight bit patterns, int32 token ids, int32 exit
layers).

Model shapes follow the Llama-3.2-1B / Llama-3.1-8B decoder shapes named for
the River-LLM evaluation ("River-LLM: Large Language Model Seamless Exit
Based on KV Share", paperlayer.ai summary, section 5 "Evaluation Setup"),
plus a tiny decoder for fast checks.  Weights are N(0, 0.02^2) rounded to the
16-bit type, RMSNorm gains are 1.0, prompt ids are uniform over the vocab.
"""
from __future__ import annotations

import ctypes
import os
import dataclasses
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None

FP16 = 0
BF16 = 1


def build(verbose: bool = False) -> str:
    """Compile libsynth.so with the host C compiler (no CUDA)."""
    import subprocess

    src = os.path.join(_HERE, "synth.c")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           src, "-o", _LIB_PATH, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(
            os.path.join(_HERE, "synth.c")):
        build()
    lib = ctypes.CDLL(_LIB_PATH)
    lib.synth_normal_act16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
    lib.synth_uniform_ids.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                      ctypes.c_int32, ctypes.c_void_p]
    lib.synth_forced_exits.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_void_p]
    lib.synth_fill_u16.argtypes = [ctypes.c_int64, ctypes.c_uint16, ctypes.c_void_p]
    for f in (lib.synth_normal_act16, lib.synth_uniform_ids, lib.synth_forced_exits, lib.synth_fill_u16):
        f.restype = ctypes.c_int
    _lib = lib
    return lib


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Decoder shape.  act_dtype 0 = fp16, 1 = bf16."""
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied_embed: int
    act_dtype: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    def param_count(self) -> int:
        d, hd = self.d_model, self.head_dim
        per_layer = (d * self.n_heads * hd + 2 * d * self.n_kv_heads * hd + self.n_heads * hd * d
                     + 3 * d * self.ffn + 2 * d)
        head = 0 if self.tied_embed else self.vocab * d
        return self.vocab * d + head + d + self.n_layers * per_layer

    def param_bytes(self) -> int:
        return 2 * self.param_count()


TINY = ModelShape("tiny", 4, 256, 4, 2, 64, 688, 1024, 0, FP16, 1e-5, 10000.0)
LLAMA_1B = ModelShape("llama3.2-1b-shape", 16, 2048, 32, 8, 64, 8192, 128256, 1, BF16, 1e-5, 500000.0)
LLAMA_8B = ModelShape("llama3.1-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256, 0, BF16, 1e-5, 500000.0)
# Two layers of the 8B shape with a 32000-entry vocab: a ~1.4 GB case whose
# per-layer matrices are still larger than L2, for profiler captures.
LAYER8B = ModelShape("llama3.1-8b-shape-2layer", 2, 4096, 32, 8, 128, 14336, 32000, 0, BF16, 1e-5, 500000.0)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: shape, river group, batch, prompt, steps, exit rule."""
    name: str
    shape: ModelShape
    group: int
    batch: int
    prompt_len: int
    steps: int
    taus: tuple
    forced: bool
    prefill_tau: float
    fixed_prefill_exit: int = -1


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 64, 1, 32, 32, (0.90,), False, 0.90),
    "llama1b": Workload("llama1b", LLAMA_1B, 128, 1, 512, 256, (0.85, 0.90, 0.95), True, 0.90),
    "llama8b": Workload("llama8b", LLAMA_8B, 128, 1, 1024, 512, (0.90,), True, 0.90),
    "batch64": Workload("batch64", LLAMA_1B, 128, 64, 256, 128, (), True, 0.90),
    "long64k": Workload("long64k", LLAMA_8B, 128, 1, 65536, 256, (0.90,), False, 0.90, 20),
    "layer8b": Workload("layer8b", LAYER8B, 128, 1, 64, 16, (0.90,), True, 0.90),
}

SEED_WEIGHTS = 1234
SEED_PROMPT = 42
SEED_FORCED = 7

# Tensor order of the weight list handed to both sides:
#   0: token embedding E [V, d]
#   1: final RMSNorm gain [d]
#   2: LM head [V, d] (None when tied to E)
#   3 + 9*l + j, j = 0..8: attn gain [d], W_q [H*hd, d], W_k [Hkv*hd, d],
#      W_v [Hkv*hd, d], W_o [d, H*hd], mlp gain [d], W_gate [F, d],
#      W_up [F, d], W_down [d, F]
LAYER_TENSORS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown")


def tensor_shapes(s: ModelShape) -> List[Optional[tuple]]:
    d, hd, F = s.d_model, s.head_dim, s.ffn
    out: List[Optional[tuple]] = [(s.vocab, d), (d,), None if s.tied_embed else (s.vocab, d)]
    for _ in range(s.n_layers):
        out += [(d,), (s.n_heads * hd, d), (s.n_kv_heads * hd, d), (s.n_kv_heads * hd, d),
                (d, s.n_heads * hd), (d,), (F, d), (F, d), (d, F)]
    return out


def _one_bits(dtype: int) -> int:
    return 0x3F80 if dtype == BF16 else 0x3C00


def make_weights(s: ModelShape, seed: int = SEED_WEIGHTS, std: float = 0.02,
                 nthreads: Optional[int] = None) -> List[Optional[np.ndarray]]:
    """All weights as uint16 arrays holding act16 bit patterns."""
    lib = _load()
    nthreads = nthreads or (os.cpu_count() or 1)
    shapes = tensor_shapes(s)
    out: List[Optional[np.ndarray]] = []
    for tid, shp in enumerate(shapes):
        if shp is None:
            out.append(None)
            continue
        a = np.empty(shp, dtype=np.uint16)
        if len(shp) == 1:  # RMSNorm gains are 1.0
            lib.synth_fill_u16(a.size, _one_bits(s.act_dtype), a.ctypes.data)
        else:
            rc = lib.synth_normal_act16(seed, tid, std, a.size, s.act_dtype, a.ctypes.data, nthreads)
            assert rc == 0
        out.append(a)
    return out


def normal_act16(seed: int, tid: int, n: int, dtype: int, std: float = 0.02) -> np.ndarray:
    lib = _load()
    a = np.empty(n, dtype=np.uint16)
    lib.synth_normal_act16(seed, tid, std, n, dtype, a.ctypes.data, os.cpu_count() or 1)
    return a


def make_prompt(vocab: int, batch: int, length: int, seed: int = SEED_PROMPT) -> np.ndarray:
    lib = _load()
    a = np.empty((batch, length), dtype=np.int32)
    lib.synth_uniform_ids(seed, 1, a.size, vocab, a.ctypes.data)
    return a


def uniform_ids(seed: int, tid: int, n: int, vocab: int) -> np.ndarray:
    lib = _load()
    a = np.empty(n, dtype=np.int32)
    lib.synth_uniform_ids(seed, tid, n, vocab, a.ctypes.data)
    return a


def forced_exits(step: int, batch: int, n_layers: int, seed: int = SEED_FORCED) -> np.ndarray:
    """Exit layers for one decode step: 55% uniform in 1..5, 45% uniform in 6..L."""
    lib = _load()
    a = np.empty(batch, dtype=np.int32)
    lib.synth_forced_exits(seed, step, batch, n_layers, a.ctypes.data)
    return a


def act16_to_f32(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode 16-bit patterns to float32 (display and test helper)."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)
