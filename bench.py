#!/usr/bin/env python3
"""Decode benchmark: River-LLM token-level early exit at batch 1 on one GB300.

One step = one decode step of the whole hot path (embedding, every layer on
the backbone or river path with the exit decision, K/V append into the one
shared cache, LM head + greedy pick) for one token.  Default workload: the
Llama-3.1-8B-shaped decoder (bf16, river W4A16 group 128), 1024-token random
prompt, tau = 0.90; the Llama-3.2-1B-shaped workload is reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload llama8b|llama1b|layer8b] [--modes tau,forced,full,river]
                  [--engine chain|persistent] [--no-cpu-baseline] [--no-secondary]
                  [--no-fidelity] [--no-extra] [--only batch64|long64k] [--prompt-len N]

value : decode tokens/s, device-timed with CUDA events on the model's stream;
        tokens chained on the device (step i+1 consumes step i's id).
e2e   : the same metric through rv_decode_step with host buffers (token H2D,
        id + exit layer D2H inside the timed region), wall clock.
Also in the line: every mode of the decode step (tau rule, forced exits,
full backbone, all river) with its achieved GB/s, the river vs backbone layer
time (layer_us), the roofline line of the dominant kernel of the tau step
(the river's gate/up GEMV; the backbone's beside it), single-kernel timings
(GEMVs, LM head, decode attention), backbone offloading (layers 1..3 kept),
fidelity of the RTN and HQQ rivers against the full backbone, the CPU oracle
baseline, the 1B shape with its tau sweep (0.85, 0.90, 0.95), the batch-64
mixed-exit workload and the 64K-context workload (KV bytes, decode rate,
the decode attention's K/V read rate).
Multi-GPU: independent replicas (the batch-1 decode step does not shard).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

ENGINE_NAMES = {0: "chain", 1: "persistent"}
METRIC = "decode tokens/s at bs1 (1B/8B shapes) and achieved HBM GB/s vs ~8 TB/s peak"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gemv_gateup_llama8b.md")
MODES = ("tau", "forced", "full", "river")


# ------------------------------------------------------------------ helpers

def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.samples, self.proc, self.thread = index, [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def rd():
            for line in self.proc.stdout:
                self.samples.append([x.strip() for x in line.split(",")])

        self.thread = threading.Thread(target=rd, daemon=True)
        self.thread.start()

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in self.samples:
            try:
                sm.append(float(s[1]))
                mx.append(float(s[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, s[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def layer_bytes(shape, group):
    """Algorithmic HBM bytes of one backbone layer and of its river copy:
    the four weight matrices (int4 codes + fp16 scale and zero per group for
    the river) and the two RMSNorm gains."""
    d, F = shape.d_model, shape.ffn
    qd, kvd = shape.n_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    mats = [(qd + 2 * kvd, d), (d, qd), (2 * F, d), (d, F)]
    bb = sum(2 * n * k for n, k in mats) + 2 * 2 * d
    rv_ = sum(n * k // 2 + n * (-(-k // group)) * 4 for n, k in mats) + 2 * 2 * d
    return bb, rv_


def token_bytes(shape, group, exit_layer, ctx):
    """bytes(e, T) = e W_bb + (L - e) W_rv + W_lm + embedding row + K/V read
    over the T cached positions and the new one + K/V written in every layer."""
    L, d = shape.n_layers, shape.d_model
    bb, rv_ = layer_bytes(shape, group)
    kv_pos = L * 2 * shape.n_kv_heads * shape.head_dim * 2
    e = int(exit_layer)
    return e * bb + (L - e) * rv_ + 2 * shape.vocab * d + 2 * d + (ctx + 1) * kv_pos + kv_pos


def kernel_hash():
    h = hashlib.sha256()
    for f in ("decode_b1.cu", "gemv_core.cuh", "kernels.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "token_level_early_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(path):
    """Per-launch DRAM bytes of the gate/up GEMV (path "int4" or "bf16") from
    the committed ncu summary, when it was taken on the current kernel
    source; else None."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    vals = {}
    with open(PROFILE_SUMMARY) as f:
        for line in f:
            t = line.strip()
            if t.startswith("- ") and ":" in t:
                k, v = t[2:].split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256") != kernel_hash():
        return None
    try:
        return float(vals[f"traffic_bytes_per_launch_{path}"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ our arm

def run_workload(wl_name, steps, warmup, dev_index, want_cpu, rank0, log, modes=MODES, engine_name="chain",
                 want_offload=False):
    import torch
    import token_level_early_gb300 as rv

    engine = {"chain": rv.ENGINE_CHAIN, "persistent": rv.ENGINE_PERSISTENT}[engine_name]

    wl = synth.WORKLOADS[wl_name]
    shape = wl.shape
    L = shape.n_layers
    tau = wl.taus[0] if wl.taus else 0.90
    torch.cuda.set_device(dev_index)
    t0 = time.time()
    w = synth.make_weights(shape)
    log(f"[{wl_name}] weights generated in {time.time() - t0:.1f}s")
    prompt = synth.make_prompt(shape.vocab, 1, wl.prompt_len)
    max_seq = wl.prompt_len + (len(MODES) + 2 + len(wl.taus)) * (warmup + steps) + steps + 72  # + CPU baseline
    stream = torch.cuda.Stream()
    t0 = time.time()
    m = rv.Model(shape, w, 1, max_seq, stream=stream.cuda_stream)
    m.quantize_river(wl.group, 1)
    m.set_engine(engine)
    log(f"[{wl_name}] load + river in {time.time() - t0:.1f}s")
    t0 = time.time()
    first, e_seq = m.prefill(prompt, wl.prefill_tau)
    log(f"[{wl_name}] prefill {wl.prompt_len} tokens in {time.time() - t0:.1f}s, exit layer {int(e_seq[0])}")

    n_ids = (len(MODES) + 2 + len(wl.taus)) * (warmup + steps) + 1
    d_ids = torch.zeros(n_ids, dtype=torch.int32, device="cuda")
    d_exit = torch.zeros_like(d_ids)
    d_forced = torch.from_numpy(np.concatenate([synth.forced_exits(i, 1, L) for i in range(warmup + steps)])).cuda()
    d_zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_full = torch.full((1,), L, dtype=torch.int32, device="cuda")
    d_ids[0] = int(first[0])
    torch.cuda.synchronize()
    pos = [0]

    def run_mode(mode, n, sampler=None, tau=tau):
        i0 = pos[0]
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
        ev0.record(stream)
        for i in range(n):
            k = i0 + i
            forced = {"tau": None, "forced": d_forced[i:].data_ptr(), "full": d_full.data_ptr(),
                      "river": d_zero.data_ptr()}[mode]
            m.decode_step_dev(d_ids[k:].data_ptr(), 1, tau, forced, d_ids[k + 1:].data_ptr(),
                              d_exit[k + 1:].data_ptr())
        ev1.record(stream)
        ev1.synchronize()
        clocks = sampler.stop() if sampler else None
        m.sync_status()
        pos[0] += n
        return ev0.elapsed_time(ev1), d_exit[i0 + 1:i0 + n + 1].cpu().numpy(), clocks

    results = {}
    for mode in modes:
        run_mode(mode, warmup)
        ctx0 = wl.prompt_len + pos[0]
        ms, exits, clocks = run_mode(mode, steps, ClockSampler(dev_index) if mode == "tau" else None)
        by = sum(token_bytes(shape, wl.group, e, ctx0 + i) for i, e in enumerate(exits))
        results[mode] = {"tokens_per_s": steps / (ms / 1e3), "ms_per_step": ms / steps,
                         "achieved_gbs": by / (ms / 1e3) / 1e9, "mean_exit_layer": float(np.mean(exits)),
                         "bytes_per_token": by / steps}
        if clocks is not None:
            results[mode]["clocks"] = clocks

    # the workload's tau sweep (the tau-rule step at every tau it names)
    sweep = {}
    if "tau" in modes and len(wl.taus) > 1:
        for t_ in wl.taus:
            run_mode("tau", warmup, tau=t_)
            ctx0 = wl.prompt_len + pos[0]
            ms, exits, _ = run_mode("tau", steps, tau=t_)
            by = sum(token_bytes(shape, wl.group, e, ctx0 + i) for i, e in enumerate(exits))
            sweep[f"{t_:.2f}"] = {"tokens_per_s": steps / (ms / 1e3), "achieved_gbs": by / (ms / 1e3) / 1e9,
                                  "mean_exit_layer": float(np.mean(exits))}

    # the headline mode again on the other batch-1 engine, for comparison
    other = rv.ENGINE_PERSISTENT if engine == rv.ENGINE_CHAIN else rv.ENGINE_CHAIN
    m.set_engine(other)
    run_mode(modes[0], warmup)
    ms_c, _, _ = run_mode(modes[0], steps)
    results[modes[0]][ENGINE_NAMES[other] + "_engine_tokens_per_s"] = steps / (ms_c / 1e3)
    m.set_engine(engine)

    # e2e: the same tau-rule loop through the host-buffer API
    tok = int(d_ids[pos[0]].item())
    t0 = time.perf_counter()
    for _ in range(steps):
        nxt, _ = m.decode_step([tok], tau)
        tok = int(nxt[0])
    e2e_s = time.perf_counter() - t0

    kern = {}
    for name, kind, river in (("gateup_bf16", rv.TIME_GATEUP, False), ("gateup_int4", rv.TIME_GATEUP, True),
                              ("o_bf16", rv.TIME_O, False), ("o_int4", rv.TIME_O, True),
                              ("lmhead_bf16", rv.TIME_LMHEAD, False), ("attention", rv.TIME_ATTN, False)):
        ms, by = m.time_kernel(kind, 1, river, 20)
        kern[name] = {"ms": ms, "bytes": by, "gbs": by / (ms / 1e3) / 1e9}

    cpu = cpu_baseline(m, shape, w, wl, max_seq, tok, tau, log) if (want_cpu and rank0) else None

    # backbone offloading (the pages' parameter-memory comparison): keep the
    # first backbone layers on the device, cap the exits there, decode on
    offload = None
    if want_offload and L > 3:
        keep = 3
        full_bytes = m.param_bytes(0) + m.param_bytes(1)
        m.offload_backbone(keep)
        run_mode("tau", warmup)
        ctx0 = wl.prompt_len + pos[0]
        ms, exits, _ = run_mode("tau", steps)
        resident = m.param_bytes(0) + m.param_bytes(1)
        by = sum(token_bytes(shape, wl.group, e, ctx0 + i) for i, e in enumerate(exits))
        offload = {"keep_layers": keep, "resident_param_bytes": resident, "resident_param_gib": resident / 2 ** 30,
                   "full_param_gib": full_bytes / 2 ** 30, "backbone_16bit_gib": m.param_bytes(0) / 2 ** 30,
                   "river_gib": m.param_bytes(1) / 2 ** 30, "tau_tokens_per_s": steps / (ms / 1e3),
                   "achieved_gbs": by / (ms / 1e3) / 1e9, "mean_exit_layer": float(np.mean(exits)),
                   "pages": "14.96 GiB -> 6.73 GiB (backbone offloading)"}
        log(f"[{wl_name}] offload keep {keep}: {resident / 2 ** 30:.2f} GiB resident, "
            f"{offload['tau_tokens_per_s']:.1f} tokens/s")
    m.close()
    return {"modes": results, "e2e_tokens_per_s": steps / e2e_s, "kernels": kern, "cpu": cpu,
            "prefill_exit": int(e_seq[0]), "offload": offload, "tau_sweep": sweep or None}


def run_batch64(steps, warmup, dev_index, log):
    """The batched heterogeneous-exit workload: 64 sequences of the 1B shape,
    256-token prompts, per-row per-step forced exit layers (every layer of a
    step mixes backbone and river rows writing the one cache).  Decode steps
    through the device-pointer API, tokens chained on the device."""
    import torch
    import token_level_early_gb300 as rv

    wl = synth.WORKLOADS["batch64"]
    shape, B = wl.shape, wl.batch
    L = shape.n_layers
    torch.cuda.set_device(dev_index)
    w = synth.make_weights(shape)
    stream = torch.cuda.Stream()
    T = wl.prompt_len + warmup + steps + 4
    m = rv.Model(shape, w, B, T, stream=stream.cuda_stream)
    m.quantize_river(wl.group, 1)
    prompts = synth.make_prompt(shape.vocab, B, wl.prompt_len)
    t0 = time.time()
    first, _ = m.prefill(prompts, wl.prefill_tau)
    log(f"[batch64] prefill {B} x {wl.prompt_len} tokens in {time.time() - t0:.1f}s")
    ids = torch.zeros((warmup + steps + 1, B), dtype=torch.int32, device="cuda")
    ex = torch.zeros_like(ids)
    ids[0] = torch.from_numpy(first).cuda()
    forced = torch.from_numpy(np.stack([synth.forced_exits(i, B, L) for i in range(warmup + steps)])).cuda()
    torch.cuda.synchronize()

    def run(i0, n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(i0, i0 + n):
            m.decode_step_dev(ids[i].data_ptr(), B, 0.9, forced[i].data_ptr(), ids[i + 1].data_ptr(),
                              ex[i + 1].data_ptr())
        ev1.record(stream)
        ev1.synchronize()
        m.sync_status()
        return ev0.elapsed_time(ev1)

    run(0, warmup)
    ms = run(warmup, steps)
    ex_np = ex[warmup + 1:].cpu().numpy()
    m.close()
    bb, rv_ = layer_bytes(shape, wl.group)
    # both weight sets of every layer a step touches (a layer with rows on both
    # paths streams both), the LM head, and the K/V of every row
    layers_both = [(int((e < l + 1).any()), int((e >= l + 1).any())) for e in ex_np for l in range(L)]
    wbytes = sum(r * rv_ + b * bb for b, r in layers_both) / steps + 2 * shape.vocab * shape.d_model
    kv_pos = L * 2 * shape.n_kv_heads * shape.head_dim * 2
    ctx = wl.prompt_len + warmup + steps / 2
    by = wbytes + B * (ctx + 2) * kv_pos
    out = {"workload": f"{shape.name} decode, batch {B}, {wl.prompt_len}-token prompts, per-row forced exits",
           "tokens_per_s": B * steps / (ms / 1e3), "ms_per_step": ms / steps, "steps": steps,
           "achieved_gbs": by / (ms / steps / 1e3) / 1e9, "bytes_per_step": by,
           "mean_exit_layer": float(ex_np.mean())}
    log(f"[batch64] {out['tokens_per_s']:.0f} tokens/s, {out['ms_per_step']:.2f} ms/step")
    return out


def run_long64k(steps, warmup, dev_index, log):
    """The long-context workload: the 8B shape, a 65536-token prompt with the
    sequence exit fixed at layer 20, then tau 0.90 decode steps; reports the
    KV cache bytes (unchanged by building the river), the decode rate and the
    decode attention's K/V read rate at this context."""
    import torch
    import token_level_early_gb300 as rv

    wl = synth.WORKLOADS["long64k"]
    shape = wl.shape
    torch.cuda.set_device(dev_index)
    w = synth.make_weights(shape)
    stream = torch.cuda.Stream()
    T = wl.prompt_len + warmup + steps + 4
    m = rv.Model(shape, w, 1, T, stream=stream.cuda_stream)
    del w
    kv0 = m.kv_bytes()
    m.quantize_river(wl.group, 1)
    kv1 = m.kv_bytes()
    prompt = synth.make_prompt(shape.vocab, 1, wl.prompt_len)
    t0 = time.time()
    first, e_seq = m.prefill(prompt, wl.prefill_tau, fixed_exit=wl.fixed_prefill_exit)
    pre_s = time.time() - t0
    log(f"[long64k] prefill {wl.prompt_len} tokens in {pre_s:.1f}s (exit layer {int(e_seq[0])})")
    ids = torch.zeros(warmup + steps + 1, dtype=torch.int32, device="cuda")
    ex = torch.zeros_like(ids)
    ids[0] = int(first[0])
    torch.cuda.synchronize()

    def run(i0, n):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for i in range(i0, i0 + n):
            m.decode_step_dev(ids[i:].data_ptr(), 1, wl.taus[0], None, ids[i + 1:].data_ptr(), ex[i + 1:].data_ptr())
        ev1.record(stream)
        ev1.synchronize()
        m.sync_status()
        return ev0.elapsed_time(ev1)

    run(0, warmup)
    ctx0 = wl.prompt_len + warmup
    ms = run(warmup, steps)
    exits = ex[warmup + 1:].cpu().numpy()
    by = sum(token_bytes(shape, wl.group, e, ctx0 + i) for i, e in enumerate(exits))
    a_ms, a_by = m.time_kernel(rv.TIME_ATTN, 1, False, 20)
    m.close()
    peak, _ = peak_hbm()
    out = {"workload": f"{shape.name} decode, batch 1, {wl.prompt_len}-token prompt (sequence exit fixed at "
                       f"layer {wl.fixed_prefill_exit}), tau {wl.taus[0]}",
           "tokens_per_s": steps / (ms / 1e3), "ms_per_step": ms / steps, "steps": steps,
           "achieved_gbs": by / (ms / 1e3) / 1e9, "mean_exit_layer": float(np.mean(exits)),
           "kv_cache_bytes": kv0, "kv_cache_bytes_after_river": kv1, "prefill_s": pre_s,
           "kv_read_bytes_per_step": 2 * shape.n_kv_heads * shape.head_dim * 2 * (ctx0 + steps // 2) * shape.n_layers,
           "attention": {"layer": 1, "ms": a_ms, "bytes": a_by, "gbs": a_by / (a_ms / 1e3) / 1e9,
                         "frac_of_measured_hbm": a_by / (a_ms / 1e3) / 1e9 / peak}}
    log(f"[long64k] {out['tokens_per_s']:.1f} tokens/s; attention {out['attention']['gbs']:.0f} GB/s")
    return out


def cpu_baseline(gm, shape, w, wl, max_seq, tok, tau, log, budget_s=20.0):
    """The oracle as it stands, on this host's cores: decode steps from the
    GPU run's cache state (same model, same context length), time-bounded."""
    import oracle
    import token_level_early_gb300 as rv

    kv = gm.dump(rv.DUMP_KV)
    lens = gm.dump(rv.DUMP_LENS)
    nthreads = os.cpu_count() or 1
    om = oracle.Model(shape, w, 1, max_seq, nthreads=nthreads)
    om.quantize_river(wl.group, 1)
    om.set_kv(kv, lens)
    del kv
    n, t0 = 0, time.perf_counter()
    while n < 64:
        out = om.decode_step([tok], tau)
        tok = int(out["next_ids"][0])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    # one more step on a single core (the oracle's results do not depend on
    # its thread count)
    one = None
    if om.set_threads(1) == 0:
        t1 = time.perf_counter()
        out = om.decode_step([tok], tau)
        one = 1.0 / (time.perf_counter() - t1)
    om.close()
    log(f"[cpu] oracle {n} decode steps in {dt:.1f}s on {nthreads} threads; 1 thread: {one}")
    return {"value": n / dt, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "single_core_value": one,
            "sample": f"{n} oracle decode steps (tau {tau}) of the {shape.name} workload at context "
                      f"{int(lens[0])}, started from the GPU run's KV cache; one more step on 1 thread"}


def kl_div(a, b):
    """KL(softmax(a) || softmax(b)) in float64."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    la = a - a.max()
    lb = b - b.max()
    la -= np.log(np.exp(la).sum())
    lb -= np.log(np.exp(lb).sum())
    return float(np.sum(np.exp(la) * (la - lb)))


def fidelity(wl_name, steps, dev_index, log):
    """River vs full backbone on one token stream (the backbone's greedy ids):
    per step, does the tau-rule model pick the same next token, and
    KL(backbone || river) of the two next-token distributions.  Measured for
    both river quantizers (RTN and HQQ), with the time each takes to build
    the river."""
    import torch
    import token_level_early_gb300 as rv

    wl = synth.WORKLOADS[wl_name]
    shape = wl.shape
    L = shape.n_layers
    tau = wl.taus[0] if wl.taus else 0.90
    torch.cuda.set_device(dev_index)
    w = synth.make_weights(shape)
    prompt = synth.make_prompt(shape.vocab, 1, wl.prompt_len)
    T = wl.prompt_len + steps + 8
    bb = rv.Model(shape, w, 1, T)
    rivers, build_s = {}, {}
    for name, method in (("rtn", rv.QUANT_RTN), ("hqq", rv.QUANT_HQQ)):
        m_ = rv.Model(shape, w, 1, T)
        m_.set_quantizer(method)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        m_.quantize_river(wl.group, 1)
        build_s[name] = time.perf_counter() - t0
        rivers[name] = m_
    for m_ in (bb, *rivers.values()):
        m_.set_debug(True)
    nb, _ = bb.prefill(prompt, tau, fixed_exit=L)
    for m_ in rivers.values():
        m_.prefill(prompt, wl.prefill_tau)
    tok = int(nb[0])
    full = np.array([L], dtype=np.int32)
    match = {k: 0 for k in rivers}
    kls = {k: [] for k in rivers}
    exits = {k: [] for k in rivers}
    for _ in range(steps):
        ib, _ = bb.decode_step([tok], tau, full)
        lb = bb.dump(rv.DUMP_LOGITS)[0].copy()
        for k, m_ in rivers.items():
            ir, er = m_.decode_step([tok], tau)
            match[k] += int(ib[0] == ir[0])
            kls[k].append(kl_div(lb, m_.dump(rv.DUMP_LOGITS)[0]))
            exits[k].append(int(er[0]))
        tok = int(ib[0])
    bb.close()
    for m_ in rivers.values():
        m_.close()
    out = {"workload": wl_name, "tau": tau, "steps": steps,
           "pages": "98.03% next-token match, KL 0.0045 (trained models)"}
    for k in rivers:
        out[k] = {"next_token_match": match[k] / steps, "kl_mean": float(np.mean(kls[k])),
                  "kl_max": float(np.max(kls[k])), "mean_exit_layer": float(np.mean(exits[k])),
                  "river_build_s": build_s[k]}
        log(f"[fidelity] {wl_name} {k}: match {out[k]['next_token_match']:.3f}, KL mean {out[k]['kl_mean']:.4g}, "
            f"river built in {build_s[k]:.2f} s")
    return out


# ------------------------------------------------------------------ reference arm

def run_reference(wl_name, steps, warmup, budget_s=150.0):
    """The CPU oracle on the host cores: batch-1 decode steps from an empty
    cache (attention over fewer positions is under 1% of a step's work),
    stopping early when the time budget is spent."""
    import oracle

    wl = synth.WORKLOADS[wl_name]
    shape = wl.shape
    w = synth.make_weights(shape)
    nthreads = os.cpu_count() or 1
    om = oracle.Model(shape, w, 1, warmup + steps + 2, nthreads=nthreads)
    om.quantize_river(wl.group, 1)
    tau = wl.taus[0] if wl.taus else 0.90
    tok = int(synth.make_prompt(shape.vocab, 1, 1)[0, 0])
    tok = int(om.decode_step([tok], tau)["next_ids"][0])  # one untimed step
    n, t0 = 0, time.perf_counter()
    while n < steps:
        tok = int(om.decode_step([tok], tau)["next_ids"][0])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    om.close()
    return n, dt, nthreads


# ------------------------------------------------------------------ main

def slowest_over_ranks(ms, e2e_tokens_per_s, device):
    """Replicas: the slowest rank's step time and e2e rate (a barrier, then one
    MAX all-reduce); the whole-job value is world_size tokens per step."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms, 1.0 / e2e_tokens_per_s], dtype=torch.float64, device=device)
    dist.barrier()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0].item()), 1.0 / float(t[1].item())


def layer_us(res, L):
    """River vs backbone layer time (the analogue of the pages' 2.4x): the
    all-river and full-backbone steps minus the LM head's own time, per
    layer (the embedding and step set-up are a few microseconds)."""
    m, k = res["modes"], res["kernels"]
    if "full" not in m or "river" not in m or "lmhead_bf16" not in k:
        return None
    head = k["lmhead_bf16"]["ms"]
    bb = (m["full"]["ms_per_step"] - head) * 1e3 / L
    rv_ = (m["river"]["ms_per_step"] - head) * 1e3 / L
    return {"backbone": bb, "river": rv_, "ratio": bb / rv_, "pages": "exit layers ~2.4x faster than backbone layers"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b", choices=["llama8b", "llama1b", "layer8b"])
    ap.add_argument("--modes", default=",".join(MODES),
                    help="decode modes to time (tau, forced, full, river); the first is the headline")
    ap.add_argument("--engine", default="chain", choices=["chain", "persistent"],
                    help="batch-1 decode engine timed for the headline (the other is timed for comparison)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-fidelity", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batch-64 and 64K-context workloads")
    ap.add_argument("--prompt-len", type=int, default=0,
                    help="override the workload's prompt length (profiling cases, e.g. long-context attention)")
    ap.add_argument("--only", choices=["batch64", "long64k"],
                    help="time only this workload (its own JSON line; for profiling commands)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local = env_rank()
    rank0 = rank == 0

    def log(msg):
        if rank0:
            print(msg, file=sys.stderr, flush=True)

    if args.prompt_len > 0:
        import dataclasses
        synth.WORKLOADS[args.workload] = dataclasses.replace(synth.WORKLOADS[args.workload],
                                                             prompt_len=args.prompt_len)
    wl = synth.WORKLOADS[args.workload]
    tau = wl.taus[0] if wl.taus else 0.90
    cfg = {"workload": f"{wl.shape.name} decode, batch 1, {wl.prompt_len}-token random prompt, tau {tau}, "
                       f"river W4A16 group {wl.group}",
           "layers": wl.shape.n_layers, "d_model": wl.shape.d_model, "ffn": wl.shape.ffn, "vocab": wl.shape.vocab,
           "batch": 1, "prompt_len": wl.prompt_len, "tau": tau, "river_group": wl.group, "engine": args.engine,
           "parallelism": f"replicas{world}" if world > 1 else "single",
           "l2": "inputs larger than L2: every step streams GBs of weights (L2 is 129 MB)"}

    if args.impl == "reference":
        if not rank0:
            return
        n, dt, cores = run_reference(args.workload, args.steps, args.warmup)
        v = n / dt
        line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": n,
                "requested_steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / n * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg, "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": f"{n} oracle decode steps at batch 1 from an empty cache "
                                           f"(150 s budget)"},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import token_level_early_gb300 as rv

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    rv.lib()
    if args.only:
        if not rank0 or world > 1:
            return
        fn = run_batch64 if args.only == "batch64" else run_long64k
        r = fn(args.steps, args.warmup, local, log)
        print(json.dumps({"metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s", "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "config": {"workload": r["workload"]}, args.only: r}), flush=True)
        return
    modes = tuple(x for x in args.modes.split(",") if x in MODES) or MODES
    res = run_workload(args.workload, args.steps, args.warmup, local, not args.no_cpu_baseline, rank0, log, modes,
                       args.engine, want_offload="tau" in modes)
    tau_r = res["modes"][modes[0]]
    ms = tau_r["ms_per_step"]
    e2e = res["e2e_tokens_per_s"]
    if world > 1:
        ms, e2e = slowest_over_ranks(ms, e2e, "cuda")
    sec = None
    if not args.no_secondary and world == 1 and args.workload != "layer8b":
        other = "llama1b" if args.workload == "llama8b" else "llama8b"
        r2 = run_workload(other, args.steps, args.warmup, local, False, rank0, log, MODES, args.engine)
        t2 = r2["modes"]["tau"]
        sec = {"workload": other, "tau": synth.WORKLOADS[other].taus[0], "tokens_per_s": t2["tokens_per_s"],
               "achieved_gbs": t2["achieved_gbs"], "mean_exit_layer": t2["mean_exit_layer"],
               "tau_sweep": r2.get("tau_sweep"),
               "forced_tokens_per_s": r2["modes"]["forced"]["tokens_per_s"],
               "full_backbone_tokens_per_s": r2["modes"]["full"]["tokens_per_s"],
               "all_river_tokens_per_s": r2["modes"]["river"]["tokens_per_s"],
               "e2e_tokens_per_s": r2["e2e_tokens_per_s"], "kernels": r2["kernels"]}
    fid = fidelity(args.workload, 32, local, log) if (rank0 and not args.no_fidelity) else None
    extra = {}
    if rank0 and world == 1 and not args.no_extra and args.workload == "llama8b":
        extra["batch64"] = run_batch64(min(args.steps, 128), args.warmup, local, log)
        extra["long64k"] = run_long64k(min(args.steps, 64), args.warmup, local, log)
    if not rank0:
        return
    peak, peak_kind = peak_hbm()

    def roof_of(name, kernel, path):
        k = res["kernels"][name]
        return {"bound": "hbm", "kernel": kernel, "achieved": k["gbs"], "peak": peak, "unit": "GB/s",
                "frac": k["gbs"] / peak,
                "peak_source": f"{peak_kind} HBM copy bandwidth (MEASURED_PEAKS.json hbm_gbs), burst",
                "traffic": profile_traffic(path), "bytes_per_launch": k["bytes"], "ms_per_launch": k["ms"]}

    # the dominant kernel of the headline (tau) step is the river's gate/up:
    # most of its layers run in the river
    roof = roof_of("gateup_int4", "k_gemv_b1<int4 river weights, RMSNorm prologue, SwiGLU epilogue> "
                                  "(gate/up, layer 1)", "int4")
    roof_bb = roof_of("gateup_bf16", "k_gemv_b1<bf16, RMSNorm prologue, SwiGLU epilogue> (gate/up, layer 1)",
                      "bf16")
    L = wl.shape.n_layers
    modes = {m_: {k_: v_ for k_, v_ in r.items() if k_ != "clocks"} for m_, r in res["modes"].items()}
    line = {"metric": METRIC, "value": world * 1e3 / ms, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": cfg,
            "achieved_gbs": tau_r["achieved_gbs"], "achieved_frac_of_measured_hbm": tau_r["achieved_gbs"] / peak,
            "mean_exit_layer": tau_r["mean_exit_layer"], "prefill_exit_layer": res["prefill_exit"],
            "modes": modes,
            "speedup_vs_full_backbone": (tau_r["tokens_per_s"] / res["modes"]["full"]["tokens_per_s"]
                                         if "full" in res["modes"] else None),
            "layer_us": layer_us(res, L),
            "roofline": roof, "roofline_backbone": roof_bb,
            "step_roofline": {"achieved": tau_r["achieved_gbs"], "peak": peak, "unit": "GB/s",
                              "frac": tau_r["achieved_gbs"] / peak,
                              "what": "algorithmic bytes of the whole tau step / its time"},
            "kernels": res["kernels"], "cpu_baseline": res["cpu"], "offload": res["offload"],
            "fidelity": fid,
            "e2e": {"value": world * e2e, "unit": "tokens/s", "h2d_bytes_per_step": 4 * 6,
                    "d2h_bytes_per_step": 4 * 4},
            # per step: the scalar-setting kernel, then the captured chain (step init, embedding, five
            # kernels per layer, LM head) or the one persistent kernel
            "gpu_launches": args.steps * ((5 * L + 4) if args.engine == "chain" else 2), "clocks": tau_r.get("clocks"),
            "dtype_detail": "bf16 weights/activations/KV, int4 river weights with fp16 scale/zero, fp32 accumulation"}
    if sec:
        line["secondary"] = sec
    if extra:
        line.update(extra)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
