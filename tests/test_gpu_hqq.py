"""GPU parity of the HQQ river quantizer (Badri and Shaji 2023, half-quadratic
quantization; the pages' river quantizer, paperlayer.ai appendix A.1).

Every HQQ step is IEEE fp32 arithmetic in a fixed order on both sides, so the
packed codes, fp16 scales and fp16 zeros are compared bit for bit:

- tiny (fp16, ragged down-projection groups): every layer, all 7 projections,
  then decode parity with the HQQ river against the oracle's HQQ river;
- Llama-3.2-1B shape (bf16, group 128): the first and last layer, all 7
  projections, on sampled rows the oracle quantizes group by group."""
import time

import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv
from gpu_util import log, sampled_step
from ongrid import unpack_canonical

pytestmark = pytest.mark.gpu
PROJ_TENSOR = (1, 2, 3, 4, 6, 7, 8)  # RV_PROJ_* -> position in a layer's weight list


def layer_matrix(w, layer, proj):
    return w[3 + 9 * (layer - 1) + PROJ_TENSOR[proj]]


def test_hqq_tiny_bit_exact_and_decode():
    shape = synth.TINY
    L = shape.n_layers
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 1, 64)
    om = oracle.Model(shape, w, 1, 64)
    gr = rv.Model(shape, w, 1, 8)
    gm.set_quantizer(rv.QUANT_HQQ)
    assert om.set_quantizer(1) == 0
    gm.quantize_river(64, 1)
    om.quantize_river(64, 1)
    gr.quantize_river(64, 1)  # RTN, for contrast
    moved = 0
    for layer in range(1, L + 1):
        for proj in range(7):
            g = gm.export_river(layer, proj)
            o = om.export_river(layer, proj)
            for a, b in zip(g, o):
                assert np.array_equal(a, b), (layer, proj)
            r = gr.export_river(layer, proj)
            assert np.array_equal(g[1], r[1])  # the same min/max scale
            moved += int((g[2] != r[2]).sum())
    assert moved > 0  # HQQ moved zeros off RTN's integer ones
    gr.close()

    gm.set_debug(True)
    prompt = synth.make_prompt(shape.vocab, 1, 24, seed=31)
    g_next, g_exit = gm.prefill(prompt, 0.5)
    o = om.prefill(prompt, 0.5, tf_exit=g_exit, tf_ids=g_next, debug=True)
    assert o["exit_layer"][0] == g_exit[0] and o["next_ids"][0] == g_next[0]
    tok = [int(g_next[0])]
    exits = []
    for step in range(8):
        tau = (0.3, 0.9, 0.6, 2.0)[step % 4]
        forced = np.array([step % (L + 1)], dtype=np.int32) if step in (3, 7) else None
        nxt, ex = sampled_step(gm, om, tok, tau, forced, 1, L, shape.act_dtype, 1, f"hqq:tiny:{step}")
        exits.append(int(ex[0]))
        tok = [int(nxt[0])]
    assert min(exits) < L
    gm.close()
    om.close()


def test_hqq_llama1b_sampled_rows():
    wl = synth.WORKLOADS["llama1b"]
    shape = wl.shape
    L, act, g = shape.n_layers, shape.act_dtype, wl.group
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 1, 16)
    gm.set_quantizer(rv.QUANT_HQQ)
    t0 = time.perf_counter()
    gm.quantize_river(g, 1)
    t_hqq = time.perf_counter() - t0
    rng = np.random.default_rng(9)
    groups = 0
    for layer in (1, L):
        for proj in range(7):
            q, s, z = gm.export_river(layer, proj)
            codes = unpack_canonical(q)
            W = layer_matrix(w, layer, proj)
            N, K = W.shape
            for n in rng.choice(N, 6, replace=False):
                for gi in range(-(-K // g)):
                    oq, os_, oz, rc = oracle.hqq_group(W[n, gi * g:(gi + 1) * g], act)
                    assert rc == 0
                    assert np.array_equal(codes[n, gi * g:gi * g + oq.size], oq), (layer, proj, n, gi)
                    assert int(s[n, gi]) == os_ and int(z[n, gi]) == oz, (layer, proj, n, gi)
                    groups += 1
    log({"tag": "hqq:llama1b", "groups_checked": groups, "quantize_s": t_hqq})
    gm.close()
