"""The allocation-free greedy LM head must give what the decode step gives.

rv_greedy_head_noalloc is for callers that may not allocate device memory;
it keeps its cross-block scratch in an array built into the library.  Here it
is fed the decode step's own final hidden state and must reproduce that
step's greedy id and logits, on two calls in a row (the second call reuses
the array the first one left behind).  This file is collected last."""
import numpy as np
import pytest

import oracle
import synth
import token_level_early_gb300 as rv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "llama1b"])
def test_noalloc_head_matches_decode_step(name):
    import torch

    wl = synth.WORKLOADS[name]
    shape = wl.shape
    L, V, d = shape.n_layers, shape.vocab, shape.d_model
    w = synth.make_weights(shape)
    gm = rv.Model(shape, w, 1, 16)
    gm.quantize_river(wl.group, 1)
    gm.set_debug(True)
    head = w[0] if shape.tied_embed else w[2]
    d_head = torch.from_numpy(head.view(np.int16)).cuda()
    d_norm = torch.from_numpy(w[1].view(np.int16)).cuda()
    d_next = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d_logits = torch.zeros(V, dtype=torch.float32, device="cuda")
    tok = 5
    for _ in range(2):
        nxt, _ = gm.decode_step([tok], 0.9)
        h = torch.from_numpy(gm.dump(rv.DUMP_HIDDEN)[L, 0].copy()).cuda()
        ref = gm.dump(rv.DUMP_LOGITS)[0]
        torch.cuda.synchronize()
        rv.greedy_head_noalloc(d_head.data_ptr(), d_norm.data_ptr(), h.data_ptr(), V, d, shape.act_dtype,
                               shape.rms_eps, d_next.data_ptr(), d_logits.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert int(d_next.item()) == int(nxt[0])
        assert np.abs(d_logits.cpu().numpy() - ref).max() <= 5e-2
        tok = int(nxt[0])
    gm.close()


def test_noalloc_head_rejects_sizes_beyond_its_limits():
    import torch

    buf = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = buf.data_ptr()
    for vocab, dm in ((6, 256), (1024, 16392), (1024, 12)):
        with pytest.raises(rv.RVError) as e:
            rv.greedy_head_noalloc(p, p, p, vocab, dm, 1, 1e-5, p, None, None)
        assert e.value.code == rv.RV_EINVAL


@pytest.mark.parametrize("d_model,vocab", [(16384, 1024), (264, 256)])
def test_noalloc_head_synthetic_shapes_against_oracle(d_model, vocab):
    """Shapes no model of the decode step uses: the advertised maximum width
    (16384) and a width that is a multiple of 8 but not of 32.  Random hidden
    state, RMSNorm gain and LM head; the greedy id must equal the oracle's
    (unless the oracle's top two logits are within 1e-2) and the logits must
    agree within 5e-2."""
    import torch

    shape = synth.ModelShape(f"head-{d_model}", 1, d_model, 1, 1, 8, 8, vocab, 0, synth.BF16)
    w = synth.make_weights(shape, seed=21)
    rng = np.random.default_rng(5)
    gain = (1.0 + 0.1 * rng.standard_normal(d_model)).astype(np.float32)
    w[1] = (gain.view(np.uint32) >> 16).astype(np.uint16)  # bf16 bits (truncated: any 16-bit value will do)
    h = rng.standard_normal((1, d_model)).astype(np.float32)
    om = oracle.Model(shape, w, 1, 2)
    ol, oid = om.head(h.astype(np.float64))
    om.close()
    d_head = torch.from_numpy(w[2].view(np.int16)).cuda()
    d_norm = torch.from_numpy(w[1].view(np.int16)).cuda()
    d_h = torch.from_numpy(h[0].copy()).cuda()
    d_next = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    d_logits = torch.zeros(vocab, dtype=torch.float32, device="cuda")
    for _ in range(2):  # two calls in a row on the shared scratch array
        d_next.fill_(-1)
        torch.cuda.synchronize()
        rv.greedy_head_noalloc(d_head.data_ptr(), d_norm.data_ptr(), d_h.data_ptr(), vocab, d_model, synth.BF16,
                               shape.rms_eps, d_next.data_ptr(), d_logits.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        logits = d_logits.cpu().numpy()
        assert np.abs(logits - ol[0]).max() <= 5e-2
        top2 = np.sort(ol[0])[-2:]
        if top2[1] - top2[0] >= 1e-2:
            assert int(d_next.item()) == int(oid[0])
        else:
            assert ol[0][int(d_next.item())] >= top2[1] - 1e-2
