"""The allocation-free greedy LM head must give what the decode step gives.

rv_greedy_head_noalloc is for callers that may not allocate device memory;
it keeps its cross-block scratch in an array built into the library.  Here it
is fed the decode step's own final hidden state and must reproduce that
step's greedy id and logits, on two calls in a row (the second call reuses
the array the first one left behind).  This file is collected last."""
import numpy as np
import pytest

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
