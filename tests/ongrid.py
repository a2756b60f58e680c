"""Test helper: weights that lie exactly on the int4 round-to-nearest grid.

Each group of g weights along a row is w = (q - z) * s with s a power of two
(so every w is exact in the 16-bit type), z an integer in 0..15 and q in
0..15 with both 0 and 15 present (so the group's min and max pin s and z).
Quantizing such a group must give back exactly (q, s, z).
"""
import numpy as np


def ongrid_matrix(rng, N: int, K: int, g: int, act: int):
    G = -(-K // g)
    q = rng.integers(0, 16, size=(N, K)).astype(np.int64)
    s_exp = rng.integers(6, 10, size=(N, G))
    z = rng.integers(0, 16, size=(N, G)).astype(np.int64)
    for n in range(N):
        for gi in range(G):
            k0, k1 = gi * g, min(K, (gi + 1) * g)
            pos = rng.permutation(np.arange(k0, k1))[:2]
            q[n, pos[0]] = 0
            q[n, pos[1]] = 15
    s = np.ldexp(1.0, -s_exp)
    s_full = np.repeat(s, g, axis=1)[:, :K]
    z_full = np.repeat(z, g, axis=1)[:, :K]
    w = (q - z_full) * s_full
    if act == 0:
        bits = w.astype(np.float16).view(np.uint16)
        assert np.array_equal(bits.view(np.float16).astype(np.float64), w)
    else:
        import torch
        bits = torch.from_numpy(w.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    s_bits = s.astype(np.float16).view(np.uint16)
    z_bits = z.astype(np.float16).view(np.uint16)
    return bits, q.astype(np.uint8), s_bits, z_bits


def pack_canonical(q: np.ndarray) -> np.ndarray:
    """Reference packing written from the documented layout: word w of a row
    holds q[8w + j] in bits 4j..4j+3."""
    N, K = q.shape
    out = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(8):
        out |= (q[:, j::8].astype(np.uint32) & 0xF) << (4 * j)
    return out


def unpack_canonical(p: np.ndarray) -> np.ndarray:
    N, W = p.shape
    q = np.zeros((N, W * 8), dtype=np.uint8)
    for j in range(8):
        q[:, j::8] = (p >> (4 * j)) & 0xF
    return q


def ongrid_weights(shape, g: int, seed: int = 0):
    """Full weight list (synth order) with every projection on the grid; RMSNorm
    gains random in [0.5, 1.5); embeddings N(0, 0.02)."""
    import synth

    rng = np.random.default_rng(seed)
    act = shape.act_dtype
    ws = synth.make_weights(shape, seed=seed + 100)
    truth = {}
    shapes = synth.tensor_shapes(shape)
    for l in range(shape.n_layers):
        for j, name in enumerate(synth.LAYER_TENSORS):
            tid = 3 + 9 * l + j
            shp = shapes[tid]
            if len(shp) == 1:
                gam = rng.uniform(0.5, 1.5, shp[0])
                if act == 0:
                    ws[tid] = gam.astype(np.float16).view(np.uint16)
                else:
                    import torch
                    ws[tid] = torch.from_numpy(gam.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
                continue
            bits, q, s, z = ongrid_matrix(rng, shp[0], shp[1], g, act)
            ws[tid] = bits
            truth[(l + 1, name)] = (q, s, z)
    return ws, truth
