"""CPU checks of the benchmark's byte accounting (achieved GB/s divides these
by the device time) against the per-layer and per-token figures derived from
the model shapes in the scope table: 8B shape 436.21 MB of weights per
backbone layer, 115.87 MB per river layer (g = 128), 15.01 GB per
full-backbone token at empty context; 1B shape 121.63 MB, 32.31 MB, 2.47 GB.
The bench also counts each layer's two RMSNorm gains."""
import importlib.util
import os

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("shape,bb_mb,rv_mb,full_gb", [
    (synth.LLAMA_8B, 436.21, 115.87, 15.01),
    (synth.LLAMA_1B, 121.63, 32.31, 2.47),
])
def test_layer_and_token_bytes(bench, shape, bb_mb, rv_mb, full_gb):
    bb, rv = bench.layer_bytes(shape, 128)
    norms = 2 * 2 * shape.d_model  # the layer's two 16-bit RMSNorm gains, read by both paths
    assert abs((bb - norms) / 1e6 - bb_mb) < 0.01 and abs((rv - norms) / 1e6 - rv_mb) < 0.01
    L = shape.n_layers
    full = bench.token_bytes(shape, 128, L, 0)
    assert abs(full / 1e9 - full_gb) < 0.01
    # each layer moved from the backbone to the river saves bb - rv bytes
    assert bench.token_bytes(shape, 128, L - 1, 0) == full - (bb - rv)
    # one more cached position adds one K/V read of every layer
    kv_pos = L * 2 * shape.n_kv_heads * shape.head_dim * 2
    assert bench.token_bytes(shape, 128, L, 100) - bench.token_bytes(shape, 128, L, 99) == kv_pos


def test_layer_us(bench):
    res = {"modes": {"full": {"ms_per_step": 2.8}, "river": {"ms_per_step": 1.8}},
           "kernels": {"lmhead_bf16": {"ms": 0.2}}}
    lu = bench.layer_us(res, 32)
    assert lu["backbone"] == pytest.approx(2600 / 32) and lu["river"] == pytest.approx(1600 / 32)
    assert lu["ratio"] == pytest.approx(2.6 / 1.6)
    assert bench.layer_us({"modes": {"tau": {}}, "kernels": {}}, 32) is None


def test_profile_traffic_follows_kernel_hash(bench, tmp_path, monkeypatch):
    f = tmp_path / "p.md"
    f.write_text(f"- kernel_source_sha256: {bench.kernel_hash()}\n- traffic_bytes_per_launch_int4: 123\n"
                 "- traffic_bytes_per_launch_bf16: 456\n")
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(f))
    assert bench.profile_traffic("int4") == 123.0
    assert bench.profile_traffic("bf16") == 456.0
    f.write_text("- kernel_source_sha256: 0000000000000000\n- traffic_bytes_per_launch_int4: 123\n")
    assert bench.profile_traffic("int4") is None
