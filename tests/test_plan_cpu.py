"""The decode attention's launch plan (rv_decode_attention_plan: host
arithmetic only, no GPU work).  The decode step keys its captured graph by
this plan, and the GPU plan test (tests/test_gpu_attention_plans.py) crosses
the 8B shape's switch between 2048 and 2049 cached positions.  Concrete
cases worked out by hand from the rule stated in include/rv.h, then bounds
and monotonicity over a sweep."""
import ctypes

import pytest

import token_level_early_gb300 as rv

N_SM = 152  # SMs of a GB300


def plan(batch, hkv, n_sm, max_cluster, max_splits, context):
    return rv.decode_attention_plan(batch, hkv, n_sm, max_cluster, max_splits, context)


def test_llama_shapes_switch_past_2048_positions():
    # 8 KV heads, one row: a cluster of 16 splits (16 x 8 = 128 blocks <= 304);
    # each split's 4 warps take at most one 32-position tile while the
    # context is <= 16 x 4 x 32 = 2048 positions
    assert plan(1, 8, N_SM, 16, 38, 0) == (0, 16)
    assert plan(1, 8, N_SM, 16, 38, 1100) == (0, 16)
    assert plan(1, 8, N_SM, 16, 38, 2048) == (0, 16)
    # past it: 152 / 8 = 19 blocks per KV head, merged through global memory
    assert plan(1, 8, N_SM, 16, 38, 2049) == (1, 19)
    assert plan(1, 8, N_SM, 16, 38, 65536) == (1, 19)


def test_smaller_clusters_switch_earlier():
    # a device whose largest cluster is 8: 8 x 4 x 32 = 1024 positions
    assert plan(1, 8, N_SM, 8, 38, 1024) == (0, 8)
    assert plan(1, 8, N_SM, 8, 38, 1025) == (1, 19)
    assert plan(1, 8, N_SM, 1, 38, 128) == (0, 1)
    assert plan(1, 8, N_SM, 1, 38, 129) == (1, 19)


def test_batches_shrink_the_cluster():
    # 4 rows x 8 KV heads = 32 (row, head) pairs: the cluster doubles while
    # the doubled grid stays within two blocks per SM (2 x cs x 32 <= 304:
    # 1 -> 2 -> 4 -> 8; 16 would need 512 blocks), so clusters of 8 and the
    # switch at 8 x 4 x 32 = 1024 positions
    assert plan(4, 8, N_SM, 16, 38, 1024) == (0, 8)
    assert plan(4, 8, N_SM, 16, 38, 1025) == (1, 4)  # 152 // 32 = 4 blocks per pair
    # 2 rows: 16 pairs, clusters of 16 (256 blocks), switch at 2048
    assert plan(2, 8, N_SM, 16, 38, 2048) == (0, 16)
    assert plan(2, 8, N_SM, 16, 38, 2049) == (1, 9)  # 152 // 16 = 9


def test_rows_that_fill_the_gpu_keep_the_cluster_plan():
    # 64 rows x 8 KV heads = 512 pairs > 152: one block per pair, no split,
    # whatever the context
    for ctx in (0, 256, 4096, 65536):
        assert plan(64, 8, N_SM, 16, 38, ctx) == (0, 1)
    # 10 rows x 8 = 80 pairs: 152 // 80 = 1 < 2 blocks per pair
    assert plan(10, 8, N_SM, 16, 38, 65536)[0] == 0


def test_split_cap():
    # one KV head: 152 blocks would be possible, the caller's cap and the
    # library's 128 bound them
    assert plan(1, 1, N_SM, 16, 38, 100000) == (1, 38)
    assert plan(1, 1, N_SM, 16, 500, 100000) == (1, 128)
    assert plan(1, 1, N_SM, 16, 1, 100000) == (1, 1)


def test_bounds_and_monotonicity_over_a_sweep():
    for n_sm in (132, 148, 152):
        for batch in (1, 2, 3, 4, 8, 16, 64):
            for hkv in (1, 2, 4, 8):
                for mc in (1, 2, 4, 8, 16):
                    seen_global = False
                    for ctx in list(range(0, 4200, 37)) + [8191, 8192, 16384, 65536, 131072]:
                        p, s = plan(batch, hkv, n_sm, mc, 64, ctx)
                        assert p in (0, 1)
                        if p == 0:
                            assert not seen_global, (n_sm, batch, hkv, mc, ctx)  # never back
                            assert s >= 1 and s & (s - 1) == 0 and s <= mc
                            assert s == 1 or s * hkv * batch <= 2 * n_sm
                        else:
                            seen_global = True
                            assert 2 <= s <= min(64, 128, n_sm // (hkv * batch))


def test_rejects_bad_arguments_before_any_work():
    lib = rv.lib()
    out = ctypes.c_int(0)
    E = rv.RV_EINVAL
    assert lib.rv_decode_attention_plan(1, 8, N_SM, 16, 38, 100, None) == E
    for args in ((0, 8, N_SM, 16, 38, 100), (1, 0, N_SM, 16, 38, 100), (1, 8, 0, 16, 38, 100),
                 (1, 8, N_SM, 16, 0, 100), (1, 8, N_SM, 16, 38, -1), (1, 8, N_SM, 3, 38, 100),
                 (1, 8, N_SM, 32, 38, 100), (1, 8, N_SM, 0, 38, 100)):
        assert lib.rv_decode_attention_plan(*args, ctypes.byref(out)) == E, args
    with pytest.raises(rv.RVError):
        plan(0, 8, N_SM, 16, 38, 100)
