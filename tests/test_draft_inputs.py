"""Host checks of the random-weight draft fixture (synth/draft.py), the input
source of the in-situ scoring tests: its rotary embedding and QK-norm behave
as their definitions say, its output is deterministic, and its block-paged
cache holds exactly the dense keys (the oracle's own gather of the pages)."""

import numpy as np

import oracle
from synth import DraftShape, draft_attention_inputs, page_keys
from synth.draft import rms_normalize, rope
from synth.inputs import f32_from_bf16_bits


def test_rope_identity_norm_and_relative_position():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 2, 64)).astype(np.float32)
    y = rng.standard_normal((7, 2, 64)).astype(np.float32)
    # position 0 is the identity
    assert np.array_equal(rope(x[:1], np.array([0]), 32, 1e4), x[:1])
    # rotation keeps the norm; dimensions past rotary_dim are untouched
    r = rope(x, np.arange(7) * 37, 32, 1e4)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-5)
    assert np.array_equal(r[..., 32:], x[..., 32:])
    # <rope(x, m), rope(y, n)> depends on m - n only
    for m, n in ((5, 2), (1000, 997), (3, 0)):
        a = np.sum(rope(x, np.full(7, m), 32, 1e4) * rope(y, np.full(7, n), 32, 1e4), axis=-1)
        b = np.sum(rope(x, np.full(7, m - n), 32, 1e4) * y, axis=-1)
        np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-4)


def test_qk_norm_gives_unit_rms():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((10, 3, 256)).astype(np.float32) * 7.0
    ms = np.mean(rms_normalize(x, 1e-6).astype(np.float64) ** 2, axis=-1)
    np.testing.assert_allclose(ms, 1.0, rtol=1e-5)


def test_fixture_is_deterministic_and_shaped():
    shape = DraftShape(hidden=128, n_layers=2, head_dim=64, rotary_dim=16, n_lookahead=3, seed=9)
    q1, k1, off1 = draft_attention_inputs(shape, [40, 0, 17])
    q2, k2, off2 = draft_attention_inputs(shape, [40, 0, 17])
    assert q1.shape == (3, 2, 3, 8, 64) and k1.shape == (2, 57, 2, 64)
    assert list(off1) == [0, 40, 40, 57]
    assert np.array_equal(q1, q2) and np.array_equal(k1, k2)
    assert not np.array_equal(k1[0], k1[1])          # layers have their own weights
    # post-norm keys: per-head RMS near the gain's RMS (about 1)
    kf = f32_from_bf16_bits(k1).astype(np.float64)
    assert 0.8 < np.sqrt(np.mean(kf ** 2)) < 1.2


def test_paged_cache_holds_the_dense_keys():
    shape = DraftShape(hidden=64, n_layers=2, head_dim=64, rotary_dim=16, n_lookahead=2, seed=3)
    _, k, off = draft_attention_inputs(shape, [33, 1, 0, 50])
    for bs in (8, 16, 32):
        pools, table = page_keys(k, off, bs, seed=1)
        assert pools[0].shape[1:] == (bs, 2, 64) and table.dtype == np.int32
        used = np.concatenate([table[b, :(int(off[b + 1] - off[b]) + bs - 1) // bs] for b in range(4)])
        assert len(np.unique(used)) == len(used) == pools[0].shape[0]   # every block once
        assert np.array_equal(oracle.kv_from_pages(pools, table, off, bs), k)
