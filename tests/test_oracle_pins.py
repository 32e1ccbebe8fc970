"""Pins of the float64 oracle against things other than itself.

Each test checks the oracle against the brute-force twin (independent
pure-Python loops and subset enumeration), a library routine (scipy/torch
softmax, numpy convolution), a closed form, or an invariant the method's
definition implies. CPU only.
"""

import math

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import bruteforce
from oracle import specprefill_oracle as so
from synth import bf16_bits_from_f32, get_workload, make_inputs
from tests._cases import random_case

TINY_CASES = [
    # lengths, Ly, Hq, Hk, d, L, params
    dict(lengths=[40], shape=(1, 2, 1, 8, 2), q_gain=3.0,
         params=dict(pool_w=3, chunk=4, mode="fixed", keep_p=0.3, normalize=False,
                     boost_first_mult=1.0, boost_last_mult=1.0)),
    dict(lengths=[37, 23], shape=(2, 4, 2, 4, 3), q_gain=2.0,
         params=dict(pool_w=5, chunk=4, mode="mass", mass=0.6, normalize=True,
                     boost_first_mult=1.5, boost_first_n=5, boost_last_mult=1.3, boost_last_n=7)),
    dict(lengths=[45], shape=(2, 2, 2, 6, 1), q_gain=2.5,
         params=dict(pool_w=13, chunk=5, mode="mass", mass=0.85, normalize=True,
                     boost_first_mult=1.5, boost_first_n=8, boost_last_mult=1.3, boost_last_n=9)),
    dict(lengths=[1, 2, 30], shape=(1, 2, 1, 4, 2), q_gain=2.0,
         params=dict(pool_w=13, chunk=3, mode="fixed", keep_p=0.15, normalize=True,
                     boost_first_mult=2.0, boost_first_n=2, boost_last_mult=1.25, boost_last_n=3)),
    dict(lengths=[33, 19], shape=(1, 3, 3, 5, 2), q_gain=1.5,
         params=dict(pool_w=7, chunk=4, mode="fixed", keep_p=0.5, normalize=False,
                     boost_first_mult=1.5, boost_first_n=4, boost_last_mult=1.3, boost_last_n=4,
                     force_bos=False, force_last_chunk=False, scale=0.37)),
]


def _case(i):
    c = TINY_CASES[i]
    ly, hq, hk, d, steps = c["shape"]
    q, k, off = random_case(100 + i, c["lengths"], ly, hq, hk, d, steps, q_gain=c["q_gain"])
    return q, k, off, c["params"]


@pytest.mark.parametrize("i", range(len(TINY_CASES)))
def test_oracle_matches_bruteforce(i):
    q, k, off, params = _case(i)
    got = oracle.run(q, k, off, **params)
    want = bruteforce.run_bruteforce(q, k, off, **params)
    for key in ("imp", "tok_score", "final_score", "chunk_score"):
        np.testing.assert_allclose(got[key], want[key], rtol=1e-12, atol=1e-15, err_msg=key)
    for key in ("chunk_keep", "kept_idx", "kept_pos", "kept_off"):
        np.testing.assert_array_equal(np.asarray(got[key]), np.asarray(want[key]), err_msg=key)


def test_single_row_is_textbook_softmax():
    """Ly=Hq=Hk=L=1, W=1, no normalisation/boost: imp is one softmax row."""
    q, k, off = random_case(7, [300], 1, 1, 1, 64, 1, q_gain=2.0)
    out = oracle.run(q, k, off, pool_w=1, chunk=32, normalize=False,
                     boost_first_mult=1.0, boost_last_mult=1.0)
    qf = so.decode_bf16(q[0, 0, 0, 0])
    kf = so.decode_bf16(k[0, :, 0, :])
    logits = kf @ qf / 8.0
    np.testing.assert_allclose(out["imp"], scipy.special.softmax(logits), rtol=1e-13, atol=0)
    np.testing.assert_allclose(out["tok_score"], out["imp"], rtol=0, atol=0)


def test_softmax_rows_sum_to_one_and_importance_bounds():
    q, k, off = random_case(8, [257], 3, 4, 2, 16, 3, q_gain=3.0)
    for layer in range(3):
        for g in range(2):
            p = oracle.attention_rows(q[0], k, 0, 257, layer, g, 2)
            assert p.shape == (3, 2, 257)
            assert np.all(p > 0)
            np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
    a = oracle.step_importance(q[0], k, 0, 257, 2)
    sums = a.sum(axis=1)
    assert np.all(sums >= 1.0 - 1e-12) and np.all(sums <= 3 * 4 + 1e-12)


def test_importance_permutation_invariance():
    q, k, off = random_case(9, [200], 3, 6, 2, 8, 2, q_gain=2.0)
    base = oracle.run(q, k, off)["imp"]
    # permute query heads inside each group of 3
    perm = np.array([2, 0, 1, 4, 5, 3])
    assert np.array_equal(oracle.run(q[:, :, :, perm], k, off)["imp"], base)
    # permute layers (queries and keys together)
    lp = np.array([1, 2, 0])
    assert np.array_equal(oracle.run(q[:, lp], k[lp], off)["imp"], base)
    # swap KV heads together with their query groups
    assert np.array_equal(oracle.run(q[:, :, :, [3, 4, 5, 0, 1, 2]], k[:, :, ::-1], off)["imp"], base)


def test_pool_properties():
    rng = np.random.default_rng(3)
    v = rng.random(101)
    # W = 1 is the identity
    np.testing.assert_array_equal(oracle.avg_pool(v, 1), v)
    # constant in -> same constant out, including the edges
    np.testing.assert_allclose(oracle.avg_pool(np.full(50, 0.25), 13), 0.25, rtol=1e-15)
    np.testing.assert_allclose(oracle.avg_pool(np.full(5, 0.5), 13), 0.5, rtol=1e-15)
    # interior equals numpy's convolution with a box kernel
    w = 13
    interior = np.convolve(v, np.ones(w), mode="valid") / w
    np.testing.assert_allclose(oracle.avg_pool(v, w)[w // 2:-(w // 2)], interior, rtol=1e-14)
    # edges divide by the number of in-range tokens
    x = oracle.avg_pool(v, w)
    assert math.isclose(x[0], v[:7].mean(), rel_tol=1e-14)
    assert math.isclose(x[3], v[:10].mean(), rel_tol=1e-14)
    assert math.isclose(x[-1], v[-7:].mean(), rel_tol=1e-14)


def test_pool_of_prompt_within_one_window_is_exactly_constant():
    """When every window covers the whole prompt (n <= W//2 + 1) all pooled
    values are the same mean, exactly; normalisation then gives all ones."""
    rng = np.random.default_rng(5)
    for n in range(1, 8):
        v = rng.random(n) * 1e-3
        x = oracle.avg_pool(v, 13)
        assert np.all(x == x[0])
        assert math.isclose(x[0], math.fsum(v) / n, rel_tol=1e-15)
        np.testing.assert_array_equal(oracle.min_max_normalize(x), np.ones(n))


def test_normalize_closed_form():
    np.testing.assert_allclose(oracle.min_max_normalize(np.array([2.0, 4.0, 6.0, 3.0])),
                               [0.0, 0.5, 1.0, 0.25], rtol=0, atol=0)
    np.testing.assert_array_equal(oracle.min_max_normalize(np.full(7, 3.5)), np.ones(7))
    y = oracle.min_max_normalize(np.random.default_rng(1).random(99))
    assert y.min() == 0.0 and y.max() == 1.0


def test_boost_positions():
    n = 300
    y = oracle.structural_boost(np.ones(n), 1.5, 64, 1.3, 128)
    f13 = float(np.float32(1.3))
    assert y[0] == 1.5 and y[63] == 1.5 and y[64] == 1.0
    assert y[n - 129] == 1.0 and y[n - 128] == f13 and y[n - 1] == f13
    # overlap (n < 192): both factors apply
    y = oracle.structural_boost(np.ones(100), 1.5, 64, 1.3, 128)
    assert y[0] == 1.5 * f13 and y[63] == 1.5 * f13 and y[64] == f13


def test_uniform_attention_gives_equal_chunks():
    """Q = 0 makes every softmax row uniform, so imp = 1/n everywhere and every
    chunk (partial last one included) scores 1/n. With n = 128 every step is
    exact in binary floating point, so the chunk scores tie exactly."""
    n = 128
    q = np.zeros((1, 2, 3, 4, 16), dtype=np.uint16)  # bf16 +0.0
    _, k, off = random_case(11, [n], 2, 4, 2, 16, 3)
    out = oracle.run(q, k, off, pool_w=13, chunk=48, normalize=False,
                     boost_first_mult=1.0, boost_last_mult=1.0, mode="fixed", keep_p=0.3)
    assert np.all(out["imp"] == 1.0 / n)
    assert np.all(out["tok_score"] == 1.0 / n)
    assert np.all(out["chunk_score"] == 1.0 / n)
    # exact ties break by ascending index: k = ceil(3 * 0.3) = 1 -> chunk 0,
    # plus the forced final (partial) chunk
    np.testing.assert_array_equal(out["chunk_keep"], [1, 0, 2])
    np.testing.assert_array_equal(out["kept_idx"], list(range(48)) + list(range(96, 128)))
    # mass mode with equal scores keeps the first ceil(mass * nc) chunks
    out = oracle.run(q, k, off, pool_w=13, chunk=16, normalize=False,
                     boost_first_mult=1.0, boost_last_mult=1.0, mode="mass", mass=0.5)
    np.testing.assert_array_equal(out["chunk_keep"], [1, 1, 1, 1, 0, 0, 0, 2])


def test_fixed_count_closed_forms():
    assert oracle.fixed_count(16, 0.30) == 5
    assert oracle.fixed_count(1024, 0.15) == 154
    assert oracle.fixed_count(4096, 0.30) == 1229
    assert oracle.fixed_count(10, 1.0) == 10
    assert oracle.fixed_count(10, 1e-6) == 1
    assert oracle.fixed_count(20, 0.5) == 10  # exact product


def test_fixed_mode_ignores_normalisation_without_boost():
    q, k, off = random_case(12, [500, 333], 2, 4, 2, 16, 2, q_gain=2.0)
    kw = dict(pool_w=13, chunk=16, mode="fixed", keep_p=0.25, boost_first_mult=1.0,
              boost_last_mult=1.0)
    a = oracle.run(q, k, off, normalize=False, **kw)
    b = oracle.run(q, k, off, normalize=True, **kw)
    np.testing.assert_array_equal(a["chunk_keep"], b["chunk_keep"])


def test_mass_extremes():
    cs = np.array([0.3, 0.1, 0.5, 0.05, 0.2])
    assert oracle.select_mass(cs, 1.0).all()
    np.testing.assert_array_equal(oracle.select_mass(cs, 1e-6), [False, False, True, False, False])
    # 0.5 + 0.3 = 0.8 of 1.15 total < 0.85 * 1.15, so 0.2 is added
    np.testing.assert_array_equal(oracle.select_mass(cs, 0.85), [True, False, True, False, True])
    assert oracle.select_mass(np.zeros(4), 0.5).all()


@pytest.mark.parametrize("seed", range(12))
def test_selection_matches_subset_enumeration(seed):
    rng = np.random.default_rng(seed)
    nc = int(rng.integers(1, 13))
    if seed % 3 == 0:
        cs = rng.integers(0, 4, nc).astype(np.float64)  # many ties
    else:
        cs = rng.random(nc)
    for p in (0.1, 0.3, 0.5, 1.0):
        got = np.flatnonzero(oracle.select_fixed(cs, p))
        assert got.tolist() == bruteforce._select(cs.tolist(), "fixed", p, 0.0)
    for m in (0.2, 0.5, 0.85, 1.0):
        got = np.flatnonzero(oracle.select_mass(cs, m))
        assert got.tolist() == bruteforce._select(cs.tolist(), "mass", 0.0, m)


def test_kept_list_invariants():
    q, k, off = random_case(13, [1000, 77, 513], 2, 4, 2, 16, 2, q_gain=2.0)
    out = oracle.run(q, k, off, chunk=32, mode="mass", mass=0.5)
    coff = out["chunk_off"]
    for b in range(3):
        lo, hi = out["kept_off"][b], out["kept_off"][b + 1]
        idx, pos = out["kept_idx"][lo:hi], out["kept_pos"][lo:hi]
        n = off[b + 1] - off[b]
        assert np.all(np.diff(idx) > 0)
        np.testing.assert_array_equal(idx - off[b], pos)
        flags = out["chunk_keep"][coff[b]:coff[b + 1]]
        sizes = [min(32, n - 32 * c) for c in range(len(flags))]
        expect = sum(s for s, f in zip(sizes, flags) if f) + (0 if flags[0] else 1)
        assert hi - lo == expect
        assert pos[0] == 0 and pos[-1] == n - 1
        assert flags[-1] & 2


def test_needles_are_kept_small_workload():
    w = get_workload("tiny")
    inp = make_inputs(w)
    out = oracle.run(inp.q, inp.k, inp.seq_off, **w.selection_kwargs())
    kept = set(out["kept_idx"].tolist())
    assert len(inp.needles) == 3
    for (b, t, h) in inp.needles:
        assert inp.seq_off[b] + t in kept
    # fixed p = 0.30 of 16 chunks: 5 ranked + forced final chunk
    assert int((out["chunk_keep"] & 1).sum()) == 5


@pytest.mark.slow
def test_mass_selection_finds_needles_08b_workload():
    """Mass mode keeps chunks until 85 % of the score mass: with needle keys
    dominating every head, each ranked-selected chunk must sit within half a
    pool window of a planted needle, and the strongest needle chunk is kept.
    (Needles sharing a query head have identical keys and split that head's
    attention, so the weakest may fall after the 85 % crossing.)"""
    w = get_workload("draft08b")
    inp = make_inputs(w)
    out = oracle.run(inp.q, inp.k, inp.seq_off, **w.selection_kwargs())
    half = w.pool_w // 2
    near = np.zeros(len(out["chunk_score"]), dtype=bool)
    for (b, t, h) in inp.needles:
        for u in range(t - half, t + half + 1):
            near[u // w.chunk] = True
    ranked = np.flatnonzero(out["chunk_keep"] & 1)
    assert len(ranked) >= 1 and near[ranked].all()
    top = oracle.rank_order(out["chunk_score"])[0]
    assert out["chunk_keep"][top] & 1 and near[top]
    assert out["final_score"].min() >= 0.0


def test_empty_prompt_changes_nothing_else():
    """An empty prompt owns no chunks and keeps nothing; removing it leaves
    every other prompt's results unchanged."""
    q, k, off = random_case(14, [90, 0, 40], 2, 4, 2, 8, 2, q_gain=2.0)
    out = oracle.run(q, k, off, chunk=8, mode="fixed", keep_p=0.3)
    q2 = q[[0, 2]]
    off2 = np.array([0, 90, 130])
    ref = oracle.run(q2, k, off2, chunk=8, mode="fixed", keep_p=0.3)
    for key in ("imp", "chunk_score", "chunk_keep", "kept_idx", "kept_pos"):
        np.testing.assert_array_equal(out[key], ref[key], err_msg=key)
    np.testing.assert_array_equal(out["kept_off"], [ref["kept_off"][0], ref["kept_off"][1],
                                                    ref["kept_off"][1], ref["kept_off"][2]])


def test_bf16_decode_exact():
    vals = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3, 65280.0], dtype=np.float32)
    bits = bf16_bits_from_f32(vals)
    dec = so.decode_bf16(bits)
    # bf16 keeps 8 significant bits: these are all representable except 1e-3
    np.testing.assert_array_equal(dec[[0, 1, 2, 3, 5]], vals[[0, 1, 2, 3, 5]].astype(np.float64))
    assert abs(dec[4] - 1e-3) <= 1e-3 * 2.0 ** -8


# --- sparse-prefill consumer: rows of the kept tokens -------------------------------


def test_gather_rows_brute_force_and_invariants():
    rng = np.random.default_rng(77)
    ly, ntot, hk, d = 3, 40, 2, 8
    cache = rng.integers(0, 1 << 16, size=(ly, ntot, hk, d), dtype=np.uint16)
    kept = [0, 3, 4, 5, 17, 39]
    out = oracle.gather_rows(cache, kept)
    assert out.shape == (ly, len(kept), hk, d) and out.dtype == cache.dtype
    # element by element with plain loops
    for layer in range(ly):
        for i, t in enumerate(kept):
            for g in range(hk):
                for x in range(d):
                    assert out[layer, i, g, x] == cache[layer, t, g, x]
    # the identity list returns the cache; a permutation and its inverse cancel
    assert np.array_equal(oracle.gather_rows(cache, range(ntot)), cache)
    perm = rng.permutation(ntot)
    back = oracle.gather_rows(oracle.gather_rows(cache, perm), np.argsort(perm))
    assert np.array_equal(back, cache)
    # an empty list gives no rows
    assert oracle.gather_rows(cache, []).shape == (ly, 0, hk, d)


# ---------------------------------------------------------------- listing rule


def test_listing_keep_count_rounds_the_product_in_float32():
    # 0.4f = 0.4000000059604645; 5 * 0.4f = 2.0000000298 in exact arithmetic,
    # which rounds to 2.0 in float32: the listing keeps 2 chunks, the exact
    # rule (float64 product of the float32 p) keeps 3
    assert oracle.listing_keep_count(5, 0.4) == 2
    assert oracle.fixed_count(5, 0.4) == 3
    # 16 * 0.3f = 4.8000002 -> 5; 1024 * 0.15f = 153.6 -> 154; tiny p -> 1
    assert oracle.listing_keep_count(16, 0.3) == 5
    assert oracle.listing_keep_count(1024, 0.15) == 154
    assert oracle.listing_keep_count(10, 0.01) == 1
    assert oracle.listing_keep_count(7, 1.0) == 7


def test_listing_forced_tokens_and_eff_min():
    assert oracle.listing_forced_tokens(1) == [0]
    assert oracle.listing_forced_tokens(4) == [0, 1, 2, 3]
    assert oracle.listing_forced_tokens(5) == [0, 1, 2, 3, 4]
    assert oracle.listing_forced_tokens(100) == [0, 1, 2, 3, 98, 99]
    assert oracle.listing_eff_min(400, 128) == 40
    assert oracle.listing_eff_min(30, 128) == 4
    assert oracle.listing_eff_min(5000, 128) == 128
    assert oracle.listing_eff_min(5000, 8) == 8


def test_listing_cap_hand_worked():
    ten = list(range(10))
    assert oracle.listing_cap(ten, 4) == [0, 2, 4, 9]     # step 2, last replaced
    assert oracle.listing_cap(ten, 3) == [0, 3, 9]        # step 3
    assert oracle.listing_cap(ten, 1) == [9]              # step 10
    assert oracle.listing_cap(ten, 10) == ten
    assert oracle.listing_cap(ten, 0) == ten              # disabled
    assert oracle.listing_cap([1, 5, 7, 8, 20, 21, 22], 2) == [1, 22]


def _listing(cs, n, chunk, **kw):
    base = dict(mode="fixed", keep_p=0.3, mass=0.85, min_tok=128, max_keep=0)
    base.update(kw)
    return oracle.select_listing(np.asarray(cs, dtype=np.float64), n, chunk=chunk, **base)


def test_listing_ties_keep_every_chunk_at_the_threshold():
    # k = ceil(10 * 0.2f) = 2; the 2nd largest score 0.9 is shared by three
    # chunks, all kept; eff_min = 10 is met, no fill
    cs = [0.1, 0.9, 0.3, 0.9, 0.2, 0.5, 0.9, 0.05, 0.4, 0.6]
    s = _listing(cs, 100, 10, keep_p=0.2)
    assert s.chunk_keep.tolist() == [0, 1, 0, 1, 0, 0, 1, 0, 0, 0]
    want = [0, 1, 2, 3] + list(range(10, 20)) + list(range(30, 40)) + list(range(60, 70)) + [98, 99]
    assert s.kept_tokens.tolist() == want
    # the exact rule keeps k chunks, ties broken by index
    ex = oracle.select_prompt(np.asarray(cs), 100, chunk=10, mode="fixed", keep_p=0.15, mass=0.85,
                              force_bos=False, force_last_chunk=False)
    assert ex.chunk_keep.tolist() == [0, 1, 0, 1, 0, 0, 0, 0, 0, 0]


def test_listing_fill_up_to_eff_min():
    # n = 400, C = 32: 13 chunks (the last of 16 tokens); eff_min = 40;
    # k = ceil(13 * 0.05f) = 1 keeps chunk 5 (32 tokens) + 6 forced = 38;
    # the fill adds tokens 4 and 5 of chunk 0, the first unselected chunk
    cs = np.linspace(0.1, 0.2, 13)
    cs[5] = 0.9
    s = _listing(cs, 400, 32, keep_p=0.05)
    assert s.chunk_keep.tolist() == [1 if c == 5 else 0 for c in range(13)]
    assert s.kept_tokens.tolist() == [0, 1, 2, 3, 4, 5] + list(range(160, 192)) + [398, 399]
    # a smaller min_tok (eff_min 8) needs no fill
    s = _listing(cs, 400, 32, keep_p=0.05, min_tok=8)
    assert s.kept_tokens.tolist() == [0, 1, 2, 3] + list(range(160, 192)) + [398, 399]
    # n = 800: 25 chunks, k = ceil(25 * 0.01f) = 1 keeps chunk 1 (tokens
    # 32-63) + 6 forced = 38; eff_min = 80 asks for 42 more: tokens 4-31 of
    # chunk 0 (28), then the selected chunk 1 is skipped and tokens 64-77 of
    # chunk 2 (14) complete it
    cs2 = np.linspace(0.1, 0.2, 25)
    cs2[1] = 0.95
    s = _listing(cs2, 800, 32, keep_p=0.01, min_tok=80)
    assert s.kept_tokens.tolist() == list(range(0, 78)) + [798, 799]


def test_listing_keep_all_cases_and_cap():
    cs = [0.3, 0.1, 0.2]
    assert _listing(cs, 4, 2, keep_p=0.1).kept_tokens.tolist() == [0, 1, 2, 3]  # n <= eff_min
    s = _listing(cs, 80, 32, keep_p=1.0)
    assert s.kept_tokens.tolist() == list(range(80)) and s.chunk_keep.tolist() == [1, 1, 1]
    s = _listing(cs, 80, 32, keep_p=1.0, max_keep=8)       # 80 // 8 = 10
    assert s.kept_tokens.tolist() == [0, 10, 20, 30, 40, 50, 60, 79]


def test_listing_mass_mode_adds_forced_tokens_and_fill():
    # mass 0.5 of the total 1.0: chunk 2 (0.6) alone reaches it
    cs = [0.1, 0.1, 0.6, 0.2]
    s = _listing(cs, 100, 25, mode="mass", mass=0.5, min_tok=12)   # eff_min = 10
    assert s.chunk_keep.tolist() == [0, 0, 1, 0]
    assert s.kept_tokens.tolist() == [0, 1, 2, 3] + list(range(50, 75)) + [98, 99]


def test_listing_invariants_on_random_prompts():
    rng = np.random.default_rng(123)
    for _ in range(200):
        n = int(rng.integers(1, 700))
        chunk = int(rng.choice([4, 16, 32]))
        nc = -(-n // chunk)
        cs = np.round(rng.random(nc), 1)           # coarse values: many ties
        kw = dict(keep_p=float(rng.choice([0.05, 0.3, 0.7, 1.0])), min_tok=int(rng.integers(1, 200)),
                  max_keep=int(rng.choice([0, 5, 50])), mode=str(rng.choice(["fixed", "mass"])))
        s = _listing(cs, n, chunk, **kw)
        kt = s.kept_tokens.tolist()
        assert kt == sorted(set(kt)) and all(0 <= t < n for t in kt)
        uncapped = _listing(cs, n, chunk, **dict(kw, max_keep=0)).kept_tokens.tolist()
        assert set(oracle.listing_forced_tokens(n)) <= set(uncapped)
        assert len(uncapped) >= min(n, oracle.listing_eff_min(n, kw["min_tok"]))
        sel_tokens = {t for c in range(nc) if s.chunk_keep[c] for t in range(c * chunk, min(n, c * chunk + chunk))}
        assert sel_tokens <= set(uncapped)
        if kw["max_keep"] and len(uncapped) > kw["max_keep"]:
            assert len(kt) == kw["max_keep"] and kt[-1] == uncapped[-1] and set(kt) <= set(uncapped)
        else:
            assert kt == uncapped
        if kw["mode"] == "fixed" and kw["keep_p"] < 1.0 and n > oracle.listing_eff_min(n, kw["min_tok"]):
            k = oracle.listing_keep_count(nc, kw["keep_p"])
            # every selected chunk scores at least every unselected one, and at
            # least k chunks are selected (exactly k when the k-th score is unique)
            sel = s.chunk_keep.astype(bool)
            assert sel.sum() >= min(k, nc)
            if (~sel).any():
                assert cs[sel].min() > cs[~sel].max()


# ---------------------------------------------------------------- sliding windows


def test_auto_window_closed_forms():
    # 500 MiB / (8192 * 32) = 2000 tokens, stride 1000 (the guide's default)
    assert oracle.auto_window(8192) == (2000, 1000)
    # 500 MiB / (4096 * 32) = 4000 > 4096 - 512
    assert oracle.auto_window(4096) == (3584, 1792)
    assert oracle.auto_window(8192, 300) == (512, 256)      # raised to 512
    assert oracle.auto_window(600) == (472, 236)            # lowered to spec_ctx - 128 last
    assert oracle.auto_window(8192, 5000) == (5000, 2500)


def test_window_plan_matches_the_guides_examples():
    # 10,000 tokens, window 2000 / stride 1000: windows start every 1000
    # tokens and each keeps its first 1000 scores; the window starting at
    # 8000 already reaches the end and is the last (the fixed loop drops the
    # redundant window at 9000)
    plan = oracle.window_plan(10000, 2000, 1000)
    assert [p[0] for p in plan] == list(range(0, 9000, 1000))
    assert all(p == (s, s + 2000, 1000) for p, s in zip(plan[:-1], range(0, 8000, 1000)))
    assert plan[-1] == (8000, 10000, 2000)
    # a 4.5K prompt takes 4 windows instead of 5
    plan = oracle.window_plan(4500, 2000, 1000)
    assert len(plan) == 4 and plan[-1] == (3000, 4500, 1500)
    assert oracle.window_plan(1500, 2000, 1000) == [(0, 1500, 1500)]
    assert oracle.window_plan(0, 2000, 1000) == []


def test_window_plan_covers_every_token_once():
    rng = np.random.default_rng(9)
    for _ in range(300):
        window = int(rng.integers(2, 300))
        stride = window // 2
        n = int(rng.integers(1, 2000))
        plan = oracle.window_plan(n, window, stride)
        covered = np.zeros(n, dtype=np.int64)
        for start, end, kept in plan:
            assert 0 <= start < end <= n and end - start <= window and 1 <= kept <= end - start
            covered[start:start + kept] += 1
        assert (covered == 1).all()
        # every window but the last is full length
        assert all(end - start == window for start, end, _ in plan[:-1])


def test_merge_windows_places_each_windows_scores():
    n, window, stride = 4500, 2000, 1000
    plan = oracle.window_plan(n, window, stride)
    imps = [np.full(end - start, float(w + 1)) for w, (start, end, _) in enumerate(plan)]
    merged = oracle.merge_windows(imps, n, window, stride)
    want = np.concatenate([np.full(1000, 1.0), np.full(1000, 2.0), np.full(1000, 3.0),
                           np.full(1500, 4.0)])
    assert np.array_equal(merged, want)
    # positions inside a window map to the window's own token offsets
    imps = [np.arange(end - start, dtype=np.float64) + 10000 * w for w, (start, end, _) in enumerate(plan)]
    merged = oracle.merge_windows(imps, n, window, stride)
    for t in (0, 999, 1000, 2500, 2999, 3000, 4499):
        w = min(t // stride, len(plan) - 1)
        assert merged[t] == 10000 * w + (t - plan[w][0])


# ---------------------------------------------------------------- per-head pooling


@pytest.mark.parametrize("i", range(len(TINY_CASES)))
def test_head_pooling_matches_bruteforce(i):
    q, k, off, params = _case(i)
    params = dict(params, pool_at="head")
    got = oracle.run(q, k, off, **params)
    want = bruteforce.run_bruteforce(q, k, off, **params)
    for key in ("imp", "tok_score", "final_score", "chunk_score"):
        np.testing.assert_allclose(got[key], want[key], rtol=1e-12, atol=1e-15, err_msg=key)
    for key in ("chunk_keep", "kept_idx", "kept_pos", "kept_off"):
        np.testing.assert_array_equal(np.asarray(got[key]), np.asarray(want[key]), err_msg=key)
    # the pooled importance is the score: step 5 is the identity
    np.testing.assert_array_equal(got["tok_score"], got["imp"])


def test_pool_rows_against_convolution():
    rng = np.random.default_rng(12)
    p = rng.random((3, 2, 50))
    for w in (1, 3, 13):
        got = oracle.pool_rows(p, w)
        h = w // 2
        for idx in np.ndindex(3, 2):
            row = p[idx]
            np.testing.assert_allclose(got[idx][h:50 - h], np.convolve(row, np.ones(w) / w, "valid"),
                                       rtol=1e-13)
            # edges: mean over the in-range part of the window
            np.testing.assert_allclose(got[idx][0], row[:h + 1].mean(), rtol=1e-13)
            np.testing.assert_allclose(got[idx][-1], row[-h - 1:].mean(), rtol=1e-13)
    # one window wider than the row: every output is the row mean
    np.testing.assert_allclose(oracle.pool_rows(p[:, :, :5], 13), np.broadcast_to(
        p[:, :, :5].mean(axis=-1, keepdims=True), (3, 2, 5)), rtol=1e-13)


def test_head_pooling_equals_token_pooling_when_rows_coincide():
    """With every (layer, head) row of a step equal, pooling commutes with
    the max and, being linear, with the mean over steps: both placements
    give the same scores."""
    rng = np.random.default_rng(3)
    ly, hq, hk, d, steps, n = 3, 4, 2, 16, 3, 90
    qs = rng.standard_normal((steps, d)).astype(np.float32) * 2.0
    k1 = rng.standard_normal((n, d)).astype(np.float32)
    q = np.broadcast_to(qs[None, None, :, None, :], (1, ly, steps, hq, d)).copy()
    k = np.broadcast_to(k1[None, :, None, :], (ly, n, hk, d)).copy()
    q, k = bf16_bits_from_f32(q), bf16_bits_from_f32(k)
    off = np.array([0, n])
    kw = dict(pool_w=13, chunk=8, mode="fixed", keep_p=0.3)
    tok = oracle.run(q, k, off, **kw)
    head = oracle.run(q, k, off, pool_at="head", **kw)
    np.testing.assert_allclose(head["imp"], tok["tok_score"], rtol=1e-12)
    np.testing.assert_allclose(head["chunk_score"], tok["chunk_score"], rtol=1e-12)


def test_head_pooling_with_width_one_is_the_default_path():
    q, k, off, params = _case(1)
    params = dict(params, pool_w=1)
    a = oracle.run(q, k, off, **params)
    b = oracle.run(q, k, off, pool_at="head", **params)
    for key in ("imp", "tok_score", "chunk_score", "kept_idx"):
        np.testing.assert_array_equal(a[key], b[key])


# ---------------------------------------------------------------- paged caches


def _scatter_pages(k, seq_off, block_size, rng, spare_blocks=3):
    """Scatter dense [Ly, Ntot, Hk, d] keys into per-layer pools of shuffled
    blocks (plus unused blocks of noise); returns (pools, block_table)."""
    ly, _, hk, d = k.shape
    seq_off = np.asarray(seq_off)
    nblk = [-(-int(seq_off[b + 1] - seq_off[b]) // block_size) for b in range(len(seq_off) - 1)]
    total = sum(nblk) + spare_blocks
    perm = rng.permutation(total)
    table = np.full((len(nblk), max(max(nblk), 1) + 2), -1, dtype=np.int32)
    pools = [rng.integers(0, 1 << 16, size=(total, block_size, hk, d), dtype=np.uint16) for _ in range(ly)]
    used = 0
    for b, nb in enumerate(nblk):
        start, n = int(seq_off[b]), int(seq_off[b + 1] - seq_off[b])
        for j in range(nb):
            phys = int(perm[used]); used += 1
            table[b, j] = phys
            rows = min(block_size, n - j * block_size)
            for layer in range(ly):
                pools[layer][phys, :rows] = k[layer, start + j * block_size:start + j * block_size + rows]
    return pools, table


def test_kv_from_pages_round_trip_and_scores():
    rng = np.random.default_rng(21)
    q, k, off = random_case(31, [37, 0, 70, 5], 2, 4, 2, 16, 2, q_gain=2.0)
    for bs in (8, 16, 64):
        pools, table = _scatter_pages(k, off, bs, rng)
        dense = oracle.kv_from_pages(pools, table, off, bs)
        assert np.array_equal(dense, k)
    # element by element for one token of one prompt
    pools, table = _scatter_pages(k, off, 16, rng)
    t, b = 53, 2
    assert np.array_equal(oracle.kv_from_pages(pools, table, off, 16)[1, off[b] + t],
                          pools[1][table[b, t // 16], t % 16])
    # the scores of the paged cache are those of the dense keys
    kw = dict(pool_w=5, chunk=4, mode="fixed", keep_p=0.3)
    a = oracle.run(q, k, off, **kw)
    bb = oracle.run(q, oracle.kv_from_pages(pools, table, off, 16), off, **kw)
    assert np.array_equal(a["imp"], bb["imp"]) and np.array_equal(a["kept_idx"], bb["kept_idx"])
