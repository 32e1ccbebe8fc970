"""GPU parity of the reference-compatibility mode against the oracle,
through the C ABI: the listing's selection rule (ties at the threshold,
six forced tokens, eff_min fill, strided max-keep cap) and the sliding-window
scoring (per-window importance, merge, selection from the merged vector).

Scores agree within 1e-3 relative + 1e-5 absolute; the integer results are
compared bit for bit:
  T1  the oracle's listing selection run on the GPU's own fp32 chunk scores
      gives the GPU's flags and lists exactly;
  T2  end to end, where the oracle's cut-off has a safe margin.
"""

import numpy as np
import pytest

import oracle
from oracle import specprefill_oracle as so
from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.golden.margins import RANK_GAP

pytestmark = pytest.mark.gpu

LIST_KEYS = ("chunk_keep", "kept_idx", "kept_pos", "kept_off")


def _dev(inp_q, inp_k, off):
    return gh.to_device(type("I", (), {"q": inp_q, "k": inp_k, "seq_off": off})())


def _score(sp, q, k, off, kw):
    import torch
    qd, kd, od = _dev(q, k, off)
    p = sp.SelectionParams(**kw)
    ws = sp.make_workspace(sp.shape_of(qd, kd), p, poison=True)
    out = sp.specprefill_score(qd, kd, od, p, ws=ws)
    torch.cuda.synchronize()
    assert sp.device_status(ws) == 0
    return gh.out_to_numpy(out)


def _t1(got, seq_off, kw):
    t1 = oracle.select_from_chunk_scores(got["chunk_score"].astype(np.float64), seq_off, **kw)
    for key in LIST_KEYS:
        np.testing.assert_array_equal(got[key], t1[key], err_msg=f"T1 {key}")
    return t1


def _listing_margin_ok(cs, kw):
    """Fixed mode: relative gap between the k-th and (k+1)-th largest
    scores; mass mode: the exact rule's margins (same ranking prefix)."""
    cs = np.asarray(cs, dtype=np.float64)
    nc = cs.shape[0]
    if kw["mode"] == "mass":
        from tests.golden.margins import margins_ok, prompt_margins
        return margins_ok(prompt_margins(cs, "mass", kw.get("keep_p", 0.3), kw["mass"]))
    k = so.listing_keep_count(nc, kw["keep_p"])
    if k >= nc:
        return True
    r = np.sort(cs)[::-1]
    return (r[k - 1] - r[k]) / r[k - 1] >= RANK_GAP


def _t2(got, ref, seq_off, kw):
    coff = ref["chunk_off"]
    safe = 0
    for b in range(len(seq_off) - 1):
        if not _listing_margin_ok(ref["chunk_score"][coff[b]:coff[b + 1]], kw):
            continue
        safe += 1
        g0, g1 = got["kept_off"][b], got["kept_off"][b + 1]
        r0, r1 = ref["kept_off"][b], ref["kept_off"][b + 1]
        np.testing.assert_array_equal(got["kept_idx"][g0:g1], ref["kept_idx"][r0:r1], err_msg=f"T2 b={b}")
        np.testing.assert_array_equal(got["kept_pos"][g0:g1], ref["kept_pos"][r0:r1])
    return safe


BASE = dict(pool_w=13, chunk=32, keep_p=0.3, mass=0.85, normalize=True, boost_first_mult=1.5, boost_first_n=64,
            boost_last_mult=1.3, boost_last_n=128, force_bos=True, force_last_chunk=True,
            rule="listing", min_tok=128, max_keep=0)

CASES = [
    # lengths, Ly, Hq, Hk, d, L, selection
    ([4000], 2, 8, 2, 128, 4, dict(mode="fixed", keep_p=0.3)),
    ([4000], 2, 8, 2, 128, 4, dict(mode="fixed", keep_p=0.3, max_keep=500)),       # capped
    ([900, 300, 3, 0, 1200], 1, 4, 2, 64, 3, dict(mode="fixed", keep_p=0.05)),      # fill, tiny, empty
    ([2500, 700], 2, 4, 1, 256, 2, dict(mode="mass", mass=0.85, max_keep=300)),
    ([1500, 60], 1, 4, 2, 64, 2, dict(mode="fixed", keep_p=1.0, max_keep=200)),      # keep all + cap
    ([3000], 1, 8, 2, 128, 8, dict(mode="fixed", keep_p=0.2, chunk=64, pool_w=1, min_tok=400)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_listing_rule_matches_oracle(cuda_lib, case):
    lengths, ly, hq, hk, d, steps, sel = CASES[case]
    kw = dict(BASE)
    kw.update(sel)
    q, k, off = random_case(700 + case, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    got = _score(cuda_lib, q, k, off, kw)
    ref = oracle.run(q, k, off, **kw)
    for key in ("imp", "tok_score", "chunk_score"):
        assert gh.within_tol(got[key], ref[key]) <= 0, key
    t1 = _t1(got, off, kw)
    assert _t2(got, ref, off, kw) >= 1
    # each case exercises what it is there for
    lens = np.diff(off)
    if kw["max_keep"]:
        per = np.diff(t1["kept_off"])
        assert (per <= kw["max_keep"]).all() and (per == kw["max_keep"]).any()


def test_listing_fill_and_forced_tokens_are_exercised(cuda_lib):
    """A low keep fraction on short prompts: the ranked chunks plus the six
    forced tokens stay below eff_min, so the fill decides the tail of the
    list (the oracle confirms a fill happened)."""
    kw = dict(BASE, mode="fixed", keep_p=0.02, pool_w=13)
    lengths = [1000, 640, 480]
    q, k, off = random_case(811, lengths, 1, 4, 2, 64, 2, q_gain=2.0)
    got = _score(cuda_lib, q, k, off, kw)
    t1 = _t1(got, off, kw)
    for b, n in enumerate(lengths):
        kept = t1["kept_pos"][t1["kept_off"][b]:t1["kept_off"][b + 1]]
        assert len(kept) == so.listing_eff_min(n, kw["min_tok"])
        assert set(so.listing_forced_tokens(n)) <= set(kept.tolist())


def test_listing_ties_keep_every_chunk_at_the_threshold(cuda_lib):
    """Zero keys give uniform attention, so every token has the same
    importance (no pooling), normalisation maps it to 1, and the boost makes
    two chunks 1.5, four chunks 1.3 and the rest 1. k = ceil(32 * 0.1f) = 4
    falls inside the 1.3 tie: the listing keeps all six chunks scoring at
    least 1.3 (the exact rule keeps 4)."""
    q, k, off = random_case(5, [1024], 1, 4, 2, 64, 2)
    k = np.zeros_like(k)
    kw = dict(BASE, mode="fixed", keep_p=0.1, pool_w=1)
    got = _score(cuda_lib, q, k, off, kw)
    _t1(got, off, kw)
    assert int((got["chunk_keep"] & 1).sum()) == 6
    exact = _score(cuda_lib, q, k, off, dict(kw, rule="exact", force_last_chunk=False))
    assert int((exact["chunk_keep"] & 1).sum()) == 4


def test_sliding_window_scoring_matches_oracle(cuda_lib):
    """A 5000-token prompt scored in windows of 1024 (stride 512), each
    window with its own keys and lookahead queries as the pages' tool
    re-prefills the draft per window: per-window importance on the GPU (the
    windows as a batch of prompts), merged on the GPU, selected with the
    listing rule from the merged vector (no pooling, as in the tool)."""
    import torch
    sp = cuda_lib
    n, (window, stride) = 5000, (1024, 512)
    plan = oracle.window_plan(n, window, stride)
    lengths = [e - s for s, e, _ in plan]
    q, k, woff = random_case(902, lengths, 2, 8, 2, 128, 4, q_gain=2.0)
    qd, kd, wod = _dev(q, k, woff)
    p_imp = sp.SelectionParams()
    imp_w = sp.attn_importance(qd, kd, wod, p_imp)
    merged = sp.merge_windows(imp_w, n, window, stride)
    kw = dict(BASE, mode="fixed", keep_p=0.3, pool_w=1, max_keep=2000)
    off = np.array([0, n], dtype=np.int32)
    res = sp.select_from_importance(merged, torch.from_numpy(off).cuda(), sp.SelectionParams(**kw))
    torch.cuda.synchronize()
    got = gh.out_to_numpy(res)
    # oracle: the same windows, merged, selected
    ref_w = oracle.importance(q, k, woff)
    ref_imp = oracle.merge_windows([ref_w[woff[i]:woff[i + 1]] for i in range(len(plan))], n, window, stride)
    assert gh.within_tol(got["imp"], ref_imp) <= 0
    # the merge is a copy: bit-exact against the GPU's own window scores
    iw = imp_w.cpu().numpy()
    want = np.concatenate([iw[woff[i]:woff[i] + kept] for i, (_, _, kept) in enumerate(plan)])
    assert np.array_equal(got["imp"], want)
    ref = oracle.score_from_importance(ref_imp, off, **kw)
    for key in ("tok_score", "chunk_score"):
        assert gh.within_tol(got[key], ref[key]) <= 0, key
    _t1(got, off, kw)
    assert _t2(got, ref, off, kw) == 1


def test_select_from_importance_composes_to_the_fused_call(cuda_lib):
    """sp_attn_importance followed by sp_select_from_importance equals
    sp_specprefill_score bit for bit (exact and listing rules)."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(66, [3000, 1100], 2, 8, 2, 128, 4, q_gain=2.0)
    qd, kd, od = _dev(q, k, off)
    for kw in (dict(mode="mass", mass=0.85), dict(BASE, mode="fixed", keep_p=0.2, max_keep=300)):
        p = sp.SelectionParams(**kw)
        fused = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p))
        imp = sp.attn_importance(qd, kd, od, p)
        two = gh.out_to_numpy(sp.select_from_importance(imp, od, p))
        torch.cuda.synchronize()
        for key in fused:
            assert np.array_equal(fused[key], two[key]), key
