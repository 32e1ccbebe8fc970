"""Mass-mode selection near the threshold: the GPU walks the ranking on
fixed-point chunk scores (round(s * 2^S), S from the prompt's largest score
and chunk count: S = 52 - (floor(log2 max) + 1) - ceil(log2(nc + 1))), so
its running sums differ from exact ones by at most nc / 2 units of 2^-S and
its threshold ceil(mass * total) by at most one more unit. Its decision can
therefore differ from the oracle's float64 walk only when the crossing lies
within beta = (nc + 1) * 2^-S of mass * total; scores of at least
2^(23 - S) are represented exactly. Cases (chunk = 1, so the chunk scores
are the given importance values exactly; pool 1, no normalisation, no
boost):
  * a crossing far outside beta: the GPU keeps exactly the oracle's chunks
    (T1), on the fused rank path and on the stage entry point sp_select;
  * a crossing inside beta among scores that the fixed point rounds: the
    GPU keeps the oracle's chunks or one crossing chunk more or fewer."""

import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

N_BIG, N_TAIL = 64, 100
MASS = np.float32(1.0 - 8 * 2.0 ** -24)


def _beta(scores):
    nc = len(scores)
    smax = float(np.max(scores))
    s = 52 - (math.floor(math.log2(smax)) + 1) - math.ceil(math.log2(nc + 1))
    return (nc + 1) * 2.0 ** -s, s


def _case(within):
    """64 distinct dyadic scores, then 100 equal small scores v (not
    multiples of 2^-S) whose running sum crosses mass * total; v is chosen
    so that the crossing's distance from the threshold is far above beta,
    or below it."""
    big = ((512 + 4 * np.arange(N_BIG)) / 1024.0).astype(np.float32)[::-1]
    B = float(np.sum(big.astype(np.float64)))
    m = float(MASS)
    v0 = np.float32(3.0e-7)
    vs = (v0.view(np.uint32) + np.arange(-200000, 200000, dtype=np.int64)).astype(np.uint32).view(np.float32)
    vv = vs.astype(np.float64)
    theta = m * (B + N_TAIL * vv)
    k = np.ceil((theta - B) / vv)
    r = B + k * vv - theta                       # distance of the crossing from the threshold
    scores = np.concatenate([big, np.zeros(N_TAIL, np.float32)])
    beta, S = _beta(np.concatenate([big, np.full(N_TAIL, v0, np.float32)]))
    exact_grid = np.mod(vv * 2.0 ** S, 1.0) != 0.0    # the fixed point rounds v
    if within:
        ok = (r > 0) & (r < beta / 2) & exact_grid & (k > 5) & (k < N_TAIL - 5)
    else:
        ok = (r > 1e4 * beta) & (k > 5) & (k < N_TAIL - 5)
    i = int(np.flatnonzero(ok)[0])
    scores[N_BIG:] = vs[i]
    return scores, float(r[i]), beta


def _gpu_flags(sp, scores, stage):
    import torch
    kw = dict(pool_w=1, chunk=1, mode="mass", keep_p=0.3, mass=float(MASS), normalize=False, boost_first_mult=1.0,
              boost_last_mult=1.0, force_bos=True, force_last_chunk=True)
    p = sp.SelectionParams(**kw)
    n = len(scores)
    off = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    imp = torch.from_numpy(scores.copy()).cuda()
    if stage:
        cs = imp.clone()
        coff = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        keep = sp.select(cs, coff, off, n, p)
        flags = keep.cpu().numpy()
        got_cs = scores
    else:
        out = sp.select_from_importance(imp, off, p)
        flags = out.chunk_keep[:n].cpu().numpy()
        got_cs = out.chunk_score[:n].cpu().numpy()
    torch.cuda.synchronize()
    assert np.array_equal(got_cs.view(np.uint32), scores.view(np.uint32))   # chunk scores exact
    ref = oracle.select_from_chunk_scores(scores.astype(np.float64), np.array([0, n]), **kw)
    return flags, ref["chunk_keep"]


@pytest.mark.parametrize("stage", [False, True])
def test_crossing_far_from_threshold_is_exact(cuda_lib, stage):
    scores, r, beta = _case(within=False)
    assert r > 1e4 * beta
    flags, ref = _gpu_flags(cuda_lib, scores, stage)
    np.testing.assert_array_equal(flags, ref)


@pytest.mark.parametrize("stage", [False, True])
def test_crossing_within_the_rounding_bound(cuda_lib, stage):
    scores, r, beta = _case(within=True)
    assert 0 < r < beta
    flags, ref = _gpu_flags(cuda_lib, scores, stage)
    got_sel = (flags & 1).astype(bool)
    ref_sel = (ref & 1).astype(bool)
    assert np.array_equal(flags & 2, ref & 2)              # the forced final chunk
    assert np.array_equal(got_sel[:N_BIG], ref_sel[:N_BIG])  # every large chunk kept
    # the walk keeps a prefix of the equal small chunks (index order); it
    # may end one chunk before or after the oracle's crossing
    k_got, k_ref = int(got_sel[N_BIG:].sum()), int(ref_sel[N_BIG:].sum())
    assert np.array_equal(got_sel[N_BIG:N_BIG + k_got], np.ones(k_got, bool))
    assert abs(k_got - k_ref) <= 1
